// kvr_convert.cuh -- element conversion of the relayout kernel (BF16 <-> FP8 E4M3, sm_103a).
//
// Device functions only, included by relayout.cu. A unit is 16 elements: 32
// bytes on the BF16 side, 16 on the FP8 side.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

// -- element conversion (BF16 <-> FP8 E4M3) ------------------------------------
//
// Definitions (kv_relayout.h): quantize q = E4M3(x * (1/s)), nearest-even,
// saturating at +-448, NaN kept with its sign; dequantize y = BF16(q * s),
// nearest-even, a NaN code -> sign | 0x7FC0. Both run two elements per
// instruction where the hardware allows it: a packed fp32 product
// (mul.rn.f32x2: two independent IEEE products, each rounded to nearest-even,
// subnormals kept) and the paired conversions to and from E4M3 / BF16. A NaN
// product's sign is not fixed by IEEE 754 (the GPU returns a positive one), so
// the input signs are put back explicitly: on quantizing, every code gets its
// input's sign bit (a no-op for all but NaN, since 1/s > 0 keeps the product's
// sign, signed zeros included); on dequantizing, units that hold a NaN code
// are patched after the conversion.

// {x0, x1} * {s, s}: two fp32 products (element 0 in the low half).
static __device__ __forceinline__ uint64_t mul_f32x2(uint64_t x, uint64_t s2) {
    uint64_t y;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(y) : "l"(x), "l"(s2));
    return y;
}

// {s, s} as one 64-bit operand of mul_f32x2.
static __device__ __forceinline__ uint64_t splat_f32x2(float s) {
    const uint64_t b = __float_as_uint(s);
    return b | (b << 32);
}

static __device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Two BF16 (element 0 in the low half of `w`) -> two E4M3 codes (element 0 in
// bits 7..0) of the signed products, nearest-even, saturated to +-448 (a NaN
// product gives 0x7F).
static __device__ __forceinline__ uint32_t quant2(uint32_t w, uint64_t inv2) {
    const uint64_t x = (uint64_t)(w << 16) | ((uint64_t)(w & 0xFFFF0000u) << 32);
    const uint64_t y = mul_f32x2(x, inv2);
    unsigned short d;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
        : "=h"(d)
        : "f"(__uint_as_float((uint32_t)(y >> 32))), "f"(__uint_as_float((uint32_t)y)));
    return d;
}

// Four BF16 (a: elements 0, 1; b: 2, 3) -> four E4M3 codes in one word, each
// with its input's sign bit (bytes 1 and 3 of a and b hold the BF16 signs).
static __device__ __forceinline__ uint32_t quant4(uint32_t a, uint32_t b, uint64_t inv2) {
    const uint32_t codes = quant2(a, inv2) | (quant2(b, inv2) << 16);
    return codes | (prmt(a, b, 0x7531u) & 0x80808080u);
}

// 16 BF16 (two 16-byte pieces) -> 16 E4M3 codes (one 16-byte piece).
static __device__ __forceinline__ uint4 quant16(const uint4 &a, const uint4 &b, float inv) {
    const uint64_t inv2 = splat_f32x2(inv);
    uint4 o;
    o.x = quant4(a.x, a.y, inv2);
    o.y = quant4(a.z, a.w, inv2);
    o.z = quant4(b.x, b.y, inv2);
    o.w = quant4(b.z, b.w, inv2);
    return o;
}

// Two E4M3 codes (element 0 in bits 7..0 of `c`) -> two BF16 (element 0 in
// the low half): exact decode to f16x2, exact widening to fp32, packed fp32
// products, nearest-even rounding to BF16 (overflow to infinity). NaN codes
// are left to dequant_nan_patch.
static __device__ __forceinline__ uint32_t dequant2(unsigned short c, uint64_t s2) {
    uint32_t h2, out;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
    float f0, f1;
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\tcvt.f32.f16 %0, l;\n\t"
        "cvt.f32.f16 %1, h;\n\t}"
        : "=f"(f0), "=f"(f1)
        : "r"(h2));
    const uint64_t y = mul_f32x2((uint64_t)__float_as_uint(f0) |
                                     ((uint64_t)__float_as_uint(f1) << 32),
                                 s2);
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;"
        : "=r"(out)
        : "f"(__uint_as_float((uint32_t)(y >> 32))), "f"(__uint_as_float((uint32_t)y)));
    return out;
}

// Codes x.1111.111 (NaN) among the four of `w`: bit 7 of each such byte.
static __device__ __forceinline__ uint32_t e4m3_nan_bits(uint32_t w) {
    return ((w & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u;
}

// The BF16 of every NaN code of `w` (codes 0, 1 in *lo; 2, 3 in *hi) set to the
// code's sign | 0x7FC0; the others unchanged.
static __device__ __forceinline__ void dequant_nan_patch(uint32_t w, uint32_t *lo, uint32_t *hi) {
    const uint32_t nan = e4m3_nan_bits(w);
    // 0xFFFF over the BF16 lanes of NaN codes (byte msb replicated)
    const uint32_t m_lo = prmt(nan, 0u, 0x9988u), m_hi = prmt(nan, 0u, 0xBBAAu);
    // each code's byte moved to the high byte of its BF16 lane: its sign lands on bit 15
    const uint32_t v_lo = (prmt(w, 0u, 0x1404u) & 0x80008000u) | 0x7FC07FC0u;
    const uint32_t v_hi = (prmt(w, 0u, 0x3424u) & 0x80008000u) | 0x7FC07FC0u;
    *lo = (*lo & ~m_lo) | (v_lo & m_lo);
    *hi = (*hi & ~m_hi) | (v_hi & m_hi);
}

// 16 E4M3 codes (one 16-byte piece) -> 16 BF16 (two 16-byte pieces). The NaN
// patch runs only for words that hold a NaN code (none in finite KV data).
static __device__ __forceinline__ void dequant16(const uint4 &c, float s, uint4 *lo, uint4 *hi) {
    const uint64_t s2 = splat_f32x2(s);
    lo->x = dequant2((unsigned short)c.x, s2);
    lo->y = dequant2((unsigned short)(c.x >> 16), s2);
    if (e4m3_nan_bits(c.x) != 0u) dequant_nan_patch(c.x, &lo->x, &lo->y);
    lo->z = dequant2((unsigned short)c.y, s2);
    lo->w = dequant2((unsigned short)(c.y >> 16), s2);
    if (e4m3_nan_bits(c.y) != 0u) dequant_nan_patch(c.y, &lo->z, &lo->w);
    hi->x = dequant2((unsigned short)c.z, s2);
    hi->y = dequant2((unsigned short)(c.z >> 16), s2);
    if (e4m3_nan_bits(c.z) != 0u) dequant_nan_patch(c.z, &hi->x, &hi->y);
    hi->z = dequant2((unsigned short)c.w, s2);
    hi->w = dequant2((unsigned short)(c.w >> 16), s2);
    if (e4m3_nan_bits(c.w) != 0u) dequant_nan_patch(c.w, &hi->z, &hi->w);
}
