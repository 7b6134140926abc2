/*
 * kv_oracle.c -- plain, slow, obviously correct CPU definition of the
 * prefill -> decode KV-cache relayout.
 *
 * TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and the CPU
 * baseline / reference legs of bench.py may build, load or call this file.
 * The CUDA library never links, includes or calls it, and this file shares
 * no header, helper or constant with the CUDA library.
 *
 * What it follows (page "PD 分离与 KV 传输", ai-infra-handbooks,
 * serving/distributed/pd-disagg):
 *   - section "实现", pd.py prefill(): the prefill instance gathers every
 *     layer's K/V of the prompt, token by token, through its own block table,
 *     into a [seq, kv_heads, head_dim] array;
 *   - section "实现", pd.py admit(): the decode instance writes token p of
 *     the prompt to slot  block_ids[p // block_size] * block_size
 *     + p % block_size  of its own pool, for p < n only (so the slots of a
 *     partial last block past the prompt are never touched);
 *   - section "布局转换", item "TP 不同": the prefill side holds 1/Tp of the
 *     KV heads per card and the decode side 1/Td; a head moves from one
 *     card's shard to another's;
 *   - section "传输的代价": KV per token times prompt length is the amount
 *     of data moved.
 *
 * Readings taken where the page is silent:
 *   - pool layout, one buffer per TP shard: [L][C][N][B][H_local][D] of
 *     es-byte elements (C = 2 for K and V, C = 1 for an MLA latent);
 *   - TP shard s holds the contiguous head range [s*H/T, (s+1)*H/T) when
 *     T <= H (H_local = H/T); when T > H (more cards than KV heads, e.g. an
 *     MLA latent under TP) each head is held whole by T/H consecutive cards,
 *     shards h*T/H .. (h+1)*T/H - 1 (H_local = 1), and the hand-off reads a
 *     head from the first prefill card that holds it and writes it to every
 *     decode card that holds it;
 *   - one block table per side, shared by all shards of that side;
 *   - elements are copied as es raw bytes: no conversion, NaN payloads kept.
 *
 * Every function here is a plain loop nest; there is no blocking, fusion or
 * reordering beyond the definition.
 */
#include <stdint.h>
#include <stddef.h>

/* A TP degree a side can have for H KV heads: a divisor of H (each card a
 * head range) or a multiple of it (each head on T/H cards). */
static int tp_ok(int64_t kv_heads, int64_t tp)
{
    return tp >= 1 && kv_heads >= 1 && (kv_heads % tp == 0 || tp % kv_heads == 0);
}

/* Heads on one card, and cards that hold one head. */
static int64_t heads_per_card(int64_t kv_heads, int64_t tp)
{
    return tp <= kv_heads ? kv_heads / tp : 1;
}

static int64_t cards_per_head(int64_t kv_heads, int64_t tp)
{
    return tp <= kv_heads ? 1 : tp / kv_heads;
}

/* Bytes of KV cache one token occupies, summed over layers, components,
 * heads and head dimension ("KV/token", section "传输的代价"). */
int64_t kvo_bytes_per_token(int32_t num_layers, int32_t num_components,
                            int32_t kv_heads, int32_t head_dim,
                            int32_t elem_bytes)
{
    return (int64_t)num_layers * num_components * kv_heads * head_dim * elem_bytes;
}

/* Bytes one hand-off moves for a batch of prompts: KV/token times the
 * prompt lengths (section "传输的代价"; pd.py's own counter sums the
 * gathered K and V of every layer). */
int64_t kvo_transfer_bytes(int32_t num_layers, int32_t num_components,
                           int32_t kv_heads, int32_t head_dim,
                           int32_t elem_bytes, int32_t num_requests,
                           const int32_t *seq_lens)
{
    int64_t tokens = 0;
    for (int32_t r = 0; r < num_requests; ++r)
        tokens += seq_lens[r];
    return tokens * kvo_bytes_per_token(num_layers, num_components, kv_heads,
                                        head_dim, elem_bytes);
}

/*
 * The relayout itself, for layers [layer_begin, layer_end).
 *
 * src_pools[sp] is the prefill shard sp (of src_tp), layout
 *   [num_layers][num_components][src_num_blocks][src_block][H/src_tp][head_dim];
 * dst_pools[dp] is the decode shard dp (of dst_tp), layout
 *   [num_layers][num_components][dst_num_blocks][dst_block][H/dst_tp][head_dim].
 * Request r owns src_bt[src_off[r] ...] and dst_bt[dst_off[r] ...]; entry k
 * of a table is the physical block that holds tokens [k*B, (k+1)*B).
 *
 * Returns 0, or -1 when a TP degree neither divides the head count nor is a
 * multiple of it.
 */
int kvo_relayout(int32_t layer_begin, int32_t layer_end,
                 int32_t num_layers, int32_t num_components,
                 int32_t kv_heads, int32_t head_dim, int32_t elem_bytes,
                 int32_t src_tp, int32_t dst_tp,
                 int32_t src_block, int32_t dst_block,
                 int64_t src_num_blocks, int64_t dst_num_blocks,
                 const uint8_t *const *src_pools, uint8_t *const *dst_pools,
                 int32_t num_requests, const int32_t *seq_lens,
                 const int64_t *src_off, const int32_t *src_bt,
                 const int64_t *dst_off, const int32_t *dst_bt)
{
    if (!tp_ok(kv_heads, src_tp) || !tp_ok(kv_heads, dst_tp))
        return -1;
    (void)num_layers;
    const int64_t src_heads = heads_per_card(kv_heads, src_tp); /* heads per prefill card */
    const int64_t dst_heads = heads_per_card(kv_heads, dst_tp); /* heads per decode card */
    const int64_t src_copies = cards_per_head(kv_heads, src_tp);
    const int64_t dst_copies = cards_per_head(kv_heads, dst_tp);
    const int64_t C = num_components;
    const int64_t D = head_dim;

    for (int32_t r = 0; r < num_requests; ++r) {
        const int64_t n = seq_lens[r];
        for (int64_t l = layer_begin; l < layer_end; ++l) {
            for (int64_t c = 0; c < C; ++c) {
                for (int64_t t = 0; t < n; ++t) {
                    /* prefill side: block table entry t / Bp, offset t % Bp */
                    const int64_t sblk = src_bt[src_off[r] + t / src_block];
                    const int64_t soff = t % src_block;
                    /* decode side: slot = block_ids[t // Bd] * Bd + t % Bd */
                    const int64_t dblk = dst_bt[dst_off[r] + t / dst_block];
                    const int64_t doff = t % dst_block;
                    for (int64_t h = 0; h < kv_heads; ++h)
                    for (int64_t k = 0; k < dst_copies; ++k) {
                        /* head h is read from the first prefill card holding it ... */
                        const int64_t sp = (h / src_heads) * src_copies;
                        const int64_t sh = h % src_heads;
                        /* ... and goes to the k-th decode card holding it */
                        const int64_t dp = (h / dst_heads) * dst_copies + k;
                        const int64_t dh = h % dst_heads;
                        for (int64_t e = 0; e < D; ++e) {
                            const int64_t s_elem =
                                ((((l * C + c) * src_num_blocks + sblk) * src_block + soff)
                                     * src_heads + sh) * D + e;
                            const int64_t d_elem =
                                ((((l * C + c) * dst_num_blocks + dblk) * dst_block + doff)
                                     * dst_heads + dh) * D + e;
                            const uint8_t *from = src_pools[sp] + s_elem * elem_bytes;
                            uint8_t *to = dst_pools[dp] + d_elem * elem_bytes;
                            for (int32_t b = 0; b < elem_bytes; ++b)
                                to[b] = from[b];
                        }
                    }
                }
            }
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * dtype-converting relayout (page "PD 分离与 KV 传输", section "布局转换",
 * item on data types: one side keeps BF16 KV, the other FP8 KV, and the
 * conversion belongs around the transfer). The page fixes neither the FP8
 * format nor the scale; the readings taken here:
 *   - FP8 is E4M3 as in the OCP 8-bit floating point specification: 1 sign,
 *     4 exponent bits (bias 7), 3 mantissa bits, subnormals, no infinities,
 *     S.1111.111 is NaN, largest finite value 448;
 *   - quantize:   q = E4M3(x * fl32(1 / s)), round to nearest, ties to even,
 *     magnitudes above 448 (and infinities) saturate to +-448, a NaN x gives
 *     S.1111.111 with the sign of x;
 *   - dequantize: y = BF16(float(q) * s), round to nearest, ties to even, a
 *     NaN code gives sign | 0x7FC0 with the sign of the code;
 *   - s is one positive scale per (layer, component), or per (layer,
 *     component, KV head).
 * All products are single fp32 multiplications (as the C float type gives).
 * ------------------------------------------------------------------------- */
#include <math.h>
#include <string.h>

#define KVO_BF16 1
#define KVO_E4M3 2

/* Exact value of the non-negative E4M3 code c (0..126), from its fields. */
static double e4m3_magnitude(int c)
{
    const int e = c >> 3, m = c & 7;
    if (e == 0)
        return ldexp((double)m, -9);         /* subnormal: m/8 * 2^(1-7) */
    return ldexp((double)(8 + m), e - 10);   /* (1 + m/8) * 2^(e-7) */
}

float kvo_e4m3_decode(uint8_t code)
{
    if ((code & 0x7F) == 0x7F)
        return NAN;
    const double v = e4m3_magnitude(code & 0x7F);
    return (float)((code & 0x80) ? -v : v);
}

uint8_t kvo_e4m3_encode(float v)
{
    uint32_t bits;
    memcpy(&bits, &v, 4);
    const uint8_t sign = (bits >> 31) ? 0x80 : 0x00;
    if (v != v)
        return sign | 0x7F;
    const double a = fabs((double)v);
    if (a >= 448.0)
        return sign | 0x7E;
    /* largest code whose value does not exceed a (values grow with the code) */
    int lo = 0, hi = 126;
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (e4m3_magnitude(mid) <= a)
            lo = mid;
        else
            hi = mid - 1;
    }
    const double below = a - e4m3_magnitude(lo);
    const double above = e4m3_magnitude(lo + 1) - a;
    int code;
    if (below < above)
        code = lo;
    else if (above < below)
        code = lo + 1;
    else
        code = (lo & 1) ? lo + 1 : lo;      /* tie: the even code */
    return (uint8_t)(sign | code);
}

/* fp32 -> bf16 bits, nearest with ties to even, by comparing the two
 * neighbouring bf16 values (the upper neighbour of the largest finite bf16
 * is taken as 2^128, which rounds to infinity). */
uint16_t kvo_bf16_encode(float v)
{
    uint32_t bits;
    memcpy(&bits, &v, 4);
    const uint16_t sign = (uint16_t)((bits >> 16) & 0x8000);
    if (v != v)
        return sign | 0x7FC0;
    const uint32_t mag = bits & 0x7FFFFFFFu;
    const uint32_t lo = mag & 0xFFFF0000u;
    if (lo == mag)
        return (uint16_t)(sign | (lo >> 16));
    float flo;
    memcpy(&flo, &lo, 4);
    const double vlo = (double)flo;
    double vhi;
    if (lo == 0x7F7F0000u) {
        vhi = ldexp(1.0, 128);
    } else {
        const uint32_t hib = lo + 0x10000u;
        float fhi;
        memcpy(&fhi, &hib, 4);
        vhi = (double)fhi;
    }
    const double a = fabs((double)v);
    uint32_t pick;
    if (a - vlo < vhi - a)
        pick = lo;
    else if (vhi - a < a - vlo)
        pick = lo + 0x10000u;
    else
        pick = ((lo >> 16) & 1) ? lo + 0x10000u : lo;
    return (uint16_t)(sign | (pick >> 16));
}

/* The relayout of kvo_relayout() with a dtype change on the way: src_dtype
 * and dst_dtype are KVO_BF16 / KVO_E4M3 (one of each); elements are 2 bytes
 * (little-endian) for BF16 and 1 byte for E4M3; scales[] has L*C entries, or
 * L*C*H when per_head is 1. Returns 0, or -1 for an unsupported request. */
int kvo_relayout_convert(int32_t layer_begin, int32_t layer_end,
                         int32_t num_layers, int32_t num_components,
                         int32_t kv_heads, int32_t head_dim,
                         int32_t src_dtype, int32_t dst_dtype,
                         int32_t per_head, const float *scales,
                         int32_t src_tp, int32_t dst_tp,
                         int32_t src_block, int32_t dst_block,
                         int64_t src_num_blocks, int64_t dst_num_blocks,
                         const uint8_t *const *src_pools, uint8_t *const *dst_pools,
                         int32_t num_requests, const int32_t *seq_lens,
                         const int64_t *src_off, const int32_t *src_bt,
                         const int64_t *dst_off, const int32_t *dst_bt)
{
    if (!tp_ok(kv_heads, src_tp) || !tp_ok(kv_heads, dst_tp))
        return -1;
    if (!((src_dtype == KVO_BF16 && dst_dtype == KVO_E4M3) ||
          (src_dtype == KVO_E4M3 && dst_dtype == KVO_BF16)))
        return -1;
    (void)num_layers;
    const int64_t src_es = src_dtype == KVO_BF16 ? 2 : 1;
    const int64_t dst_es = dst_dtype == KVO_BF16 ? 2 : 1;
    const int64_t src_heads = heads_per_card(kv_heads, src_tp);
    const int64_t dst_heads = heads_per_card(kv_heads, dst_tp);
    const int64_t src_copies = cards_per_head(kv_heads, src_tp);
    const int64_t dst_copies = cards_per_head(kv_heads, dst_tp);
    const int64_t C = num_components;
    const int64_t D = head_dim;

    for (int32_t r = 0; r < num_requests; ++r) {
        const int64_t n = seq_lens[r];
        for (int64_t l = layer_begin; l < layer_end; ++l) {
            for (int64_t c = 0; c < C; ++c) {
                for (int64_t t = 0; t < n; ++t) {
                    const int64_t sblk = src_bt[src_off[r] + t / src_block];
                    const int64_t soff = t % src_block;
                    const int64_t dblk = dst_bt[dst_off[r] + t / dst_block];
                    const int64_t doff = t % dst_block;
                    for (int64_t h = 0; h < kv_heads; ++h)
                    for (int64_t k = 0; k < dst_copies; ++k) {
                        const int64_t sp = (h / src_heads) * src_copies;
                        const int64_t sh = h % src_heads;
                        const int64_t dp = (h / dst_heads) * dst_copies + k;
                        const int64_t dh = h % dst_heads;
                        const float s = per_head ? scales[(l * C + c) * kv_heads + h]
                                                 : scales[l * C + c];
                        for (int64_t e = 0; e < D; ++e) {
                            const int64_t s_elem =
                                ((((l * C + c) * src_num_blocks + sblk) * src_block + soff)
                                     * src_heads + sh) * D + e;
                            const int64_t d_elem =
                                ((((l * C + c) * dst_num_blocks + dblk) * dst_block + doff)
                                     * dst_heads + dh) * D + e;
                            const uint8_t *from = src_pools[sp] + s_elem * src_es;
                            uint8_t *to = dst_pools[dp] + d_elem * dst_es;
                            if (src_dtype == KVO_BF16) {
                                const uint32_t xb = ((uint32_t)from[0] | ((uint32_t)from[1] << 8)) << 16;
                                float x;
                                memcpy(&x, &xb, 4);
                                if (x != x) {
                                    /* NaN keeps the input's sign (the sign of a NaN
                                     * product is not fixed by IEEE 754) */
                                    to[0] = (uint8_t)(((xb >> 24) & 0x80) | 0x7F);
                                } else {
                                    const float inv = 1.0f / s;
                                    const float y = x * inv;
                                    to[0] = kvo_e4m3_encode(y);
                                }
                            } else {
                                uint16_t b;
                                if ((from[0] & 0x7F) == 0x7F) {
                                    b = (uint16_t)(((from[0] & 0x80) << 8) | 0x7FC0);
                                } else {
                                    const float x = kvo_e4m3_decode(from[0]);
                                    const float y = x * s;
                                    b = kvo_bf16_encode(y);
                                }
                                to[0] = (uint8_t)(b & 0xFF);
                                to[1] = (uint8_t)(b >> 8);
                            }
                        }
                    }
                }
            }
        }
    }
    return 0;
}

/* Element-wise helpers over arrays (used by the tests' pins). */
void kvo_e4m3_encode_array(const float *x, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kvo_e4m3_encode(x[i]);
}

void kvo_e4m3_decode_array(const uint8_t *x, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kvo_e4m3_decode(x[i]);
}

void kvo_bf16_encode_array(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kvo_bf16_encode(x[i]);
}

/* ---------------------------------------------------------------------------
 * Any physical layout (page "PD 分离与 KV 传输", section "布局转换": attention
 * backends differ in physical layout -- whether K and V are stored together,
 * and the order of the head and token dimensions). Reading taken: each side
 * is, per (TP shard, layer, component), a strided view [block][token][head][dim]
 * whose head rows (dim) are contiguous; base[(shard * L + layer) * C + comp]
 * is the address of element [0][0][0][0] of that view, and the block, token
 * and head strides (in bytes) are shared by all views of a side. The standard
 * layout [L][C][N][B][H/T][D] is one such choice; per-layer buffers, K and V
 * in separate buffers, K/V interleaved per block and head-major blocks are
 * others, and so is a contiguous [tokens][heads][dim] staging buffer (pd.py's
 * gathered shape) seen as blocks of one token.
 *
 * src_dtype / dst_dtype: 0 (elements copied as elem_bytes raw bytes; both
 * must then be 0) or KVO_BF16 / KVO_E4M3 (converted as kvo_relayout_convert).
 * ------------------------------------------------------------------------- */
static void convert_element(int32_t src_dtype, const uint8_t *from, uint8_t *to, float s)
{
    if (src_dtype == KVO_BF16) {
        const uint32_t xb = ((uint32_t)from[0] | ((uint32_t)from[1] << 8)) << 16;
        float x;
        memcpy(&x, &xb, 4);
        if (x != x) {
            to[0] = (uint8_t)(((xb >> 24) & 0x80) | 0x7F);
        } else {
            const float inv = 1.0f / s;
            to[0] = kvo_e4m3_encode(x * inv);
        }
    } else {
        uint16_t b;
        if ((from[0] & 0x7F) == 0x7F) {
            b = (uint16_t)(((from[0] & 0x80) << 8) | 0x7FC0);
        } else {
            b = kvo_bf16_encode(kvo_e4m3_decode(from[0]) * s);
        }
        to[0] = (uint8_t)(b & 0xFF);
        to[1] = (uint8_t)(b >> 8);
    }
}

int kvo_relayout_general(int32_t layer_begin, int32_t layer_end,
                         int32_t num_layers, int32_t num_components,
                         int32_t kv_heads, int32_t head_dim,
                         int32_t src_dtype, int32_t dst_dtype, int32_t elem_bytes,
                         int32_t per_head, const float *scales,
                         int32_t src_tp, int32_t dst_tp,
                         int32_t src_block, int32_t dst_block,
                         const uint64_t *src_base, int64_t s_block_stride,
                         int64_t s_token_stride, int64_t s_head_stride,
                         const uint64_t *dst_base, int64_t d_block_stride,
                         int64_t d_token_stride, int64_t d_head_stride,
                         int32_t num_requests, const int32_t *seq_lens,
                         const int64_t *src_off, const int32_t *src_bt,
                         const int64_t *dst_off, const int32_t *dst_bt)
{
    if (!tp_ok(kv_heads, src_tp) || !tp_ok(kv_heads, dst_tp))
        return -1;
    const int converting = src_dtype != 0;
    if (converting && !((src_dtype == KVO_BF16 && dst_dtype == KVO_E4M3) ||
                        (src_dtype == KVO_E4M3 && dst_dtype == KVO_BF16)))
        return -1;
    if (!converting && dst_dtype != 0)
        return -1;
    const int64_t src_es = !converting ? elem_bytes : (src_dtype == KVO_BF16 ? 2 : 1);
    const int64_t dst_es = !converting ? elem_bytes : (dst_dtype == KVO_BF16 ? 2 : 1);
    const int64_t src_heads = heads_per_card(kv_heads, src_tp);
    const int64_t dst_heads = heads_per_card(kv_heads, dst_tp);
    const int64_t src_copies = cards_per_head(kv_heads, src_tp);
    const int64_t dst_copies = cards_per_head(kv_heads, dst_tp);
    const int64_t C = num_components;
    const int64_t L = num_layers;

    for (int32_t r = 0; r < num_requests; ++r) {
        const int64_t n = seq_lens[r];
        for (int64_t l = layer_begin; l < layer_end; ++l) {
            for (int64_t c = 0; c < C; ++c) {
                for (int64_t t = 0; t < n; ++t) {
                    const int64_t sblk = src_bt[src_off[r] + t / src_block];
                    const int64_t soff = t % src_block;
                    const int64_t dblk = dst_bt[dst_off[r] + t / dst_block];
                    const int64_t doff = t % dst_block;
                    for (int64_t h = 0; h < kv_heads; ++h)
                    for (int64_t k = 0; k < dst_copies; ++k) {
                        const int64_t sp = (h / src_heads) * src_copies;
                        const int64_t sh = h % src_heads;
                        const int64_t dp = (h / dst_heads) * dst_copies + k;
                        const int64_t dh = h % dst_heads;
                        const uint8_t *src_row = (const uint8_t *)(uintptr_t)
                            src_base[(sp * L + l) * C + c] + sblk * s_block_stride +
                            soff * s_token_stride + sh * s_head_stride;
                        uint8_t *dst_row = (uint8_t *)(uintptr_t)
                            dst_base[(dp * L + l) * C + c] + dblk * d_block_stride +
                            doff * d_token_stride + dh * d_head_stride;
                        const float s = !converting ? 0.0f
                                        : per_head ? scales[(l * C + c) * kv_heads + h]
                                                   : scales[l * C + c];
                        for (int64_t e = 0; e < head_dim; ++e) {
                            const uint8_t *from = src_row + e * src_es;
                            uint8_t *to = dst_row + e * dst_es;
                            if (!converting) {
                                for (int64_t b = 0; b < elem_bytes; ++b)
                                    to[b] = from[b];
                            } else {
                                convert_element(src_dtype, from, to, s);
                            }
                        }
                    }
                }
            }
        }
    }
    return 0;
}
