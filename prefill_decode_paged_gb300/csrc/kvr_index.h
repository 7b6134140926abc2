// kvr_index.h -- work decomposition and address arithmetic of the relayout kernel.
//
// Compiled both by nvcc (into the kernel) and by a host compiler (plan
// construction; the test emulator that walks every launch on the CPU), so it
// holds plain structs and inline functions only.
//
// Work decomposition. A work ITEM is one tile of one request's tokens,
// [t0, t0 + ntok), for all components and all KV heads. Tiles start at
// multiples of the tile size T, itself a multiple of the decode block size
// Bd (T = Bd unless decode blocks are small, then several decode blocks per
// tile). One launch covers (layers of the launch) x items x slices TASKS, one
// CTA per task; a slice is a contiguous part of the item's 16-byte chunks, so
// a per-layer launch with few items still fills the GPU.
//
// Inside an item, ROW r (one head row: D elements) is ordered
// [token o][component c][head h], and chunk q = r * row_chunks + k is the
// k-th UNIT of row r. A decode side with more TP shards than KV heads holds
// each head on Td/H consecutive shards: a row's decode rows are then
// [token][component][head][decode copy] (table rows r * Td/H + copy), and
// each unit is loaded once and stored to every copy.
// A unit is 16 bytes of the row when elements are copied as bits; when the
// element type changes on the way (BF16 <-> FP8 E4M3) it is 16 elements: 32
// bytes on the BF16 side, 16 on the FP8 side. Consecutive
// threads read and write consecutive units of one head row, and the rows of
// one token follow each other.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define KVR_HD __host__ __device__ __forceinline__
#else
#define KVR_HD inline
#endif

#ifndef KVR_MAX_TP
#define KVR_MAX_TP 16
#endif

// Division by a run-time invariant d >= 1 for dividends n < 2^31, by one
// 32x32->64 multiply and a shift (Granlund & Montgomery, "Division by
// invariant integers using multiplication", PLDI 1994, Theorem 4.2 with
// N = 31): with l = ceil(log2 d) and m = ceil(2^(31+l) / d), which fits in
// 32 bits, floor(n / d) = floor(n * m / 2^(31+l)) for all 0 <= n < 2^31.
struct KvrDiv {
    uint32_t d;
    uint32_t mul;
    uint32_t shift;

    KVR_HD uint32_t div(uint32_t n) const {
        return (uint32_t)(((uint64_t)n * mul) >> shift);
    }
};

inline KvrDiv kvr_make_div(uint32_t d) {
    uint32_t l = 0;
    while ((1ull << l) < d) ++l;
    const uint64_t num = 1ull << (31 + l);
    KvrDiv r;
    r.d = d;
    r.mul = (uint32_t)((num + d - 1) / d);
    r.shift = 31 + l;
    return r;
}

// One work item: a token tile of one request. 16 bytes.
struct KvrItem {
    int32_t sbt_off;    // index of the request's first prefill block id in the flat table
    int32_t dbt_off;    // index of the request's first decode block id in the flat table
    int32_t t0;         // first token of the tile (a multiple of the tile size)
    int32_t ntok;       // tokens in the tile, >= 1
};

// Element conversion done on the way.
enum KvrConv : int32_t {
    KVR_CONV_NONE = 0,          // bit copy of es-byte elements
    KVR_CONV_BF16_TO_E4M3 = 1,  // quantize: q = E4M3(x * (1/s))
    KVR_CONV_E4M3_TO_BF16 = 2,  // dequantize: y = BF16(q * s)
};

struct KvrGeom {
    int32_t L, C, H, Hp, Hd, Bp, Bd;
    int32_t src_row_bytes;      // D * source element bytes, a multiple of 16
    int32_t dst_row_bytes;      // D * destination element bytes, a multiple of 16
    int32_t row_chunks;         // units per row
    int32_t src_unit_bytes;     // bytes one unit reads (16, or 32 from a BF16 side)
    int32_t dst_unit_bytes;     // bytes one unit writes (16, or 32 to a BF16 side)
    int32_t conv;               // KvrConv
    int32_t per_head;           // conversion scales per (layer, component[, head])
    KvrDiv div_rc;
    KvrDiv div_Hx;              // by Hx (below): decode head rows per (token, component)
    KvrDiv div_C;
    KvrDiv div_sgrp;            // by Hp * dcopies: rows of one prefill shard's heads
    KvrDiv div_Hd, div_Bp, div_Bd;
    // byte strides of each side's [block][token][head] view (rows are contiguous)
    int64_t s_block_stride, s_token_stride, s_head_stride;
    int64_t d_block_stride, d_token_stride, d_head_stride;
    // TP degrees above H replicate heads: scopies = Tp/H prefill shards (the
    // first is read) and dcopies = Td/H decode shards (all written) hold one
    // head; 1 when the side's TP degree divides H. Hx = H * dcopies rows per
    // (token, component).
    int32_t scopies, dcopies, Hx;
    KvrDiv div_dcop;            // by dcopies
    int32_t win_rows;           // prefill rows per row window when dcopies > 1
};

// Kernel parameter block (passed by value as a __grid_constant__).
struct KvrArgs {
    KvrGeom g;
    const KvrItem *items;
    const int32_t *sbt;                 // flat prefill block ids
    const int32_t *dbt;                 // flat decode block ids
    const float *factors;               // conversion: 1/s (quantize) or s (dequantize)
    const uint64_t *src_base;           // [Tp][L][C] addresses of the prefill views
    const uint64_t *dst_base;           // [Td][L][C] addresses of the decode views
    int32_t layer0;                     // first layer of this launch
    int32_t slices;                     // tasks per item
    int32_t no_wait;                    // 1: wait for the previous grid after the copies, not
                                        // before them (the caller's call)
    uint32_t tasks_per_layer;           // n_items * slices
    KvrDiv div_tasks_per_layer, div_slices;
    uint32_t prefetch_ctas;             // bit copy, prefetching instance, no replicated
                                        // heads: CTAs below this index prefetch their rows
                                        // (all: 0xFFFFFFFF)
#ifdef KVR_DEVICE_CHECKS
    // Checked builds only: [lo, hi) byte ranges the prefill rows (the first
    // n_src_regions pairs) and decode rows (the next n_dst_regions) must lie in;
    // NULL: no check. A row outside them sets *check_error and is dropped.
    const uint64_t *check_regions;
    int32_t n_src_regions, n_dst_regions;
    unsigned int *check_error;
#endif
};

// Does [a, a + bytes) lie inside one of the n [lo, hi) pairs of `reg`?
KVR_HD bool kvr_span_in(const uint64_t *reg, int32_t n, uint64_t a, uint64_t bytes) {
    for (int32_t k = 0; k < n; ++k)
        if (a >= reg[2 * k] && a + bytes <= reg[2 * k + 1]) return true;
    return false;
}

// Launch modes (kernel instances).
enum KvrMode : int32_t {
    KVR_MODE_WHOLE = 0,           // whole prompt or a long layer range: wait, then copy
    KVR_MODE_LAYER = 1,           // per layer: row table before the wait
    KVR_MODE_LAYER_PREFETCH = 2,  // per layer, ordered, one wave: also prefetch the rows to L2
};

// Task -> (layer, item, chunk range [q0, q1) of the item). Chunks are units of
// the prefill rows: with replicated decode heads each is stored to every copy.
// W = 2 (threads move pairs of adjacent units; rows hold an even number of
// units): the slices split the item's pairs, so q0 and q1 are even.
template <int W = 1>
KVR_HD void kvr_task(const KvrArgs &a, uint32_t task, const KvrItem *items, int32_t *layer,
                     KvrItem *item, uint32_t *q0, uint32_t *q1) {
    const uint32_t lt = a.div_tasks_per_layer.div(task);
    const uint32_t rem = task - lt * a.tasks_per_layer;
    const uint32_t idx = a.div_slices.div(rem);
    const uint32_t slice = rem - idx * (uint32_t)a.slices;
    const KvrItem it = items[idx];
    const uint64_t total = (uint64_t)it.ntok * a.g.C * a.g.H * a.g.row_chunks;
    *layer = a.layer0 + (int32_t)lt;
    *item = it;
    if (W == 1) {
        *q0 = (uint32_t)(total * slice / (uint32_t)a.slices);
        *q1 = (uint32_t)(total * (slice + 1) / (uint32_t)a.slices);
    } else {
        *q0 = 2u * (uint32_t)((total / 2) * slice / (uint32_t)a.slices);
        *q1 = 2u * (uint32_t)((total / 2) * (slice + 1) / (uint32_t)a.slices);
    }
}

// Row r of an item -> address of its prefill row, address of its decode row,
// and the index of its conversion scale. REP: a side's TP degree exceeds H
// (scopies or dcopies above 1); without it every head sits on one shard per
// side and the row's head is hv itself, which keeps the index chain of the
// plain relayout as short as it can be.
template <bool REP>
KVR_HD void kvr_row(const KvrGeom &g, int32_t layer, const KvrItem &it, const int32_t *sbt,
                    const int32_t *dbt, const uint64_t *src_base, const uint64_t *dst_base,
                    uint32_t r, uint64_t *saddr, uint64_t *daddr, uint32_t *fidx) {
    const uint32_t oc = g.div_Hx.div(r);
    // head h = hv / dcopies, copy hv % dcopies (Hx = H without replication)
    const uint32_t hv = r - oc * (uint32_t)(REP ? g.Hx : g.H);
    const uint32_t o = g.div_C.div(oc);
    const uint32_t c = oc - o * (uint32_t)g.C;
    const uint32_t t = (uint32_t)it.t0 + o;
    // prefill side: logical block t / Bp of the request, row t % Bp in it
    const uint32_t sbi = g.div_Bp.div(t);
    const uint32_t so = t - sbi * (uint32_t)g.Bp;
    const int64_t sb = sbt[it.sbt_off + (int32_t)sbi];
    // decode side: logical block t / Bd, row t % Bd
    const uint32_t dbi = g.div_Bd.div(t);
    const uint32_t dof = t - dbi * (uint32_t)g.Bd;
    const int64_t db = dbt[it.dbt_off + (int32_t)dbi];
    // head h: prefill shard (h / Hp) * scopies (the first that holds it), local
    // h % Hp; decode shard (h / Hd) * dcopies + copy, local h % Hd, which is
    // hv / Hd and hv % Hd (Hd = 1 whenever dcopies > 1)
    uint32_t h, s_sh, s_loc;
    if (REP) {
        const uint32_t sg = g.div_sgrp.div(hv);
        s_loc = g.div_dcop.div(hv - sg * (uint32_t)g.Hp * (uint32_t)g.dcopies);
        s_sh = sg * (uint32_t)g.scopies;
        h = sg * (uint32_t)g.Hp + s_loc;
    } else {
        h = hv;
        s_sh = g.div_sgrp.div(h);                     // Hp * dcopies = Hp
        s_loc = h - s_sh * (uint32_t)g.Hp;
    }
    const uint32_t d_sh = g.div_Hd.div(hv);
    const uint32_t d_loc = hv - d_sh * (uint32_t)g.Hd;
    const uint32_t plane = (uint32_t)layer * (uint32_t)g.C + c;
    const uint64_t sv = src_base[s_sh * (uint32_t)g.L * (uint32_t)g.C + plane];
    const uint64_t dv = dst_base[d_sh * (uint32_t)g.L * (uint32_t)g.C + plane];
    *saddr = sv + (uint64_t)(sb * g.s_block_stride + (int64_t)so * g.s_token_stride +
                             (int64_t)s_loc * g.s_head_stride);
    *daddr = dv + (uint64_t)(db * g.d_block_stride + (int64_t)dof * g.d_token_stride +
                             (int64_t)d_loc * g.d_head_stride);
    *fidx = g.per_head ? plane * (uint32_t)g.H + h : plane;
}

// Whether a plan's rows need the replicated-head arithmetic of kvr_row.
KVR_HD bool kvr_replicated(const KvrGeom &g) { return g.scopies > 1 || g.dcopies > 1; }
