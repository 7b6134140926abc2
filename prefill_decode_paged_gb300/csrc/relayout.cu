// relayout.cu -- fused gather -> head re-shard -> scatter of paged KV cache (sm_103a).
//
// One kernel does the whole hand-off of the page "PD 分离与 KV 传输"
// (ai-infra-handbooks, serving/distributed/pd-disagg; sections "实现" and
// "布局转换"): each 16-byte chunk of a head row is read from the prefill
// shard that holds the head, at the row the prefill block table gives for
// the token, and written to the decode shard that holds the head, at the row
// the decode block table gives. There is no intermediate buffer: the gather,
// the TP re-shard and the scatter are one load and one store per chunk. With
// more TP shards than KV heads, a head is read from the first prefill shard
// that holds it and stored to every decode shard that holds it; with a dtype
// change (BF16 <-> FP8 E4M3), each unit of 16 elements is converted between
// its load and its store.
//
// It is data movement bound by HBM bandwidth (no tensor cores): every chunk
// is read once and written once, so the DRAM traffic floor is the KV bytes of
// the prompts read plus written. The kernel keeps several independent 16-byte
// loads in flight per thread before their stores, uses streaming cache hints
// on both sides (neither the prefill rows nor the decode rows are touched
// again by this kernel), and opts into programmatic dependent launch so that
// back-to-back per-layer launches overlap their launch latency, block-table
// reads and (ordered launches of one wave) an L2 prefetch of their prefill
// rows with the previous launch's tail. Built with KVR_DEVICE_CHECKS (tests),
// it also checks every row against the plan's pools before touching it.
#include <cuda_runtime.h>
#include <string.h>

#include <algorithm>
#include <new>

#include "kv_relayout.h"
#include "kvr_convert.cuh"
#include "kvr_index.h"
#include "plan.h"

struct kvr_plan {
    KvrHostPlan host;
    void *dev_meta = nullptr;       // items, view bases, block ids, factors
    const KvrItem *dev_items = nullptr;
    const uint64_t *dev_src_base = nullptr;
    const uint64_t *dev_dst_base = nullptr;
    const int32_t *dev_sbt = nullptr;
    const int32_t *dev_dbt = nullptr;
    const float *dev_factors = nullptr;
    int device = 0;
#ifdef KVR_DEVICE_CHECKS
    uint64_t *dev_regions = nullptr;      // checked builds: the pool regions, then the error word
    unsigned int *dev_check_error = nullptr;
#endif
};

namespace {

__device__ __forceinline__ uint4 load_stream(const unsigned char *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Fetch [addr, addr + bytes) into L2 (a hint: no completion to wait for, no
// register written; bytes a multiple of 16, addr 16-byte aligned). The SM's
// bulk copy unit takes these requests one at a time.
__device__ __forceinline__ void prefetch_l2(uint64_t addr, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(addr), "r"(bytes) : "memory");
}

// The same hint as one prefetch.global.L2 per 128-byte line of [addr, addr +
// bytes), from the thread that computed the row: no bulk copy unit in the way,
// so a per-layer CTA is ready to run sooner (256 bulk requests per CTA took ~1
// us to issue), but the rows reach L2 later. Measured on ordered 70B layers:
// the converting launches gain (BF16 -> FP8 5236 -> 5302, FP8 -> BF16 4295 ->
// 4591 GB/s), the bit copy loses (6204 -> 6035), so it keeps the bulk form.
// The lines hold bytes of the row, so they lie in its pages: nothing is touched
// outside the pools.
// LOAD_FIRST: the row's first line is asked for by a load whose value is
// dropped instead of a prefetch (BF16 -> FP8 instances; their 256-byte rows
// take one load and one prefetch): 70B ordered layers 5569 -> 5629 GB/s, and
// 5238 -> 5380 on pools the driver placed after other allocations, where the
// prefetches alone lose more (the FP8 -> BF16 and bit-copy instances gain
// nothing from it). The load is volatile, a relaxed system-scope access in
// the PTX memory model: it may race with a producer still writing the row
// without undefined behaviour, and its value is never used.
template <bool LOAD_FIRST>
__device__ __forceinline__ void prefetch_l2_lines(uint64_t addr, uint32_t bytes) {
    uint64_t p = addr & ~(uint64_t)127;
    if (LOAD_FIRST) {
        asm volatile("{ .reg .u32 t; ld.volatile.global.u32 t, [%0]; }" ::"l"(addr));
        p += 128;
    }
    for (; p < addr + bytes; p += 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

#ifdef KVR_DEVICE_CHECKS
// Checked builds: a row whose prefill or decode bytes leave the plan's pool
// regions is flagged in *check_error and dropped (both addresses 0: nothing
// is read, prefetched or written for it).
__device__ __forceinline__ void kvr_check_row(const KvrArgs &a, uint64_t *sa, uint64_t *da) {
    if (a.check_regions == nullptr) return;
    if (!kvr_span_in(a.check_regions, a.n_src_regions, *sa, (uint64_t)a.g.src_row_bytes) ||
        !kvr_span_in(a.check_regions + 2 * a.n_src_regions, a.n_dst_regions, *da,
                     (uint64_t)a.g.dst_row_bytes)) {
        atomicOr(a.check_error, 1u);
        *sa = 0;
        *da = 0;
    }
}
#define KVR_CHECK_ROW(a, sa, da) kvr_check_row((a), &(sa), &(da))
#define KVR_SRC_DROPPED(row) ((row).x == 0)
#define KVR_DST_DROPPED(row) ((row).y == 0)
#else
#define KVR_CHECK_ROW(a, sa, da) ((void)0)
#define KVR_SRC_DROPPED(row) false
#define KVR_DST_DROPPED(row) false
#endif

// 32 bytes (two 16-byte pieces) with one load / one store: p 32-byte aligned.
__device__ __forceinline__ void load_stream32(const unsigned char *p, uint4 *lo, uint4 *hi) {
    asm volatile(
        "ld.global.nc.L1::no_allocate.L2::256B.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(lo->x), "=r"(lo->y), "=r"(lo->z), "=r"(lo->w), "=r"(hi->x), "=r"(hi->y),
          "=r"(hi->z), "=r"(hi->w)
        : "l"(p));
}

__device__ __forceinline__ void store_stream32(unsigned char *p, const uint4 &lo,
                                               const uint4 &hi) {
    asm volatile("st.global.cs.v8.u32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p),
                 "r"(lo.x), "r"(lo.y), "r"(lo.z), "r"(lo.w), "r"(hi.x), "r"(hi.y), "r"(hi.z),
                 "r"(hi.w)
                 : "memory");
}

__device__ __forceinline__ void store_stream(unsigned char *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// CTAs per SM each converting instance is compiled for (caps its registers:
// 256 threads x 64 registers fill an SM's register file 4 times); 0 leaves the
// bit copy's registers to the compiler. The dequantizer measured faster at 4
// CTAs (64 registers) than at 5 (48 registers, which spills); a minimum of 4
// for the bit copy (the 64 registers it takes anyway) cost 2-7 % (70B: 6945 ->
// 6814 GB/s whole-prompt, 6193 -> 6000 per layer).
#ifndef KVR_MIN_CTAS_DEQUANT
#define KVR_MIN_CTAS_DEQUANT 4
#endif
constexpr int kvr_min_ctas(int U, int CONV) {
    return CONV == KVR_CONV_E4M3_TO_BF16            ? KVR_MIN_CTAS_DEQUANT
           : CONV == KVR_CONV_BF16_TO_E4M3 && U <= 2 ? 5
           : CONV == KVR_CONV_BF16_TO_E4M3           ? 4
                                                     : 0;
}

// U: units each thread keeps in flight before its stores. CONV: KvrConv.
// MODE: KVR_MODE_WHOLE, KVR_MODE_LAYER or KVR_MODE_LAYER_PREFETCH. Per-layer
// modes build the first row window before waiting for the previous grid
// (hides the block-table reads in the previous launch's tail; whole-prompt
// launches wait first, which measured 1.7 % faster there); the prefetching
// one also asks L2 for those rows before the wait.
// A unit reads NL and writes NS 16-byte pieces (1 and 1 for a bit copy).
// REP: the plan replicates heads (a TP degree above H; see kvr_row).
// W: units per access. W = 2 (plans whose rows hold an even number of units and
// lie 32 bytes aligned; kvr_launch_pairs): each thread moves a pair of adjacent
// units of one row with 32-byte loads and stores, U / 2 pairs in flight: one
// row lookup and address per pair halves the index work per byte (70B, ordered
// per-layer launches: BF16 -> FP8 5281 -> 5568, FP8 -> BF16 4605 -> 5513 GB/s;
// whole-prompt: quantizing 6901 -> 7080, Qwen3-32B 4 x 32K bit copy 6864 ->
// 6956; replicated MLA latent, TP8 -> TP8: 6678 -> 6767).
template <int U, int CONV, int MODE, bool REP, int W>
__global__ void __launch_bounds__(KVR_THREADS, kvr_min_ctas(U, CONV))
    kvr_relayout_kernel(const __grid_constant__ KvrArgs a) {
    static_assert(W == 1 || W == 2, "one unit or a pair of units per access");
    constexpr bool EARLY = MODE != KVR_MODE_WHOLE;
    constexpr bool PF = MODE == KVR_MODE_LAYER_PREFETCH;
    constexpr int NL = CONV == KVR_CONV_BF16_TO_E4M3 ? 2 : 1;
    constexpr int NS = CONV == KVR_CONV_E4M3_TO_BF16 ? 2 : 1;
    constexpr uint32_t SU = 16u * NL, DU = 16u * NS;   // bytes read / written per unit
    // (prefill row address, decode row address) of the rows this CTA copies,
    // and the rows' conversion factors
    __shared__ ulonglong2 rows[KVR_ROW_WINDOW];
    __shared__ float row_factor[CONV == KVR_CONV_NONE ? 1 : KVR_ROW_WINDOW];

    // Wait for the grid this launch follows in its stream before touching any
    // pool, then let the next launch start early (programmatic dependent
    // launch; both are no-ops without it). Per-layer launches wait later, and
    // let the next launch start only once they have waited: a launch that does
    // not wait first (no_wait) may only begin after everything queued before
    // the last launch that did wait has finished.
    if (!EARLY && !a.no_wait) asm volatile("griddepcontrol.wait;" ::: "memory");
    if (!EARLY || a.no_wait) asm volatile("griddepcontrol.launch_dependents;");

    int32_t layer;
    KvrItem it;
    uint32_t q0, q1;
    kvr_task<W>(a, blockIdx.x, a.items, &layer, &it, &q0, &q1);
    if (q0 >= q1) {
        // a CTA without rows still orders itself after the previous grid (and a
        // launch without the early wait still completes after it)
        if (EARLY || a.no_wait) asm volatile("griddepcontrol.wait;" ::: "memory");
        return;
    }
    const uint32_t rc = (uint32_t)a.g.row_chunks;
    const uint32_t r_end = a.g.div_rc.div(q1 - 1) + 1;

    if constexpr (REP) {
        // Replicated heads: units are those of the prefill rows ([token][component]
        // [head]); the table holds each row's dcopies decode rows, one after
        // another, and a unit is loaded once and stored to every copy.
        const uint32_t dc = (uint32_t)a.g.dcopies;
        const uint32_t wn = (uint32_t)a.g.win_rows;   // prefill rows per window
        bool waited = !EARLY;
        for (uint32_t w0 = a.g.div_rc.div(q0); w0 < r_end; w0 += wn) {
            const uint32_t w1 = min(w0 + wn, r_end);
            const uint32_t t_end = (w1 - w0) * dc;
            for (uint32_t t = threadIdx.x; t < t_end; t += KVR_THREADS) {
                uint32_t fidx;
                uint64_t sa, da;
                kvr_row<true>(a.g, layer, it, a.sbt, a.dbt, a.src_base, a.dst_base,
                              w0 * dc + t, &sa, &da, &fidx);
                KVR_CHECK_ROW(a, sa, da);
                // the first decode copy of each prefill row asks for it (converting
                // instances here; see the plain branch)
                if (PF && CONV != KVR_CONV_NONE && !waited && t - (t / dc) * dc == 0 &&
                    !KVR_SRC_DROPPED(make_ulonglong2(sa, da)))
                    prefetch_l2_lines<CONV == KVR_CONV_BF16_TO_E4M3>(
                        sa, (uint32_t)a.g.src_row_bytes);
                rows[t] = make_ulonglong2(sa, da);
                if (CONV != KVR_CONV_NONE) row_factor[t] = a.factors[fidx];
            }
            if (PF && CONV == KVR_CONV_NONE && !waited) {
                // the first copy of each row this thread built (see the plain branch)
                for (uint32_t t = threadIdx.x; t < t_end; t += KVR_THREADS)
                    if (t - (t / dc) * dc == 0 && !KVR_SRC_DROPPED(rows[t]))
                        prefetch_l2(rows[t].x, (uint32_t)a.g.src_row_bytes);
            }
            if (EARLY && !waited) {
                if (!a.no_wait) {
                    asm volatile("griddepcontrol.wait;" ::: "memory");
                    asm volatile("griddepcontrol.launch_dependents;");
                }
                waited = true;
            }
            __syncthreads();
            const uint32_t qa = max(q0, w0 * rc), qb = min(q1, w1 * rc);
            if constexpr (W == 2) {
                // pairs (q, q + 1), q even, of one prefill row, each loaded once and
                // stored to every decode copy (the plan checked every row's 32-byte
                // alignment)
                constexpr int UP = U > 1 ? U / 2 : 1;
                const uint32_t pa = qa >> 1, pb = qb >> 1;
                for (uint32_t base = pa + threadIdx.x; base < pb; base += UP * KVR_THREADS) {
                    uint4 v[UP][2 * NL];
                    float f[UP];
#pragma unroll
                    for (int k = 0; k < UP; ++k) {
                        const uint32_t pq = base + (uint32_t)k * KVR_THREADS;
                        f[k] = 0.0f;
                        if (pq < pb) {
                            const uint32_t q = pq * 2u;
                            const uint32_t r = a.g.div_rc.div(q);
                            const uint32_t u = q - r * rc;
                            const ulonglong2 p = rows[(r - w0) * dc];
                            if (!KVR_SRC_DROPPED(p)) {
#pragma unroll
                                for (int j = 0; j < NL; ++j)
                                    load_stream32((const unsigned char *)p.x + u * SU + 32u * j,
                                                  &v[k][2 * j], &v[k][2 * j + 1]);
                            }
                            if (CONV != KVR_CONV_NONE) f[k] = row_factor[(r - w0) * dc];
                        }
                    }
#pragma unroll
                    for (int k = 0; k < UP; ++k) {
                        const uint32_t pq = base + (uint32_t)k * KVR_THREADS;
                        if (pq >= pb) continue;
                        const uint32_t q = pq * 2u;
                        const uint32_t r = a.g.div_rc.div(q);
                        const uint32_t u = q - r * rc;
                        const uint32_t ti = (r - w0) * dc;
                        if (KVR_SRC_DROPPED(rows[ti])) continue;
                        if (CONV == KVR_CONV_E4M3_TO_BF16) {
                            // one unit's 32 BF16 bytes at a time (fewer live registers)
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                uint4 lo, hi;
                                dequant16(v[k][h], f[k], &lo, &hi);
                                for (uint32_t c = 0; c < dc; ++c) {
                                    if (KVR_DST_DROPPED(rows[ti + c])) continue;
                                    store_stream32(
                                        (unsigned char *)rows[ti + c].y + u * DU + 32u * h, lo, hi);
                                }
                            }
                        } else {
                            uint4 lo, hi;
                            if (CONV == KVR_CONV_NONE) {
                                lo = v[k][0];
                                hi = v[k][1];
                            } else {
                                lo = quant16(v[k][0], v[k][1], f[k]);
                                hi = quant16(v[k][2], v[k][3], f[k]);
                            }
                            for (uint32_t c = 0; c < dc; ++c) {
                                if (KVR_DST_DROPPED(rows[ti + c])) continue;
                                store_stream32((unsigned char *)rows[ti + c].y + u * DU, lo, hi);
                            }
                        }
                    }
                }
            } else {
                for (uint32_t base = qa + threadIdx.x; base < qb; base += U * KVR_THREADS) {
                    uint4 v[U][NL];
                    float f[U];
#pragma unroll
                    for (int k = 0; k < U; ++k) {
                        const uint32_t q = base + (uint32_t)k * KVR_THREADS;
                        f[k] = 0.0f;
                        if (q < qb) {
                            const uint32_t r = a.g.div_rc.div(q);
                            const uint32_t u = q - r * rc;
                            const ulonglong2 p = rows[(r - w0) * dc];
                            if (!KVR_SRC_DROPPED(p)) {
#pragma unroll
                                for (int j = 0; j < NL; ++j)
                                    v[k][j] =
                                        load_stream((const unsigned char *)p.x + u * SU + 16u * j);
                            }
                            if (CONV != KVR_CONV_NONE) f[k] = row_factor[(r - w0) * dc];
                        }
                    }
                    // the unit's row and offset are recomputed here rather than kept
                    // from the loads (fewer live registers across the loads)
#pragma unroll
                    for (int k = 0; k < U; ++k) {
                        const uint32_t q = base + (uint32_t)k * KVR_THREADS;
                        if (q >= qb) continue;
                        const uint32_t r = a.g.div_rc.div(q);
                        const uint32_t u = q - r * rc;
                        const uint32_t ti = (r - w0) * dc;
                        if (KVR_SRC_DROPPED(rows[ti])) continue;
                        uint4 lo, hi;
                        if (CONV == KVR_CONV_NONE) {
                            lo = v[k][0];
                        } else if (CONV == KVR_CONV_BF16_TO_E4M3) {
                            lo = quant16(v[k][0], v[k][NL - 1], f[k]);
                        } else {
                            dequant16(v[k][0], f[k], &lo, &hi);
                        }
                        for (uint32_t c = 0; c < dc; ++c) {
                            if (KVR_DST_DROPPED(rows[ti + c])) continue;
                            unsigned char *to = (unsigned char *)rows[ti + c].y + u * DU;
                            store_stream(to, lo);
                            if (CONV == KVR_CONV_E4M3_TO_BF16) store_stream(to + 16, hi);
                        }
                    }
                }
            }
            __syncthreads();
        }
    } else {
        bool waited = !EARLY;
        for (uint32_t w0 = a.g.div_rc.div(q0); w0 < r_end; w0 += KVR_ROW_WINDOW) {
            const uint32_t w1 = min(w0 + (uint32_t)KVR_ROW_WINDOW, r_end);
            // 1. one thread per row: the row's two addresses (block tables read here).
            // The work list, tables and factors are plan data that no kernel writes,
            // so with EARLY the first window is built before waiting for the
            // previous grid.
            for (uint32_t r = w0 + threadIdx.x; r < w1; r += KVR_THREADS) {
                uint32_t fidx;
                uint64_t sa, da;
                kvr_row<false>(a.g, layer, it, a.sbt, a.dbt, a.src_base, a.dst_base, r, &sa,
                               &da, &fidx);
                KVR_CHECK_ROW(a, sa, da);
                // converting instances ask L2 for the row here (see prefetch_l2_lines)
                if (PF && CONV != KVR_CONV_NONE && !waited &&
                    !KVR_SRC_DROPPED(make_ulonglong2(sa, da)))
                    prefetch_l2_lines<CONV == KVR_CONV_BF16_TO_E4M3>(
                        sa, (uint32_t)a.g.src_row_bytes);
                rows[r - w0] = make_ulonglong2(sa, da);
                if (CONV != KVR_CONV_NONE) row_factor[r - w0] = a.factors[fidx];
            }
            if (PF && CONV == KVR_CONV_NONE && !waited && blockIdx.x < a.prefetch_ctas) {
                // Before the grid-dependency wait, pull the prefill rows this
                // thread just entered into L2, so the loads after the wait hit
                // L2 instead of starting cold: the wait drains the previous
                // grid, and its tail no longer leaves HBM idle. Correct for any
                // previous grid: L2 is where writes from every SM meet, so rows
                // a producer writes after this prefetch replace the prefetched
                // lines there, and the loads after the wait see its writes.
                // A single-layer launch on the whole device leaves it to its
                // first CTAs (prefetch_ctas, kvr_prefetch_ctas): the later ones
                // become resident only as the previous launch's CTAs exit,
                // when issuing 256 bulk requests (~1 us) delays their copy more
                // than the prefetch saves.
                for (uint32_t r = w0 + threadIdx.x; r < w1; r += KVR_THREADS)
                    if (!KVR_SRC_DROPPED(rows[r - w0]))
                        prefetch_l2(rows[r - w0].x, (uint32_t)a.g.src_row_bytes);
            }
            if (EARLY && !waited) {
                if (!a.no_wait) {
                    asm volatile("griddepcontrol.wait;" ::: "memory");
                    asm volatile("griddepcontrol.launch_dependents;");
                }
                waited = true;
            }
            __syncthreads();
            // 2. the units of those rows: U in flight per thread
            const uint32_t qa = max(q0, w0 * rc), qb = min(q1, w1 * rc);
            if constexpr (W == 2) {
                // pairs (q, q + 1), q even: one row (rows hold an even number of
                // units), 32-byte aligned (the plan checked every row)
                constexpr int UP = U > 1 ? U / 2 : 1;
                const uint32_t pa = qa >> 1, pb = qb >> 1;
                for (uint32_t base = pa + threadIdx.x; base < pb; base += UP * KVR_THREADS) {
                    uint4 v[UP][2 * NL];
                    unsigned char *to[UP];
                    float f[UP];
#pragma unroll
                    for (int k = 0; k < UP; ++k) {
                        const uint32_t pq = base + (uint32_t)k * KVR_THREADS;
                        to[k] = nullptr;
                        f[k] = 0.0f;
                        if (pq < pb) {
                            const uint32_t q = pq * 2u;
                            const uint32_t r = a.g.div_rc.div(q);
                            const uint32_t u = q - r * rc;
                            const ulonglong2 p = rows[r - w0];
                            if (!KVR_SRC_DROPPED(p)) {
#pragma unroll
                                for (int j = 0; j < NL; ++j)
                                    load_stream32((const unsigned char *)p.x + u * SU + 32u * j,
                                                  &v[k][2 * j], &v[k][2 * j + 1]);
                                to[k] = (unsigned char *)p.y + u * DU;
                            }
                            if (CONV != KVR_CONV_NONE) f[k] = row_factor[r - w0];
                        }
                    }
#pragma unroll
                    for (int k = 0; k < UP; ++k) {
                        if (to[k] == nullptr) continue;
                        if (CONV == KVR_CONV_NONE) {
                            store_stream32(to[k], v[k][0], v[k][1]);
                        } else if (CONV == KVR_CONV_BF16_TO_E4M3) {
                            store_stream32(to[k], quant16(v[k][0], v[k][1], f[k]),
                                           quant16(v[k][2], v[k][3], f[k]));
                        } else {
                            uint4 lo, hi;
                            dequant16(v[k][0], f[k], &lo, &hi);
                            store_stream32(to[k], lo, hi);
                            dequant16(v[k][1], f[k], &lo, &hi);
                            store_stream32(to[k] + 32, lo, hi);
                        }
                    }
                }
            } else {
                for (uint32_t base = qa + threadIdx.x; base < qb; base += U * KVR_THREADS) {
                    uint4 v[U][NL];
                    unsigned char *to[U];
                    float f[U];
#pragma unroll
                    for (int k = 0; k < U; ++k) {
                        const uint32_t q = base + (uint32_t)k * KVR_THREADS;
                        to[k] = nullptr;
                        f[k] = 0.0f;
                        if (q < qb) {
                            const uint32_t r = a.g.div_rc.div(q);
                            const uint32_t u = q - r * rc;
                            const ulonglong2 p = rows[r - w0];
                            if (!KVR_SRC_DROPPED(p)) {
#pragma unroll
                                for (int j = 0; j < NL; ++j)
                                    v[k][j] =
                                        load_stream((const unsigned char *)p.x + u * SU + 16u * j);
                                to[k] = (unsigned char *)p.y + u * DU;
                            }
                            if (CONV != KVR_CONV_NONE) f[k] = row_factor[r - w0];
                        }
                    }
#pragma unroll
                    for (int k = 0; k < U; ++k) {
                        if (to[k] == nullptr) continue;
                        if (CONV == KVR_CONV_NONE) {
                            store_stream(to[k], v[k][0]);
                        } else if (CONV == KVR_CONV_BF16_TO_E4M3) {
                            store_stream(to[k], quant16(v[k][0], v[k][NL - 1], f[k]));
                        } else {
                            uint4 lo, hi;
                            dequant16(v[k][0], f[k], &lo, &hi);
                            store_stream(to[k], lo);
                            store_stream(to[k] + 16, hi);
                        }
                    }
                }
            }
            __syncthreads();
        }
    }
    // A launch that skipped the wait before its copies still finishes only after
    // the previous grid, so work queued after it on the stream sees both.
    if (a.no_wait) asm volatile("griddepcontrol.wait;" ::: "memory");
}

using KvrKernel = void (*)(KvrArgs);

// Kernel instance for a conversion, launch mode, head replication and access
// width (units in flight per thread: kvr_units).
template <int MODE, bool REP, int W>
KvrKernel pick_instance(int32_t conv) {
    switch (conv) {
        case KVR_CONV_BF16_TO_E4M3:
            return kvr_relayout_kernel<kvr_units(KVR_CONV_BF16_TO_E4M3, MODE, W == 2),
                                       KVR_CONV_BF16_TO_E4M3, MODE, REP, W>;
        case KVR_CONV_E4M3_TO_BF16:
            return kvr_relayout_kernel<kvr_units(KVR_CONV_E4M3_TO_BF16, MODE, W == 2),
                                       KVR_CONV_E4M3_TO_BF16, MODE, REP, W>;
        default:
            return kvr_relayout_kernel<kvr_units(KVR_CONV_NONE, MODE, W == 2), KVR_CONV_NONE,
                                       MODE, REP, W>;
    }
}

template <int MODE>
KvrKernel pick_mode(int32_t conv, bool rep, bool pairs) {
    if (rep) return pairs ? pick_instance<MODE, true, 2>(conv) : pick_instance<MODE, true, 1>(conv);
    return pairs ? pick_instance<MODE, false, 2>(conv) : pick_instance<MODE, false, 1>(conv);
}

// `pairs`: the plan's rows allow pairs of units (KvrHostPlan::pairs);
// kvr_launch_pairs decides per instance and range length (`layers`).
KvrKernel pick_kernel(int32_t conv, int mode, bool rep, bool pairs, int32_t layers) {
    pairs = kvr_launch_pairs(pairs, conv, mode, layers);
    switch (mode) {
        case KVR_MODE_LAYER:
            return pick_mode<KVR_MODE_LAYER>(conv, rep, pairs);
        case KVR_MODE_LAYER_PREFETCH:
            return pick_mode<KVR_MODE_LAYER_PREFETCH>(conv, rep, pairs);
        default:
            return pick_mode<KVR_MODE_WHOLE>(conv, rep, pairs);
    }
}

// prefetch_ctas: KvrArgs::prefetch_ctas (kvr_prefetch_ctas).
kvr_status launch(const kvr_plan *p, int32_t layer0, int32_t layers, int32_t slices,
                  int32_t mode, void *stream, bool no_wait = false,
                  uint32_t prefetch_ctas = 0xFFFFFFFFu) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVR_ERR_CUDA;
    if (dev != p->device) return KVR_ERR_INVALID_ARG;
    KvrArgs a = kvr_launch_args(p->host, p->dev_items, p->dev_sbt, p->dev_dbt, p->dev_factors,
                                p->dev_src_base, p->dev_dst_base, layer0, slices);
    a.no_wait = no_wait ? 1 : 0;
    a.prefetch_ctas = prefetch_ctas;
    const uint64_t grid = (uint64_t)layers * a.tasks_per_layer;
#ifdef KVR_DEVICE_CHECKS
    a.check_regions = p->dev_regions;
    a.n_src_regions = (int32_t)(p->host.src_regions.size() / 2);
    a.n_dst_regions = (int32_t)(p->host.dst_regions.size() / 2);
    a.check_error = p->dev_check_error;
#endif
    if (grid == 0) return KVR_OK;
    // KVR_MODE_LAYER_PREFETCH (kvr_range_launch picks it): ordered per-layer
    // launches of one wave prefetch their first window's prefill rows into L2
    // before the grid-dependency wait; all their CTAs can be resident while the
    // previous grid drains, so the rows arrive during its tail. Measured: 70B
    // layers (512 CTAs, one wave) 5292 -> 6205 GB/s; launches of several waves
    // lost 1.5-3.7 % with the prefetch in their first wave and up to 0.5 % with
    // it in every CTA, so they go without. A launch that does not wait first
    // has nothing to overlap.

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(KVR_THREADS, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = (cudaStream_t)stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg,
                              pick_kernel(p->host.g.conv, mode, kvr_replicated(p->host.g),
                                          p->host.pairs, layers),
                              a) == cudaSuccess
               ? KVR_OK
               : KVR_ERR_CUDA;
}

// The first and last byte of a pool must be memory device `dev` can access:
// its own HBM, managed memory, or pinned host memory mapped at the same
// address (so a pageable host pointer, a freed or foreign pointer, or another
// GPU's memory is refused instead of faulting inside the kernel).
kvr_status check_pool(const void *pool, int64_t bytes, int dev) {
    const unsigned char *ends[2] = {(const unsigned char *)pool,
                                    (const unsigned char *)pool + (bytes > 0 ? bytes - 1 : 0)};
    for (const unsigned char *q : ends) {
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, q) != cudaSuccess) {
            cudaGetLastError();
            return KVR_ERR_POOL_ADDRESS;
        }
        switch (at.type) {
            case cudaMemoryTypeDevice:
                if (at.device != dev) return KVR_ERR_POOL_ADDRESS;
                break;
            case cudaMemoryTypeManaged:
                break;
            case cudaMemoryTypeHost:
                if (at.devicePointer != (const void *)q) return KVR_ERR_POOL_ADDRESS;
                break;
            default:
                return KVR_ERR_POOL_ADDRESS;
        }
    }
    return KVR_OK;
}

kvr_status check_pools(const KvrHostPlan &hp, int dev) {
    for (const std::vector<uint64_t> *regs : {&hp.src_regions, &hp.dst_regions}) {
        for (size_t k = 0; k + 1 < regs->size(); k += 2) {
            const kvr_status st = check_pool((const void *)(uintptr_t)(*regs)[k],
                                             (int64_t)((*regs)[k + 1] - (*regs)[k]), dev);
            if (st != KVR_OK) return st;
        }
    }
    return KVR_OK;
}

// Where a host plan's tables go in one device buffer: items (16-byte aligned
// start), view bases, block ids, factors, back to back.
struct DevTables {
    const KvrItem *items;
    const uint64_t *src_base, *dst_base;
    const int32_t *sbt, *dbt;
    const float *factors;
};

struct Piece {
    const void *host;
    size_t bytes;
};

size_t tables_bytes(const KvrHostPlan &hp) {
    return hp.items.size() * sizeof(KvrItem) +
           (hp.src_base.size() + hp.dst_base.size()) * sizeof(uint64_t) +
           (hp.sbt.size() + hp.dbt.size()) * sizeof(int32_t) + hp.factors.size() * sizeof(float);
}

DevTables place_tables(const KvrHostPlan &hp, unsigned char *base, Piece pieces[6]) {
    size_t off = 0;
    auto put = [&](int k, const void *h, size_t bytes) {
        pieces[k] = {h, bytes};
        unsigned char *p = base + off;
        off += bytes;
        return p;
    };
    DevTables t;
    t.items = (const KvrItem *)put(0, hp.items.data(), hp.items.size() * sizeof(KvrItem));
    t.src_base = (const uint64_t *)put(1, hp.src_base.data(), hp.src_base.size() * 8);
    t.dst_base = (const uint64_t *)put(2, hp.dst_base.data(), hp.dst_base.size() * 8);
    t.sbt = (const int32_t *)put(3, hp.sbt.data(), hp.sbt.size() * 4);
    t.dbt = (const int32_t *)put(4, hp.dbt.data(), hp.dbt.size() * 4);
    const float *f = (const float *)put(5, hp.factors.data(), hp.factors.size() * 4);
    t.factors = hp.factors.empty() ? nullptr : f;
    return t;
}

#ifdef KVR_DEVICE_CHECKS
// Checked builds: copy the plan's merged pool regions (prefill, then decode) to
// the device, followed by a zeroed error word (allocated on the first call).
kvr_status upload_regions(kvr_plan *p) {
    const std::vector<uint64_t> &sr = p->host.src_regions, &dr = p->host.dst_regions;
    const size_t n = sr.size() + dr.size();
    if (p->dev_regions == nullptr) {
        if (cudaMalloc(&p->dev_regions, (n + 2) * sizeof(uint64_t)) != cudaSuccess) {
            cudaGetLastError();
            return KVR_ERR_CUDA;
        }
        p->dev_check_error = (unsigned int *)(p->dev_regions + n);
    }
    std::vector<uint64_t> all(sr);
    all.insert(all.end(), dr.begin(), dr.end());
    if ((n > 0 && cudaMemcpy(p->dev_regions, all.data(), n * sizeof(uint64_t),
                             cudaMemcpyHostToDevice) != cudaSuccess) ||
        cudaMemset(p->dev_check_error, 0, sizeof(unsigned int)) != cudaSuccess)
        return KVR_ERR_CUDA;
    return KVR_OK;
}
#endif

}  // namespace

static kvr_status make_plan(const kvr_desc *desc, const kvr_layout *src_layout,
                            const kvr_layout *dst_layout, const kvr_convert *cv,
                            kvr_plan **out) {
    if (out == nullptr) return KVR_ERR_INVALID_ARG;
    *out = nullptr;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVR_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return KVR_ERR_CUDA;

    kvr_plan *p = new (std::nothrow) kvr_plan();
    if (p == nullptr) return KVR_ERR_NOMEM;
    kvr_status st;
    try {
        const int32_t conv = cv == nullptr ? KVR_CONV_NONE
                             : cv->src_dtype == KVR_DTYPE_BF16 ? KVR_CONV_BF16_TO_E4M3
                                                                : KVR_CONV_E4M3_TO_BF16;
        // the per-layer instance this plan will launch (desc is validated below)
        const bool rep = desc != nullptr && desc->kv_heads > 0 &&
                         (desc->src_tp > desc->kv_heads || desc->dst_tp > desc->kv_heads);
        // CTAs per SM of both per-layer instances (each shapes its own grids)
        auto occupancy = [&](bool pairs, int *resident, int *resident_pf) {
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                    resident, pick_kernel(conv, KVR_MODE_LAYER, rep, pairs, 1), KVR_THREADS,
                    0) != cudaSuccess ||
                cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                    resident_pf, pick_kernel(conv, KVR_MODE_LAYER_PREFETCH, rep, pairs, 1),
                    KVR_THREADS, 0) != cudaSuccess) {
                cudaGetLastError();
                *resident = *resident_pf = 0;
            }
        };
        int resident = 0, resident_pf = 0;
        occupancy(false, &resident, &resident_pf);
        st = kvr_build_host_plan(desc, src_layout, dst_layout, cv, sms, resident, resident_pf,
                                 &p->host, nullptr, nullptr);
        // the plan runs the pair instances: shape its grids for their occupancy
        if (st == KVR_OK && p->host.pairs) {
            occupancy(true, &resident, &resident_pf);
            kvr_shape_launches(p->host, resident, resident_pf);
        }
    } catch (...) {
        st = KVR_ERR_NOMEM;
    }
    if (st == KVR_OK) st = check_pools(p->host, dev);
    if (st != KVR_OK) {
        delete p;
        return st;
    }
    p->device = dev;
    if (!p->host.items.empty()) {
        if (cudaMalloc(&p->dev_meta, tables_bytes(p->host)) != cudaSuccess) {
            cudaGetLastError();
            delete p;
            return KVR_ERR_NOMEM;
        }
        Piece pieces[6];
        const DevTables t = place_tables(p->host, (unsigned char *)p->dev_meta, pieces);
        unsigned char *to = (unsigned char *)p->dev_meta;
        for (const Piece &pc : pieces) {
            if (pc.bytes > 0 &&
                cudaMemcpy(to, pc.host, pc.bytes, cudaMemcpyHostToDevice) != cudaSuccess) {
                cudaFree(p->dev_meta);
                delete p;
                return KVR_ERR_CUDA;
            }
            to += pc.bytes;
        }
        p->dev_items = t.items;
        p->dev_src_base = t.src_base;
        p->dev_dst_base = t.dst_base;
        p->dev_sbt = t.sbt;
        p->dev_dbt = t.dbt;
        p->dev_factors = t.factors;
    }
#ifdef KVR_DEVICE_CHECKS
    if (upload_regions(p) != KVR_OK) {
        kv_relayout_plan_destroy(p);
        return KVR_ERR_CUDA;
    }
#endif
    *out = p;
    return KVR_OK;
}

extern "C" kvr_status kv_relayout_plan(const kvr_desc *desc, kvr_plan **out) {
    return make_plan(desc, nullptr, nullptr, nullptr, out);
}

extern "C" kvr_status kv_relayout_plan_ex(const kvr_desc *desc, const kvr_layout *src_layout,
                                          const kvr_layout *dst_layout, const kvr_convert *cv,
                                          kvr_plan **out) {
    return make_plan(desc, src_layout, dst_layout, cv, out);
}

extern "C" kvr_status kv_relayout_plan_convert(const kvr_desc *desc, const kvr_convert *cv,
                                               kvr_plan **out) {
    if (cv == nullptr) {
        if (out != nullptr) *out = nullptr;
        return KVR_ERR_INVALID_ARG;
    }
    return make_plan(desc, nullptr, nullptr, cv, out);
}

// -- pack / unpack: one side is a contiguous staging buffer ---------------------

static kvr_status make_staging_plan(const kvr_desc *desc, const void *staging,
                                    const kvr_convert *cv, bool pack, kvr_plan **out) {
    if (out == nullptr) return KVR_ERR_INVALID_ARG;
    *out = nullptr;
    KvrStaging sd;
    kvr_desc d;
    kvr_status st;
    try {
        st = kvr_staging_desc(desc, staging, cv, pack, &sd, &d);
    } catch (...) {
        return KVR_ERR_NOMEM;
    }
    if (st != KVR_OK) return st;
    return make_plan(&d, pack ? nullptr : &sd.layout, pack ? &sd.layout : nullptr, cv, out);
}

extern "C" kvr_status kv_relayout_plan_pack(const kvr_desc *desc, void *staging,
                                            const kvr_convert *cv, kvr_plan **out) {
    return make_staging_plan(desc, staging, cv, true, out);
}

extern "C" kvr_status kv_relayout_plan_unpack(const kvr_desc *desc, const void *staging,
                                              const kvr_convert *cv, kvr_plan **out) {
    return make_staging_plan(desc, staging, cv, false, out);
}

extern "C" kvr_status kv_relayout_layer(const kvr_plan *plan, int32_t layer, void *stream) {
    if (plan == nullptr) return KVR_ERR_INVALID_ARG;
    if (layer < 0 || layer >= plan->host.num_layers) return KVR_ERR_LAYER_RANGE;
    return kv_relayout_layers_ex(plan, layer, 1, 0u, stream);
}

extern "C" kvr_status kv_relayout_all(const kvr_plan *plan, void *stream) {
    if (plan == nullptr) return KVR_ERR_INVALID_ARG;
    // a stream on a green context with fewer SMs gets a grid shaped for them
    const int32_t green = kvr_stream_green_sms(stream);
    const int32_t slices = green > 0 && green < plan->host.sm_count
                               ? kvr_range_slices(plan->host, plan->host.num_layers, green)
                               : plan->host.slices_all;
    return launch(plan, 0, plan->host.num_layers, slices, KVR_MODE_WHOLE, stream);
}

extern "C" kvr_status kv_relayout_layers_ex(const kvr_plan *plan, int32_t first, int32_t count,
                                            uint32_t flags, void *stream) {
    if (plan == nullptr || (flags & ~KVR_LAUNCH_NO_WAIT) != 0) return KVR_ERR_INVALID_ARG;
    const int32_t L = plan->host.num_layers;
    if (first < 0 || count < 1 || first >= L || count > L - first) return KVR_ERR_LAYER_RANGE;
    const bool no_wait = (flags & KVR_LAUNCH_NO_WAIT) != 0;
    int32_t slices = 1, mode = KVR_MODE_LAYER;
    // the stream's green context, if any, shapes the grid (a driver query that
    // measured no cost on back-to-back 70B layer launches)
    const int32_t green = kvr_stream_green_sms(stream);
    kvr_range_launch(plan->host, count, green, no_wait, &slices, &mode);
    return launch(plan, first, count, slices, mode, stream, no_wait,
                  kvr_prefetch_ctas(plan->host, count, green, mode, slices));
}

extern "C" kvr_status kv_relayout_layers(const kvr_plan *plan, int32_t first, int32_t count,
                                         void *stream) {
    return kv_relayout_layers_ex(plan, first, count, 0u, stream);
}

extern "C" kvr_status kv_relayout_plan_bytes(const kvr_plan *plan, int64_t *bytes_read,
                                             int64_t *bytes_written) {
    if (plan == nullptr) return KVR_ERR_INVALID_ARG;
    if (bytes_read) *bytes_read = plan->host.bytes_read;
    if (bytes_written) *bytes_written = plan->host.bytes_written;
    return KVR_OK;
}

extern "C" kvr_status kv_relayout_plan_launch_shape(const kvr_plan *plan, int64_t *grid_all,
                                                    int64_t *grid_layer, int32_t *tile_tokens) {
    if (plan == nullptr) return KVR_ERR_INVALID_ARG;
    const int64_t n = (int64_t)plan->host.items.size();
    if (grid_all) *grid_all = n * plan->host.num_layers * plan->host.slices_all;
    // an ordered kv_relayout_layer() launch (the prefetching shape when it has one)
    if (grid_layer)
        *grid_layer = n * (plan->host.slices_layer_pf > 0 ? plan->host.slices_layer_pf
                                                          : plan->host.slices_layer);
    if (tile_tokens) *tile_tokens = plan->host.tile;
    return KVR_OK;
}

extern "C" void kv_relayout_plan_destroy(kvr_plan *plan) {
    if (plan == nullptr) return;
    if (plan->dev_meta != nullptr) cudaFree(plan->dev_meta);
#ifdef KVR_DEVICE_CHECKS
    if (plan->dev_regions != nullptr) cudaFree(plan->dev_regions);
#endif
    delete plan;
}

extern "C" kvr_status kv_relayout_debug_status(const kvr_plan *plan, uint32_t *flags) {
    if (flags != nullptr) *flags = 0;
#ifdef KVR_DEVICE_CHECKS
    if (plan == nullptr) return KVR_ERR_INVALID_ARG;
    unsigned int word = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(&word, plan->dev_check_error, sizeof(word), cudaMemcpyDeviceToHost) !=
            cudaSuccess ||
        cudaMemset(plan->dev_check_error, 0, sizeof(word)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
        return KVR_ERR_CUDA;
    if (flags != nullptr) *flags = word;
    return word != 0 ? KVR_ERR_DEVICE_BOUNDS : KVR_OK;
#else
    (void)plan;
    return KVR_ERR_UNSUPPORTED;
#endif
}

extern "C" kvr_status kv_relayout_debug_narrow(kvr_plan *plan, int64_t bytes) {
#ifdef KVR_DEVICE_CHECKS
    if (plan == nullptr || bytes < 0) return KVR_ERR_INVALID_ARG;
    for (std::vector<uint64_t> *regs : {&plan->host.src_regions, &plan->host.dst_regions})
        for (size_t k = 0; k + 1 < regs->size(); k += 2)
            (*regs)[k + 1] = (*regs)[k + 1] - (*regs)[k] > (uint64_t)bytes
                                 ? (*regs)[k + 1] - (uint64_t)bytes
                                 : (*regs)[k];
    return upload_regions(plan);
#else
    (void)plan;
    (void)bytes;
    return KVR_ERR_UNSUPPORTED;
#endif
}

// ---------------------------------------------------------------------------
// kv_relayout_all_prealloc: the whole-prompt relayout without any device
// allocation. The kernel's scratch (the work list, the view bases and the used
// block ids, normally in the plan's cudaMalloc'd buffer) lives in the
// file-scope array below instead. Every GPU that loads this library holds the
// array until the process exits.
// ---------------------------------------------------------------------------
#include <mutex>

#define KVR_PREALLOC_MAX_DEVICES 64

static __device__ __align__(256) unsigned char g_kvr_prealloc_scratch[KVR_PREALLOC_SCRATCH_BYTES];

namespace {

struct PreallocScratch {
    bool ready = false;
    unsigned char *addr = nullptr;   // device address of g_kvr_prealloc_scratch
    int sms = 0;
    std::mutex use;                  // held from a call's copy to its launch
};

PreallocScratch g_prealloc[KVR_PREALLOC_MAX_DEVICES];
std::mutex g_prealloc_setup_mu;

// Once per device, with that device current: the array's device address. In
// host code the array's name is only a host-side stand-in, so the kernel must
// be given this address, never the name.
kvr_status prealloc_setup(int dev, PreallocScratch **out) {
    std::lock_guard<std::mutex> lock(g_prealloc_setup_mu);
    PreallocScratch &s = g_prealloc[dev];
    if (!s.ready) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_kvr_prealloc_scratch) != cudaSuccess) {
            cudaGetLastError();
            return KVR_ERR_CUDA;
        }
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return KVR_ERR_CUDA;
        s.addr = (unsigned char *)p;
        s.sms = sms;
        s.ready = true;
    }
    *out = &s;
    return KVR_OK;
}

}  // namespace

extern "C" kvr_status kv_relayout_all_prealloc(const kvr_desc *desc, void *stream) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVR_ERR_CUDA;
    if (dev < 0 || dev >= KVR_PREALLOC_MAX_DEVICES) return KVR_ERR_UNSUPPORTED;
    cudaStream_t s = (cudaStream_t)stream;
    // The tables are copied from host memory that is gone when this call
    // returns, so the call enqueues nothing on a stream that is being captured.
    cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &capturing) != cudaSuccess) {
        cudaGetLastError();
        return KVR_ERR_UNSUPPORTED;
    }
    if (capturing != cudaStreamCaptureStatusNone) return KVR_ERR_UNSUPPORTED;
    PreallocScratch *sc = nullptr;
    kvr_status st = prealloc_setup(dev, &sc);
    if (st != KVR_OK) return st;

    KvrHostPlan hp;
    std::vector<unsigned char> staged;
    Piece pieces[6];
    DevTables t = {};
    try {
        st = kvr_build_host_plan(desc, nullptr, nullptr, nullptr, sc->sms, 0, 0, &hp, nullptr,
                                 nullptr);
        if (st == KVR_OK) st = check_pools(hp, dev);
        if (st == KVR_OK && tables_bytes(hp) > KVR_PREALLOC_SCRATCH_BYTES)
            st = KVR_ERR_SCRATCH_LIMIT;
        if (st == KVR_OK && !hp.items.empty()) {
            // every table in one host buffer laid out like the scratch: one copy
            t = place_tables(hp, sc->addr, pieces);
            staged.resize(tables_bytes(hp));
            size_t off = 0;
            for (const Piece &pc : pieces) {
                if (pc.bytes > 0) memcpy(staged.data() + off, pc.host, pc.bytes);
                off += pc.bytes;
            }
        }
    } catch (...) {
        st = KVR_ERR_NOMEM;
    }
    if (st != KVR_OK) return st;
    if (hp.items.empty()) return KVR_OK;

    // a stream on a green context with fewer SMs gets a grid shaped for them
    const int32_t green = kvr_stream_green_sms(stream);
    const int32_t slices = green > 0 && green < hp.sm_count
                               ? kvr_range_slices(hp, hp.num_layers, green)
                               : hp.slices_all;
    const KvrArgs a = kvr_launch_args(hp, t.items, t.sbt, t.dbt, nullptr, t.src_base,
                                      t.dst_base, 0, slices);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((uint64_t)hp.num_layers * a.tasks_per_layer), 1, 1);
    cfg.blockDim = dim3(KVR_THREADS, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    // No programmatic dependent launch: the kernel follows this call's copy of
    // its tables on `stream` and must start only after it.
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    // The copy and the launch go onto the stream back to back under the
    // device's lock, so calls from several host threads on one stream cannot
    // interleave one call's copy with another call's kernel. The array is
    // overwritten up to what this call reads, so nothing needs clearing.
    std::lock_guard<std::mutex> lock(sc->use);
    if (cudaMemcpyAsync(sc->addr, staged.data(), staged.size(), cudaMemcpyHostToDevice, s) !=
        cudaSuccess)
        return KVR_ERR_CUDA;
    return cudaLaunchKernelEx(&cfg,
                              pick_kernel(KVR_CONV_NONE, KVR_MODE_WHOLE, kvr_replicated(hp.g),
                                          hp.pairs, hp.num_layers),
                              a) == cudaSuccess
               ? KVR_OK
               : KVR_ERR_CUDA;
}
