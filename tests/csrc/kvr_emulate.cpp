// kvr_emulate.cpp -- test harness: runs the relayout kernel's work decomposition on the CPU.
//
// Links the library's own plan code (plan.cpp) and includes the kernel's index
// header (kvr_index.h), then walks every CTA and thread of a launch exactly as
// the kernel's loop does, on HOST buffers. Every computed address is checked
// against its pool before it is used. This is how the kernel's grid and index
// arithmetic are checked on the CPU; it is not part of the library.
#include <stdint.h>
#include <string.h>

#include <vector>

#include "kv_relayout.h"
#include "kvr_index.h"
#include "plan.h"

namespace {

// [start, end) byte ranges of the buffers one side may touch.
struct Ranges {
    std::vector<uint64_t> lo, hi;
    bool holds(uint64_t a, uint64_t n) const {
        for (size_t k = 0; k < lo.size(); ++k)
            if (a >= lo[k] && a + n <= hi[k]) return true;
        return false;
    }
};

// The standard layout: one pool per shard, [L][C][N][B][H_local][D].
Ranges pool_ranges(const void *const *pools, int32_t T, const kvr_desc *d, int64_t N, int32_t B,
                   int64_t es) {
    Ranges r;
    // heads per shard: H / T, or 1 when T > H (each head on T / H shards)
    const int64_t hl = T <= d->kv_heads ? d->kv_heads / T : 1;
    const int64_t bytes = (int64_t)d->num_layers * d->num_components * N * B * hl *
                          d->head_dim * es;
    for (int32_t s = 0; s < T; ++s) {
        r.lo.push_back((uint64_t)(uintptr_t)pools[s]);
        r.hi.push_back((uint64_t)(uintptr_t)pools[s] + (uint64_t)bytes);
    }
    return r;
}

Ranges given_ranges(const uint64_t *pairs, int64_t n) {
    Ranges r;
    for (int64_t k = 0; k < n; ++k) {
        r.lo.push_back(pairs[2 * k]);
        r.hi.push_back(pairs[2 * k + 1]);
    }
    return r;
}

// Walk one launch exactly as the kernel's loops do (CTA by CTA, row window by
// row window, thread by thread): count < 0 is kv_relayout_all(), otherwise
// kv_relayout_layers(first, count) (count == 1: kv_relayout_layer(first)).
// Every row must lie inside one of its side's ranges and every unit address
// be 16-byte aligned. copy != 0 (bit copies only): move the bytes. Returns the
// number of bad rows or units (all skipped), or a negative kvr_status;
// *chunks receives the units visited.
int64_t walk(const kvr_desc *d, const kvr_layout *sl, const kvr_layout *dl, const kvr_convert *cv,
             const Ranges &sr, const Ranges &dr, int sm_count, int first, int count, int copy,
             int64_t *chunks) {
    KvrHostPlan hp;
    kvr_status st = kvr_build_host_plan(d, sl, dl, cv, sm_count, 4, 4, &hp, nullptr, nullptr);
    if (st != KVR_OK) return st;
    if (hp.g.conv != KVR_CONV_NONE) copy = 0;   // converted values are checked on the GPU
    const int all = count < 0;
    if (!all && (first < 0 || count < 1 || first + count > hp.num_layers))
        return KVR_ERR_LAYER_RANGE;
    int32_t slices = hp.slices_all;
    int32_t mode = KVR_MODE_WHOLE;               // the kernel instance (an ordered launch)
    if (!all) kvr_range_launch(hp, count, 0, false, &slices, &mode);
    const int32_t layer0 = all ? 0 : first, layers = all ? hp.num_layers : count;
    const KvrArgs a = kvr_launch_args(hp, hp.items.data(), hp.sbt.data(), hp.dbt.data(),
                                      hp.factors.data(), hp.src_base.data(), hp.dst_base.data(),
                                      layer0, slices);
    const uint64_t grid = (uint64_t)layers * a.tasks_per_layer;
    const uint32_t rc = (uint32_t)a.g.row_chunks;
    // units in flight per thread, as the kernel instance the launch picks
    const bool pairs = kvr_launch_pairs(hp.pairs, hp.g.conv, mode, layers);
    const uint32_t U = (uint32_t)kvr_units(hp.g.conv, mode, pairs);
    const uint32_t su = (uint32_t)a.g.src_unit_bytes, du = (uint32_t)a.g.dst_unit_bytes;
    const int64_t n_factors = (int64_t)hp.factors.size();
    static uint64_t rows_src[KVR_ROW_WINDOW], rows_dst[KVR_ROW_WINDOW];
    // replicated heads (kvr_replicated): a window of win_rows prefill rows, a
    // table row per (prefill row, decode copy), one load and dc stores per
    // unit; otherwise dc = 1 and the table rows are the prefill rows
    const bool rep = kvr_replicated(a.g);
    const uint32_t dc = rep ? (uint32_t)a.g.dcopies : 1u;
    const uint32_t wn = rep ? (uint32_t)a.g.win_rows : (uint32_t)KVR_ROW_WINDOW;
    if (wn * dc > KVR_ROW_WINDOW || wn == 0) return KVR_ERR_UNSUPPORTED;
    int64_t bad = 0, visited = 0;
    for (uint64_t task = 0; task < grid; ++task) {
        int32_t l;
        KvrItem it;
        uint32_t q0, q1;
        if (pairs)
            kvr_task<2>(a, (uint32_t)task, a.items, &l, &it, &q0, &q1);
        else
            kvr_task<1>(a, (uint32_t)task, a.items, &l, &it, &q0, &q1);
        if (q0 > q1 || l < layer0 || l >= layer0 + layers || (pairs && (q0 | q1) % 2 != 0)) {
            ++bad;
            continue;
        }
        if (q0 == q1) continue;
        const uint32_t r_end = a.g.div_rc.div(q1 - 1) + 1;
        for (uint32_t w0 = a.g.div_rc.div(q0); w0 < r_end; w0 += wn) {
            const uint32_t w1 = w0 + wn < r_end ? w0 + wn : r_end;
            const uint32_t t_end = (w1 - w0) * dc;
            for (uint32_t tid = 0; tid < KVR_THREADS; ++tid)
                for (uint32_t t = tid; t < t_end; t += KVR_THREADS) {
                    uint32_t fidx;
                    uint64_t sa, da;
                    (rep ? kvr_row<true> : kvr_row<false>)(a.g, l, it, a.sbt, a.dbt, a.src_base,
                                                           a.dst_base, w0 * dc + t, &sa, &da,
                                                           &fidx);
                    if (!sr.holds(sa, (uint64_t)a.g.src_row_bytes) ||
                        !dr.holds(da, (uint64_t)a.g.dst_row_bytes) ||
                        (a.g.conv != KVR_CONV_NONE && (int64_t)fidx >= n_factors)) {
                        ++bad;
                        rows_src[t] = rows_dst[t] = UINT64_MAX;
                        continue;
                    }
                    rows_src[t] = sa;
                    rows_dst[t] = da;
                }
            const uint32_t qa = q0 > w0 * rc ? q0 : w0 * rc;
            const uint32_t qb = q1 < w1 * rc ? q1 : w1 * rc;
            if (pairs) {
                // pairs of adjacent units (q, q + 1), U / 2 in flight, one 32-byte
                // access each: both units in one row, both addresses 32-byte aligned,
                // loaded once and stored to each of the dc decode copies
                const uint32_t up = U > 1 ? U / 2 : 1, pa = qa / 2, pb = qb / 2;
                if (qa % 2 != 0 || qb % 2 != 0) ++bad;
                for (uint32_t tid = 0; tid < KVR_THREADS; ++tid)
                    for (uint32_t base = pa + tid; base < pb; base += up * KVR_THREADS)
                        for (uint32_t k = 0; k < up; ++k) {
                            const uint32_t pq = base + k * KVR_THREADS;
                            if (pq >= pb) continue;
                            const uint32_t q = 2 * pq;
                            const uint32_t r = a.g.div_rc.div(q);
                            const uint32_t u = q - r * rc;
                            if (r < w0 || r >= w1 || a.g.div_rc.div(q + 1) != r) {
                                ++bad;
                                continue;
                            }
                            const uint32_t ti = (r - w0) * dc;
                            for (uint32_t c = 0; c < dc; ++c) {
                                visited += 2;
                                if (rows_src[ti + c] == UINT64_MAX ||
                                    rows_src[ti + c] != rows_src[ti]) {
                                    ++bad;
                                    continue;
                                }
                                const uint64_t from = rows_src[ti] + (uint64_t)u * su;
                                const uint64_t to = rows_dst[ti + c] + (uint64_t)u * du;
                                if (from % 32 != 0 || to % 32 != 0 ||
                                    (u + 2) * su > (uint32_t)a.g.src_row_bytes ||
                                    (u + 2) * du > (uint32_t)a.g.dst_row_bytes) {
                                    ++bad;
                                    continue;
                                }
                                if (copy)
                                    memcpy((void *)(uintptr_t)to, (const void *)(uintptr_t)from,
                                           32);
                            }
                        }
                continue;
            }
            for (uint32_t tid = 0; tid < KVR_THREADS; ++tid) {
                for (uint32_t base = qa + tid; base < qb; base += U * KVR_THREADS) {
                    for (uint32_t k = 0; k < U; ++k) {
                        const uint32_t q = base + k * KVR_THREADS;
                        if (q >= qb) continue;
                        const uint32_t r = a.g.div_rc.div(q);
                        const uint32_t u = q - r * rc;
                        if (r < w0 || r >= w1) {
                            ++bad;
                            continue;
                        }
                        const uint32_t ti = (r - w0) * dc;
                        for (uint32_t c = 0; c < dc; ++c) {
                            ++visited;
                            // every copy's prefill address is the one the unit is loaded from
                            if (rows_src[ti + c] == UINT64_MAX || rows_src[ti + c] != rows_src[ti]) {
                                ++bad;
                                continue;
                            }
                            const uint64_t from = rows_src[ti] + (uint64_t)u * su;
                            const uint64_t to = rows_dst[ti + c] + (uint64_t)u * du;
                            if (from % 16 != 0 || to % 16 != 0 ||
                                (u + 1) * su > (uint32_t)a.g.src_row_bytes ||
                                (u + 1) * du > (uint32_t)a.g.dst_row_bytes) {
                                ++bad;
                                continue;
                            }
                            if (copy)
                                memcpy((void *)(uintptr_t)to, (const void *)(uintptr_t)from, 16);
                        }
                    }
                }
            }
        }
    }
    if (chunks) *chunks = visited;
    return bad;
}

int64_t dst_es(const kvr_desc *d, const kvr_convert *cv) {
    if (cv == nullptr) return d->elem_bytes;
    return cv->dst_dtype == KVR_DTYPE_BF16 ? 2 : 1;
}

}  // namespace

extern "C" {

// Relayout on host pools through the kernel's decomposition. layer < 0: all layers.
int64_t emu_relayout(const kvr_desc *d, int sm_count, int32_t layer, int64_t *chunks) {
    return walk(d, nullptr, nullptr, nullptr,
                pool_ranges(d->src_pools, d->src_tp, d, d->src_num_blocks, d->src_block_size,
                            d->elem_bytes),
                pool_ranges((const void *const *)d->dst_pools, d->dst_tp, d, d->dst_num_blocks,
                            d->dst_block_size, d->elem_bytes),
                sm_count, layer < 0 ? 0 : layer, layer < 0 ? -1 : 1, 1, chunks);
}

// Bounds/alignment check of every address of a launch (pools are never touched).
int64_t emu_check(const kvr_desc *d, int sm_count, int32_t layer, int64_t *chunks) {
    return walk(d, nullptr, nullptr, nullptr,
                pool_ranges(d->src_pools, d->src_tp, d, d->src_num_blocks, d->src_block_size,
                            d->elem_bytes),
                pool_ranges((const void *const *)d->dst_pools, d->dst_tp, d, d->dst_num_blocks,
                            d->dst_block_size, d->elem_bytes),
                sm_count, layer < 0 ? 0 : layer, layer < 0 ? -1 : 1, 0, chunks);
}

// The same check for a converting relayout (units of 16 elements).
int64_t emu_check_convert(const kvr_desc *d, const kvr_convert *cv, int sm_count, int32_t layer,
                          int64_t *chunks) {
    return walk(d, nullptr, nullptr, cv,
                pool_ranges(d->src_pools, d->src_tp, d, d->src_num_blocks, d->src_block_size,
                            d->elem_bytes),
                pool_ranges((const void *const *)d->dst_pools, d->dst_tp, d, d->dst_num_blocks,
                            d->dst_block_size, dst_es(d, cv)),
                sm_count, layer < 0 ? 0 : layer, layer < 0 ? -1 : 1, 0, chunks);
}

// Any layouts: every row must fall inside the [lo, hi) pairs given per side.
int64_t emu_walk_ex(const kvr_desc *d, const kvr_layout *sl, const kvr_layout *dl,
                    const kvr_convert *cv, const uint64_t *src_ranges, int64_t n_src,
                    const uint64_t *dst_ranges, int64_t n_dst, int sm_count, int32_t layer,
                    int32_t copy, int64_t *chunks) {
    return walk(d, sl, dl, cv, given_ranges(src_ranges, n_src), given_ranges(dst_ranges, n_dst),
                sm_count, layer < 0 ? 0 : layer, layer < 0 ? -1 : 1, copy, chunks);
}

// kv_relayout_plan_pack (pack != 0) / _unpack on host buffers: *d with one side
// replaced by the library's own staging side over `staging`
// (kvr_staging_desc), walked like emu_walk_ex; the other side is d's pools in
// the standard layout. Every row must fall inside the given ranges.
int64_t emu_staging(const kvr_desc *d, void *staging, int32_t pack, const uint64_t *src_ranges,
                    int64_t n_src, const uint64_t *dst_ranges, int64_t n_dst, int sm_count,
                    int32_t layer, int32_t copy, int64_t *chunks) {
    KvrStaging st;
    kvr_desc d2;
    const kvr_status s = kvr_staging_desc(d, staging, nullptr, pack != 0, &st, &d2);
    if (s != KVR_OK) return s;
    return walk(&d2, pack ? nullptr : &st.layout, pack ? &st.layout : nullptr, nullptr,
                given_ranges(src_ranges, n_src), given_ranges(dst_ranges, n_dst), sm_count,
                layer < 0 ? 0 : layer, layer < 0 ? -1 : 1, copy, chunks);
}

// kv_relayout_layers(first, count) on host pools through the kernel's
// decomposition (copy != 0: move the bytes; 0: bounds check only).
int64_t emu_relayout_range(const kvr_desc *d, int sm_count, int32_t first, int32_t count,
                           int32_t copy, int64_t *chunks) {
    return walk(d, nullptr, nullptr, nullptr,
                pool_ranges(d->src_pools, d->src_tp, d, d->src_num_blocks, d->src_block_size,
                            d->elem_bytes),
                pool_ranges((const void *const *)d->dst_pools, d->dst_tp, d, d->dst_num_blocks,
                            d->dst_block_size, d->elem_bytes),
                sm_count, first, count, copy, chunks);
}

// Whether the plan's rows allow pairs of units per access (KvrHostPlan::pairs):
// 1 or 0, or a negative kvr_status.
int32_t emu_plan_pairs(const kvr_desc *d, const kvr_layout *sl, const kvr_layout *dl,
                       const kvr_convert *cv) {
    KvrHostPlan hp;
    kvr_status st = kvr_build_host_plan(d, sl, dl, cv, 152, 4, 4, &hp, nullptr, nullptr);
    if (st != KVR_OK) return st;
    return hp.pairs ? 1 : 0;
}

// Work-list facts of a plan: [n_items, slices_all, slices_layer, grid_all, grid_layer, tile].
int32_t emu_plan_info(const kvr_desc *d, int sm_count, int64_t *out) {
    KvrHostPlan hp;
    kvr_status st = kvr_build_host_plan(d, nullptr, nullptr, nullptr, sm_count, 4, 4, &hp,
                                        nullptr, nullptr);
    if (st != KVR_OK) return st;
    const int64_t n = (int64_t)hp.items.size();
    out[0] = n;
    out[1] = hp.slices_all;
    out[2] = hp.slices_layer;
    out[3] = n * hp.slices_all * hp.num_layers;
    out[4] = n * hp.slices_layer;
    out[5] = hp.tile;
    return 0;
}

// KvrDiv against the hardware divide for one divisor, at the dividends most
// likely to break a multiply-shift division (around multiples of d, the top of
// the 31-bit range) plus a strided sweep. Returns the number of mismatches.
int64_t emu_fastdiv_check_one(uint32_t d, uint32_t stride) {
    int64_t bad = 0;
    const KvrDiv f = kvr_make_div(d);
    auto chk = [&](uint64_t n) {
        if (n >= (1ull << 31)) return;
        if (f.div((uint32_t)n) != (uint32_t)n / d) ++bad;
    };
    for (uint64_t k = 0; k < 64; ++k) {
        chk(k);
        chk(k * d);
        chk(k * d + d - 1);
        chk(k * d + 1);
    }
    const uint64_t top = (1ull << 31) - 1;
    for (uint64_t k = 0; k < 64 && k <= top / d; ++k) {
        const uint64_t m = (top / d - k) * d;
        chk(m);
        chk(m + d - 1);
        if (m) chk(m - 1);
        chk(top - k);
    }
    for (uint64_t n = d; n < (1ull << 31); n += (uint64_t)stride + d) chk(n);
    return bad;
}

// Divisors 1..d_max.
int64_t emu_fastdiv_check(uint32_t d_max, uint32_t stride) {
    int64_t bad = 0;
    for (uint32_t d = 1; d <= d_max; ++d) bad += emu_fastdiv_check_one(d, stride);
    return bad;
}
}

extern "C" {

// kvr_range_launch() for a plan built with the given residencies: out = [slices,
// mode, grid (CTAs), items].
// out: [slices, mode, grid, items per layer, CTAs that prefetch (kvr_prefetch_ctas)]
int32_t emu_range_launch(const kvr_desc *d, int sm_count, int resident, int resident_pf,
                         int32_t count, int32_t stream_sms, int32_t no_wait, int64_t *out) {
    KvrHostPlan hp;
    kvr_status st = kvr_build_host_plan(d, nullptr, nullptr, nullptr, sm_count, resident,
                                        resident_pf, &hp, nullptr, nullptr);
    if (st != KVR_OK) return st;
    int32_t slices = 0, mode = -1;
    kvr_range_launch(hp, count, stream_sms, no_wait != 0, &slices, &mode);
    out[0] = slices;
    out[1] = mode;
    out[2] = (int64_t)count * (int64_t)hp.items.size() * slices;
    out[3] = (int64_t)hp.items.size();
    out[4] = kvr_prefetch_ctas(hp, count, stream_sms, mode, slices);
    return 0;
}

}  // extern "C"
