// plan.cpp -- descriptor validation, byte counts and the work list (host only).
//
// The checks follow what the hand-off on the page "PD 分离与 KV 传输"
// (sections "实现" and "布局转换") needs to be well defined: each prompt
// position has a prefill block and a decode block (tables long enough, ids in
// range), no two positions land on the same decode slot (no decode block used
// twice), and every head has a home on each side: a TP degree T that divides
// H gives each shard H/T heads; a multiple of H gives each head T/H shards
// (read from the first on the prefill side, written to all on the decode side).
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <new>
#include <vector>

#include "plan.h"

namespace {

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// a * b * ... without overflowing int64; false when the product does not fit.
bool mul_fits(std::initializer_list<int64_t> xs, int64_t *out) {
    __int128 p = 1;
    for (int64_t x : xs) {
        p *= x;
        if (p > (__int128)INT64_MAX) return false;
    }
    *out = (int64_t)p;
    return true;
}

kvr_status check_table(int32_t R, const int32_t *lens, const int64_t *off, const int32_t *bt,
                       int32_t block, int64_t num_blocks) {
    if (R > 0 && (off == nullptr || lens == nullptr)) return KVR_ERR_INVALID_ARG;
    if (R > 0 && off[0] < 0) return KVR_ERR_INVALID_ARG;
    for (int32_t r = 0; r < R; ++r) {
        if (lens[r] < 0) return KVR_ERR_INVALID_ARG;
        if (off[r + 1] < off[r]) return KVR_ERR_INVALID_ARG;
    }
    for (int32_t r = 0; r < R; ++r) {
        const int64_t need = ceil_div(lens[r], block);
        if (off[r + 1] - off[r] < need) return KVR_ERR_TABLE_SHORT;
        if (need > 0 && bt == nullptr) return KVR_ERR_INVALID_ARG;
        for (int64_t k = 0; k < need; ++k) {
            const int32_t id = bt[off[r] + k];
            if (id < 0 || (int64_t)id >= num_blocks) return KVR_ERR_BLOCK_RANGE;
        }
    }
    return KVR_OK;
}

int32_t choose_slices(int64_t tasks_unsliced, int64_t avg_chunks, int sm_count,
                      int ctas_per_sm) {
    const int64_t target = (int64_t)std::max(sm_count, 1) * ctas_per_sm;
    if (tasks_unsliced <= 0 || tasks_unsliced >= target) return 1;
    const int64_t want = ceil_div(target, tasks_unsliced);
    const int64_t most = std::max<int64_t>(1, avg_chunks / KVR_MIN_SLICE_CHUNKS);
    return (int32_t)std::min(want, most);
}

// Per-layer launches are short: a partial extra wave costs a large share of
// the launch. With `slots` CTAs resident at once, a layer whose items fit in
// one wave is sliced to fill that wave without spilling over; a layer with
// more items is sliced to about three waves, so the last one is a small part.
int32_t choose_layer_slices(int64_t items, int64_t avg_chunks, int sm_count, int resident) {
    if (items <= 0) return 1;
    const int64_t slots =
        (int64_t)std::max(sm_count, 1) * (resident > 0 ? resident : KVR_LAYER_CTAS_PER_SM);
    const int64_t want = items < slots ? slots / items : ceil_div(3 * slots, items);
    const int64_t most = std::max<int64_t>(1, avg_chunks / KVR_MIN_SLICE_CHUNKS);
    return (int32_t)std::max<int64_t>(1, std::min(want, most));
}

// One side's views: base address per (shard, layer, component), shared
// strides, and the bytes one view spans.
struct Side {
    std::vector<uint64_t> base;
    int64_t bs = 0, ts = 0, hs = 0;
    int64_t span = 0;
    // a view seen as n_outer intervals of inner bytes, outer_stride apart (the
    // outer dimension is the one with the largest stride among those of extent > 1)
    int64_t outer_stride = 0, n_outer = 1, inner = 0;
};

kvr_status make_side(const kvr_layout *lay, const void *const *pools, int32_t T, int32_t L,
                     int32_t C, int64_t N, int32_t B, int32_t Hl, int64_t row, Side *out) {
    const int64_t views = (int64_t)T * L * C;
    if (views > (int64_t)1 << 26) return KVR_ERR_UNSUPPORTED;
    out->base.assign((size_t)views, 0);
    int64_t plane = 0;
    if (lay == nullptr) {
        if (pools == nullptr) return KVR_ERR_INVALID_ARG;
        for (int32_t s = 0; s < T; ++s)
            if (pools[s] == nullptr) return KVR_ERR_INVALID_ARG;
        for (int32_t s = 0; s < T; ++s)
            if ((uintptr_t)pools[s] % 16 != 0) return KVR_ERR_ALIGNMENT;
        int64_t bs = 0, total = 0;
        if (!mul_fits({(int64_t)B, Hl, row}, &bs) || !mul_fits({N, bs}, &plane) ||
            !mul_fits({plane, (int64_t)L, C}, &total))
            return KVR_ERR_UNSUPPORTED;
        out->bs = bs;
        out->ts = (int64_t)Hl * row;
        out->hs = row;
        for (int32_t s = 0; s < T; ++s)
            for (int64_t v = 0; v < (int64_t)L * C; ++v)
                out->base[s * (int64_t)L * C + v] = (uint64_t)(uintptr_t)pools[s] + v * plane;
    } else {
        if (lay->bases == nullptr) return KVR_ERR_INVALID_ARG;
        if (lay->block_stride < 0 || lay->token_stride < 0 || lay->head_stride < 0)
            return KVR_ERR_INVALID_ARG;
        for (int64_t v = 0; v < views; ++v)
            if (lay->bases[v] == nullptr) return KVR_ERR_INVALID_ARG;
        for (int64_t v = 0; v < views; ++v)
            if ((uintptr_t)lay->bases[v] % 16 != 0) return KVR_ERR_ALIGNMENT;
        out->bs = lay->block_stride;
        out->ts = lay->token_stride;
        out->hs = lay->head_stride;
        for (int64_t v = 0; v < views; ++v) out->base[v] = (uint64_t)(uintptr_t)lay->bases[v];
    }
    // a stride counts only where its dimension has more than one position
    const int64_t bs = N > 1 ? out->bs : 0, ts = B > 1 ? out->ts : 0, hs = Hl > 1 ? out->hs : 0;
    if (bs % 16 != 0 || ts % 16 != 0 || hs % 16 != 0) return KVR_ERR_ALIGNMENT;
    int64_t a = 0, b = 0, c = 0;
    if (!mul_fits({N - 1, bs}, &a) || !mul_fits({(int64_t)B - 1, ts}, &b) ||
        !mul_fits({(int64_t)Hl - 1, hs}, &c))
        return KVR_ERR_UNSUPPORTED;
    const __int128 span = (__int128)a + b + c + row;
    if (span > (__int128)INT64_MAX) return KVR_ERR_UNSUPPORTED;
    out->span = lay == nullptr ? plane : (int64_t)span;
    std::vector<std::pair<int64_t, int64_t>> dims;   // (stride, extent) of extent > 1
    if (N > 1) dims.push_back({bs, N});
    if (B > 1) dims.push_back({ts, B});
    if (Hl > 1) dims.push_back({hs, Hl});
    std::sort(dims.begin(), dims.end());
    out->inner = row;
    for (size_t k = 0; k + 1 < dims.size(); ++k) out->inner += (dims[k].second - 1) * dims[k].first;
    if (!dims.empty()) {
        out->outer_stride = dims.back().first;
        out->n_outer = dims.back().second;
    }
    for (uint64_t v : out->base)
        if (v > UINT64_MAX - (uint64_t)out->span) return KVR_ERR_UNSUPPORTED;
    return KVR_OK;
}

// Decode views must not alias: with the dimensions (of extent > 1) sorted by
// stride, each must step over everything the smaller ones span.
bool views_are_injective(int64_t N, int64_t bs, int64_t B, int64_t ts, int64_t Hl, int64_t hs,
                         int64_t row) {
    std::vector<std::pair<int64_t, int64_t>> dims;   // (stride, extent)
    if (N > 1) dims.push_back({bs, N});
    if (B > 1) dims.push_back({ts, B});
    if (Hl > 1) dims.push_back({hs, Hl});
    std::sort(dims.begin(), dims.end());
    __int128 inner = row;
    for (const auto &dm : dims) {
        if ((__int128)dm.first < inner) return false;
        inner += (__int128)(dm.second - 1) * dm.first;
    }
    return true;
}

// Do two views of one side (same strides, bases a and b) share a byte? Each
// is n_outer intervals of `inner` bytes, outer_stride apart; they meet iff a
// shift delta + k * outer_stride (|k| < n_outer) comes within `inner` of 0.
bool views_meet(uint64_t a, uint64_t b, const Side &sd) {
    const uint64_t delta = a > b ? a - b : b - a;
    const uint64_t inner = (uint64_t)sd.inner;
    if (sd.n_outer <= 1 || sd.outer_stride == 0) return delta < inner;
    const uint64_t so = (uint64_t)sd.outer_stride;
    const uint64_t q = delta / so, r = delta % so;
    if (q + 1 <= (uint64_t)sd.n_outer && r < inner) return true;
    if (q + 2 <= (uint64_t)sd.n_outer && so - r < inner) return true;
    return false;
}

// A decode view may share no byte with another decode view (exact test for
// views of equal strides) nor come near any prefill view (their spans may not
// intersect). Also returns each side's spans merged (for the device-access
// checks).
kvr_status check_regions(const Side &src, const Side &dst, std::vector<uint64_t> *src_merged,
                         std::vector<uint64_t> *dst_merged) {
    std::vector<uint64_t> db(dst.base);
    std::sort(db.begin(), db.end());
    for (size_t i = 0; i < db.size(); ++i)
        for (size_t j = i + 1; j < db.size() && db[j] < db[i] + (uint64_t)dst.span; ++j)
            if (views_meet(db[i], db[j], dst)) return KVR_ERR_POOL_OVERLAP;

    struct Reg {
        uint64_t lo, hi;
        bool dst;
    };
    std::vector<Reg> regs;
    regs.reserve(src.base.size() + dst.base.size());
    for (uint64_t b : src.base) regs.push_back({b, b + (uint64_t)src.span, false});
    for (uint64_t b : dst.base) regs.push_back({b, b + (uint64_t)dst.span, true});
    std::sort(regs.begin(), regs.end(), [](const Reg &x, const Reg &y) { return x.lo < y.lo; });
    uint64_t end_src = 0, end_dst = 0;
    for (const Reg &r : regs) {
        if (r.dst ? r.lo < end_src : r.lo < end_dst) return KVR_ERR_POOL_OVERLAP;
        (r.dst ? end_dst : end_src) = std::max(r.dst ? end_dst : end_src, r.hi);
    }
    for (int side = 0; side < 2; ++side) {
        std::vector<uint64_t> &m = side ? *dst_merged : *src_merged;
        m.clear();
        for (const Reg &r : regs) {
            if (r.dst != (side == 1)) continue;
            if (!m.empty() && r.lo <= m.back()) {
                m.back() = std::max(m.back(), r.hi);
            } else {
                m.push_back(r.lo);
                m.push_back(r.hi);
            }
        }
    }
    return KVR_OK;
}

}  // namespace

kvr_status kvr_build_host_plan(const kvr_desc *d, const kvr_layout *src_layout,
                               const kvr_layout *dst_layout, const kvr_convert *cv,
                               int sm_count, int layer_resident, int layer_resident_pf,
                               KvrHostPlan *hp, int64_t *bytes_read_out,
                               int64_t *bytes_written_out) {
    if (d == nullptr) return KVR_ERR_INVALID_ARG;
    const int32_t L = d->num_layers, C = d->num_components, H = d->kv_heads, D = d->head_dim;
    const int32_t es = d->elem_bytes, Tp = d->src_tp, Td = d->dst_tp;
    const int32_t Bp = d->src_block_size, Bd = d->dst_block_size, R = d->num_requests;
    const int64_t Np = d->src_num_blocks, Nd = d->dst_num_blocks;

    if (L < 1 || (C != 1 && C != 2) || H < 1 || D < 1 || Tp < 1 || Td < 1 || Bp < 1 ||
        Bd < 1 || Np < 1 || Nd < 1 || R < 0)
        return KVR_ERR_INVALID_ARG;
    if (es != 1 && es != 2 && es != 4) return KVR_ERR_UNSUPPORTED;
    if (Tp > KVR_MAX_TP || Td > KVR_MAX_TP) return KVR_ERR_UNSUPPORTED;
    if ((H % Tp != 0 && Tp % H != 0) || (H % Td != 0 && Td % H != 0)) return KVR_ERR_UNSUPPORTED;

    // element types: a bit copy, or BF16 <-> E4M3 with positive finite scales
    int32_t conv = KVR_CONV_NONE;
    int64_t es_dst = es;
    if (cv != nullptr) {
        const bool quant = cv->src_dtype == KVR_DTYPE_BF16 && cv->dst_dtype == KVR_DTYPE_FP8_E4M3;
        const bool dequant =
            cv->src_dtype == KVR_DTYPE_FP8_E4M3 && cv->dst_dtype == KVR_DTYPE_BF16;
        if (!quant && !dequant) return KVR_ERR_UNSUPPORTED;
        if (es != (quant ? 2 : 1)) return KVR_ERR_INVALID_ARG;
        if (cv->per_head != 0 && cv->per_head != 1) return KVR_ERR_INVALID_ARG;
        if (cv->scales == nullptr) return KVR_ERR_INVALID_ARG;
        const int64_t n_scales = (int64_t)L * C * (cv->per_head ? H : 1);
        for (int64_t i = 0; i < n_scales; ++i)
            if (!(cv->scales[i] > 0.0f) || !std::isfinite(cv->scales[i]))
                return KVR_ERR_INVALID_ARG;
        conv = quant ? KVR_CONV_BF16_TO_E4M3 : KVR_CONV_E4M3_TO_BF16;
        es_dst = quant ? 1 : 2;
    }
    int64_t src_row = 0, dst_row = 0;
    if (!mul_fits({D, es}, &src_row) || src_row > INT32_MAX || !mul_fits({D, es_dst}, &dst_row) ||
        dst_row > INT32_MAX)
        return KVR_ERR_UNSUPPORTED;
    if (src_row % 16 != 0 || dst_row % 16 != 0) return KVR_ERR_ALIGNMENT;
    // a unit is 16 bytes of a copied row, or 16 elements of a converted one
    const int64_t unit_src = conv == KVR_CONV_NONE ? 16 : 16 * (int64_t)es;
    const int64_t unit_dst = conv == KVR_CONV_NONE ? 16 : 16 * es_dst;
    const int64_t row_units = src_row / unit_src;
    // heads per shard, and shards per head (above 1 when T > H)
    const int32_t Hp = Tp <= H ? H / Tp : 1, Hd = Td <= H ? H / Td : 1;
    const int32_t scopies = Tp <= H ? 1 : Tp / H, dcopies = Td <= H ? 1 : Td / H;
    const int64_t Hx = (int64_t)H * dcopies;   // decode head rows per (token, component)

    // one item's units must stay below 2^31 (32-bit chunk indices)
    int64_t item_chunks = 0;
    if (!mul_fits({(int64_t)Bd, C, Hx, row_units}, &item_chunks) || item_chunks > INT32_MAX)
        return KVR_ERR_UNSUPPORTED;

    // the views of both sides
    Side src, dst;
    kvr_status st;
    try {
        st = make_side(src_layout, d->src_pools, Tp, L, C, Np, Bp, Hp, src_row, &src);
        if (st != KVR_OK) return st;
        st = make_side(dst_layout, d->dst_pools, Td, L, C, Nd, Bd, Hd, dst_row, &dst);
        if (st != KVR_OK) return st;
    } catch (const std::bad_alloc &) {
        return KVR_ERR_NOMEM;
    }
    if (!views_are_injective(Nd, dst.bs, Bd, dst.ts, Hd, dst.hs, dst_row))
        return KVR_ERR_POOL_OVERLAP;

    st = check_table(R, d->seq_lens, d->src_bt_offsets, d->src_bt, Bp, Np);
    if (st != KVR_OK) return st;
    st = check_table(R, d->seq_lens, d->dst_bt_offsets, d->dst_bt, Bd, Nd);
    if (st != KVR_OK) return st;

    // no decode block may receive two prompts' (or one prompt's two) tokens
    int64_t tokens = 0, used_src = 0;
    std::vector<int32_t> used;
    try {
        for (int32_t r = 0; r < R; ++r) {
            tokens += d->seq_lens[r];
            const int64_t nd = ceil_div(d->seq_lens[r], Bd);
            used_src += ceil_div(d->seq_lens[r], Bp);
            for (int64_t k = 0; k < nd; ++k) used.push_back(d->dst_bt[d->dst_bt_offsets[r] + k]);
        }
        std::sort(used.begin(), used.end());
    } catch (const std::bad_alloc &) {
        return KVR_ERR_NOMEM;
    }
    if (std::adjacent_find(used.begin(), used.end()) != used.end()) return KVR_ERR_DST_ALIAS;

    // decode views must not overlap each other or any prefill view
    std::vector<uint64_t> src_regions, dst_regions;
    try {
        st = check_regions(src, dst, &src_regions, &dst_regions);
    } catch (const std::bad_alloc &) {
        return KVR_ERR_NOMEM;
    }
    if (st != KVR_OK) return st;

    int64_t bytes_read = 0, bytes_written = 0;
    // each head is read once and written to every decode shard that holds it
    if (!mul_fits({tokens, (int64_t)L, C, H, src_row}, &bytes_read) ||
        !mul_fits({tokens, (int64_t)L, C, Hx, dst_row}, &bytes_written))
        return KVR_ERR_UNSUPPORTED;
    if (bytes_read_out) *bytes_read_out = bytes_read;
    if (bytes_written_out) *bytes_written_out = bytes_written;
    if (hp == nullptr) return KVR_OK;

    // token tiles: whole decode blocks, about KVR_TARGET_ITEM_BYTES read per layer
    // (a replicated head's rows count once per decode copy: each is a row to move)
    const int64_t blk_bytes_all_heads = (int64_t)Bd * C * Hx * src_row;
    int64_t per_tile = std::max<int64_t>(1, KVR_TARGET_ITEM_BYTES / blk_bytes_all_heads);
    per_tile = std::min<int64_t>(per_tile, INT32_MAX / ((int64_t)Bd * C * Hx * row_units));
    const int64_t tile = std::max<int64_t>(1, per_tile) * Bd;

    // launch sizes: CTAs = layers x items x slices must fit a 32-bit grid
    int64_t n_items = 0, used_dst = 0;
    for (int32_t r = 0; r < R; ++r) {
        n_items += ceil_div(d->seq_lens[r], tile);
        used_dst += ceil_div(d->seq_lens[r], Bd);
    }
    if (n_items > INT32_MAX || used_src > INT32_MAX || used_dst > INT32_MAX ||
        (int64_t)L * n_items > INT32_MAX)
        return KVR_ERR_UNSUPPORTED;

    KvrGeom &g = hp->g;
    g.L = L; g.C = C; g.H = H; g.Hp = Hp; g.Hd = Hd; g.Bp = Bp; g.Bd = Bd;
    g.scopies = scopies; g.dcopies = dcopies; g.Hx = (int32_t)Hx;
    g.win_rows = KVR_ROW_WINDOW / dcopies;          // a window holds every copy of its rows
    g.src_row_bytes = (int32_t)src_row;
    g.dst_row_bytes = (int32_t)dst_row;
    g.row_chunks = (int32_t)row_units;
    g.src_unit_bytes = (int32_t)unit_src;
    g.dst_unit_bytes = (int32_t)unit_dst;
    g.conv = conv;
    g.per_head = cv != nullptr ? cv->per_head : 0;
    g.div_rc = kvr_make_div((uint32_t)g.row_chunks);
    g.div_Hx = kvr_make_div((uint32_t)Hx);
    g.div_C = kvr_make_div((uint32_t)C);
    g.div_Hd = kvr_make_div((uint32_t)Hd);
    g.div_sgrp = kvr_make_div((uint32_t)(Hp * dcopies));
    g.div_dcop = kvr_make_div((uint32_t)dcopies);
    g.div_Bp = kvr_make_div((uint32_t)Bp);
    g.div_Bd = kvr_make_div((uint32_t)Bd);
    g.s_block_stride = src.bs;
    g.s_token_stride = src.ts;
    g.s_head_stride = src.hs;
    g.d_block_stride = dst.bs;
    g.d_token_stride = dst.ts;
    g.d_head_stride = dst.hs;
    hp->num_layers = L;
    hp->src_tp = Tp;
    hp->dst_tp = Td;
    hp->tile = (int32_t)tile;
    hp->src_base.swap(src.base);
    hp->dst_base.swap(dst.base);
    hp->src_regions.swap(src_regions);
    hp->dst_regions.swap(dst_regions);
    hp->bytes_read = bytes_read;
    hp->bytes_written = bytes_written;

    try {
        hp->items.clear();
        hp->sbt.clear();
        hp->dbt.clear();
        hp->items.reserve((size_t)n_items);
        hp->sbt.reserve((size_t)used_src);
        hp->dbt.reserve((size_t)used_dst);
        for (int32_t r = 0; r < R; ++r) {
            const int32_t n = d->seq_lens[r];
            if (n == 0) continue;
            const int32_t soff = (int32_t)hp->sbt.size();
            const int32_t doff = (int32_t)hp->dbt.size();
            for (int64_t k = 0; k < ceil_div(n, Bp); ++k)
                hp->sbt.push_back(d->src_bt[d->src_bt_offsets[r] + k]);
            for (int64_t k = 0; k < ceil_div(n, Bd); ++k)
                hp->dbt.push_back(d->dst_bt[d->dst_bt_offsets[r] + k]);
            for (int64_t t0 = 0; t0 < n; t0 += tile) {
                KvrItem it;
                it.sbt_off = soff;
                it.dbt_off = doff;
                it.t0 = (int32_t)t0;
                it.ntok = (int32_t)std::min<int64_t>(tile, n - t0);
                hp->items.push_back(it);
            }
        }
    } catch (const std::bad_alloc &) {
        return KVR_ERR_NOMEM;
    }

    try {
        hp->factors.clear();
        if (cv != nullptr) {
            const int64_t n_scales = (int64_t)L * C * (cv->per_head ? H : 1);
            for (int64_t i = 0; i < n_scales; ++i)
                hp->factors.push_back(conv == KVR_CONV_BF16_TO_E4M3 ? 1.0f / cv->scales[i]
                                                                    : cv->scales[i]);
        }
    } catch (const std::bad_alloc &) {
        return KVR_ERR_NOMEM;
    }

    // units of the prefill rows (each stored to all dcopies decode copies)
    hp->avg_chunks = n_items ? tokens * C * H * row_units / n_items : 0;
    hp->sm_count = sm_count;

    // Pairs of adjacent units per access (one 32-byte load or store where a unit
    // has 16 bytes): an even number of units per row, and every row of both
    // sides (every decode copy of a replicated head too) 32-byte aligned: view
    // bases, and the strides of dimensions with more than one position.
    auto aligned32 = [](const std::vector<uint64_t> &bases) {
        for (uint64_t b : bases)
            if (b % 32 != 0) return false;
        return true;
    };
    hp->pairs = row_units % 2 == 0 && aligned32(hp->src_base) &&
                aligned32(hp->dst_base) && (Np <= 1 || g.s_block_stride % 32 == 0) &&
                (Bp <= 1 || g.s_token_stride % 32 == 0) &&
                (Hp <= 1 || g.s_head_stride % 32 == 0) &&
                (Nd <= 1 || g.d_block_stride % 32 == 0) &&
                (Bd <= 1 || g.d_token_stride % 32 == 0) &&
                (Hd <= 1 || g.d_head_stride % 32 == 0);
    kvr_shape_launches(*hp, layer_resident, layer_resident_pf);
    return KVR_OK;
}

void kvr_shape_launches(KvrHostPlan &hp, int layer_resident, int layer_resident_pf) {
    const int64_t n_items = (int64_t)hp.items.size();
    hp.layer_resident = layer_resident;
    hp.layer_resident_pf = layer_resident_pf;
    hp.slices_layer = choose_layer_slices(n_items, hp.avg_chunks, hp.sm_count, layer_resident);
    // a layer whose items fit in one wave of the prefetching instance: its grid,
    // sized to fill that wave, stays within it (choose_layer_slices)
    hp.slices_layer_pf =
        layer_resident_pf > 0 && n_items < (int64_t)std::max(hp.sm_count, 1) * layer_resident_pf
            ? choose_layer_slices(n_items, hp.avg_chunks, hp.sm_count, layer_resident_pf)
            : 0;
    hp.slices_all = kvr_range_slices(hp, hp.num_layers, 0);
}

void kvr_range_launch(const KvrHostPlan &hp, int32_t count, int32_t stream_sms, bool no_wait,
                      int32_t *slices, int32_t *mode) {
    const int64_t tasks = (int64_t)count * (int64_t)hp.items.size();
    const bool limited = stream_sms > 0 && stream_sms < hp.sm_count;
    const int32_t sms = limited ? stream_sms : hp.sm_count;
    const int64_t slots = (int64_t)std::max(sms, 1) *
                          (hp.layer_resident > 0 ? hp.layer_resident : KVR_LAYER_CTAS_PER_SM);
    const int64_t slots_pf = (int64_t)std::max(sms, 1) * hp.layer_resident_pf;
    // A range of several layers takes the prefetching instance only if its grid
    // fills at least 3/4 of that wave; below that it runs the whole-prompt grid
    // (70B, 3 layers = 384 one-item CTAs on 608 slots: bit copy 5526 -> 5794,
    // BF16 -> FP8 4840 -> 5216, FP8 -> BF16 4565 -> 5335 GB/s; 2 and 4 layers,
    // 512 CTAs, keep it).
    const bool pf = !no_wait && tasks < slots_pf;
    const int32_t slices_pf =
        !pf ? 0
        : count == 1 && !limited
            ? hp.slices_layer_pf
            : choose_layer_slices(tasks, hp.avg_chunks, sms, hp.layer_resident_pf);
    if (pf && (count == 1 || 4 * tasks * slices_pf >= 3 * slots_pf)) {
        *slices = slices_pf;
        *mode = KVR_MODE_LAYER_PREFETCH;
    } else if (count == 1) {
        *slices = limited ? choose_layer_slices(tasks, hp.avg_chunks, sms, hp.layer_resident)
                          : hp.slices_layer;
        *mode = KVR_MODE_LAYER;
    } else if (!pf && tasks < slots) {
        *slices = choose_layer_slices(tasks, hp.avg_chunks, sms, hp.layer_resident);
        *mode = KVR_MODE_LAYER;
    } else {
        *slices = kvr_range_slices(hp, count, stream_sms);
        *mode = KVR_MODE_WHOLE;
    }
}

int32_t kvr_range_slices(const KvrHostPlan &hp, int32_t count, int32_t stream_sms) {
    const int64_t tasks = (int64_t)count * (int64_t)hp.items.size();
    const bool limited = stream_sms > 0 && stream_sms < hp.sm_count;
    int32_t s = choose_slices(tasks, hp.avg_chunks, limited ? stream_sms : hp.sm_count,
                              KVR_TARGET_CTAS_PER_SM);
    // large items (decode blocks of many tokens) of a bit copy or a dequantizing
    // relayout on the whole device are cut until a CTA moves at most
    // KVR_MAX_CTA_BYTES, so the grid does not end in a long partial wave; the
    // quantizing kernel measured faster with the larger CTAs, and so did every
    // launch on an SM-limited stream, so those stay whole (dequantizing: the cap
    // on bytes written with 4 units in flight per thread, 70B 6574 -> 6731,
    // Qwen 32K 6763 -> 6780 GB/s; either change alone lost)
    if (!limited && (hp.g.conv == KVR_CONV_NONE || hp.g.conv == KVR_CONV_E4M3_TO_BF16)) {
        // bytes written (a replicated head's unit is stored to every copy)
        const int64_t item_bytes = hp.avg_chunks * hp.g.dst_unit_bytes * hp.g.dcopies;
        const int64_t most = std::max<int64_t>(1, hp.avg_chunks / KVR_MIN_SLICE_CHUNKS);
        const int64_t want = std::min<int64_t>(most, ceil_div(item_bytes, KVR_MAX_CTA_BYTES));
        if (want > s) s = (int32_t)want;
    }
    while (tasks * s > INT32_MAX && s > 1) --s;
    return s;
}

uint32_t kvr_prefetch_ctas(const KvrHostPlan &hp, int32_t count, int32_t stream_sms, int32_t mode,
                           int32_t slices) {
    const bool limited = stream_sms > 0 && stream_sms < hp.sm_count;
    if (mode != KVR_MODE_LAYER_PREFETCH || count != 1 || limited) return 0xFFFFFFFFu;
    const uint64_t grid = (uint64_t)hp.items.size() * (uint64_t)slices;
    return (uint32_t)(grid * KVR_PREFETCH_CTAS_EIGHTHS / 8);
}

KvrArgs kvr_launch_args(const KvrHostPlan &hp, const KvrItem *dev_items, const int32_t *dev_sbt,
                        const int32_t *dev_dbt, const float *dev_factors,
                        const uint64_t *dev_src_base, const uint64_t *dev_dst_base,
                        int32_t layer0, int32_t slices) {
    KvrArgs a;
    memset(&a, 0, sizeof(a));
    a.g = hp.g;
    a.items = dev_items;
    a.sbt = dev_sbt;
    a.dbt = dev_dbt;
    a.factors = dev_factors;
    a.src_base = dev_src_base;
    a.dst_base = dev_dst_base;
    a.layer0 = layer0;
    a.slices = slices;
    a.tasks_per_layer = (uint32_t)(hp.items.size() * (size_t)slices);
    a.div_tasks_per_layer = kvr_make_div(a.tasks_per_layer ? a.tasks_per_layer : 1);
    a.div_slices = kvr_make_div((uint32_t)slices);
    a.prefetch_ctas = 0xFFFFFFFFu;
    return a;
}

kvr_status kvr_staging_extent(const kvr_desc *d, int64_t es, int64_t *total, int64_t *bytes) {
    if (d == nullptr || d->num_requests < 0 || (d->num_requests > 0 && d->seq_lens == nullptr) ||
        d->num_layers < 1 || (d->num_components != 1 && d->num_components != 2) ||
        d->kv_heads < 1 || d->head_dim < 1 || (es != 1 && es != 2 && es != 4))
        return KVR_ERR_INVALID_ARG;
    int64_t t = 0;
    for (int32_t r = 0; r < d->num_requests; ++r) {
        if (d->seq_lens[r] < 0) return KVR_ERR_INVALID_ARG;
        t += d->seq_lens[r];                 // at most 2^31 requests of < 2^31 tokens
    }
    int64_t b = 0;
    if (t > INT32_MAX ||
        !mul_fits({t, (int64_t)d->num_layers, d->num_components, d->kv_heads, d->head_dim, es},
                  &b))
        return KVR_ERR_UNSUPPORTED;
    *total = t;
    *bytes = b;
    return KVR_OK;
}

kvr_status kvr_staging_desc(const kvr_desc *desc, const void *staging, const kvr_convert *cv,
                            bool pack, KvrStaging *st, kvr_desc *out) {
    if (desc == nullptr || st == nullptr || out == nullptr) return KVR_ERR_INVALID_ARG;
    // element bytes of the buffer: the conversion (if any) happens on the way in
    int64_t es = desc->elem_bytes;
    if (pack && cv != nullptr) {
        if (cv->dst_dtype == KVR_DTYPE_BF16) es = 2;
        else if (cv->dst_dtype == KVR_DTYPE_FP8_E4M3) es = 1;
        else return KVR_ERR_UNSUPPORTED;
    }
    int64_t bytes = 0;
    const kvr_status s = kvr_staging_extent(desc, es, &st->total, &bytes);
    if (s != KVR_OK) return s;
    if (st->total == 0 || staging == nullptr) return KVR_ERR_INVALID_ARG;
    const int64_t row = (int64_t)desc->head_dim * es, tok = row * desc->kv_heads;
    const int64_t plane = st->total * tok;
    const int64_t views = (int64_t)desc->num_layers * desc->num_components;
    st->bases.resize((size_t)views);
    for (int64_t v = 0; v < views; ++v)
        st->bases[(size_t)v] = (const unsigned char *)staging + v * plane;
    st->off.assign((size_t)desc->num_requests + 1, 0);
    for (int32_t r = 0; r < desc->num_requests; ++r)
        st->off[(size_t)r + 1] = st->off[(size_t)r] + desc->seq_lens[r];
    st->ids.resize((size_t)st->total);
    for (int64_t k = 0; k < st->total; ++k) st->ids[(size_t)k] = (int32_t)k;
    st->layout.bases = st->bases.data();
    st->layout.block_stride = tok;
    st->layout.token_stride = tok;
    st->layout.head_stride = row;
    *out = *desc;
    if (pack) {
        out->dst_tp = 1;
        out->dst_block_size = 1;
        out->dst_num_blocks = st->total;
        out->dst_pools = nullptr;
        out->dst_bt_offsets = st->off.data();
        out->dst_bt = st->ids.data();
    } else {
        out->src_tp = 1;
        out->src_block_size = 1;
        out->src_num_blocks = st->total;
        out->src_pools = nullptr;
        out->src_bt_offsets = st->off.data();
        out->src_bt = st->ids.data();
    }
    return KVR_OK;
}

extern "C" kvr_status kv_relayout_staging_bytes(const kvr_desc *desc, int32_t elem_bytes,
                                                int64_t *bytes) {
    int64_t total = 0, b = 0;
    const kvr_status st = kvr_staging_extent(desc, elem_bytes, &total, &b);
    if (st == KVR_OK && bytes != nullptr) *bytes = b;
    return st;
}

extern "C" kvr_status kv_relayout_desc_bytes_ex(const kvr_desc *desc,
                                                const kvr_layout *src_layout,
                                                const kvr_layout *dst_layout,
                                                const kvr_convert *cv, int64_t *bytes_read,
                                                int64_t *bytes_written) {
    int64_t r = 0, w = 0;
    kvr_status st;
    try {
        st = kvr_build_host_plan(desc, src_layout, dst_layout, cv, 0, 0, 0, nullptr, &r, &w);
    } catch (...) {
        return KVR_ERR_NOMEM;
    }
    if (st != KVR_OK) return st;
    if (bytes_read) *bytes_read = r;
    if (bytes_written) *bytes_written = w;
    return KVR_OK;
}

extern "C" kvr_status kv_relayout_desc_convert_bytes(const kvr_desc *desc,
                                                     const kvr_convert *cv,
                                                     int64_t *bytes_read,
                                                     int64_t *bytes_written) {
    return kv_relayout_desc_bytes_ex(desc, nullptr, nullptr, cv, bytes_read, bytes_written);
}

extern "C" kvr_status kv_relayout_desc_bytes(const kvr_desc *desc, int64_t *bytes_read,
                                             int64_t *bytes_written) {
    return kv_relayout_desc_bytes_ex(desc, nullptr, nullptr, nullptr, bytes_read,
                                     bytes_written);
}

extern "C" const char *kv_relayout_strerror(kvr_status s) {
    switch (s) {
        case KVR_OK: return "ok";
        case KVR_ERR_INVALID_ARG: return "invalid argument";
        case KVR_ERR_UNSUPPORTED: return "unsupported geometry";
        case KVR_ERR_ALIGNMENT: return "pool or head row not 16-byte aligned";
        case KVR_ERR_BLOCK_RANGE: return "block id out of range";
        case KVR_ERR_TABLE_SHORT: return "block table shorter than the prompt";
        case KVR_ERR_DST_ALIAS: return "decode block id used twice";
        case KVR_ERR_LAYER_RANGE: return "layer out of range";
        case KVR_ERR_CUDA: return "CUDA runtime error";
        case KVR_ERR_NOMEM: return "out of memory";
        case KVR_ERR_POOL_OVERLAP: return "decode pool overlaps another pool";
        case KVR_ERR_SCRATCH_LIMIT: return "work list larger than the preallocated scratch";
        case KVR_ERR_POOL_ADDRESS: return "pool is not memory this GPU can access";
        case KVR_ERR_DEVICE_BOUNDS: return "a row fell outside its pools (checked build)";
    }
    return "unknown status";
}
