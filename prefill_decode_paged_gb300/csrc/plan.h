// plan.h -- host side of a relayout plan (no CUDA dependency).
#pragma once

#include <stdint.h>

#include <vector>

#include "kv_relayout.h"
#include "kvr_index.h"

// Launch shape of the relayout kernel (each may be overridden at build time).
#ifndef KVR_THREADS
#define KVR_THREADS 256          // threads per CTA
#endif
#ifndef KVR_UNROLL
#define KVR_UNROLL 8             // 16-byte loads in flight per thread before its stores
#endif
#ifndef KVR_UNROLL_LAYER
#define KVR_UNROLL_LAYER 8       // the same for per-layer bit-copy launches
#endif
#ifndef KVR_UNROLL_LAYER_CONVERT
#define KVR_UNROLL_LAYER_CONVERT 2  // per-layer FP8 -> BF16 launches (two stores per unit)
#endif
#ifndef KVR_UNROLL_LAYER_CONVERT_PAIRS
#define KVR_UNROLL_LAYER_CONVERT_PAIRS 4  // the same, pairs of units per access (2 pairs;
                                          // 70B ordered 5539 -> 5669, no wait 5746 -> 6198,
                                          // 8B / Qwen 32K / MLA layers +6 / +6 / +3 %)
#endif
#ifndef KVR_UNROLL_LAYER_QUANT
#define KVR_UNROLL_LAYER_QUANT 2    // per-layer BF16 -> FP8 launches: units (two loads each)
#endif
#ifndef KVR_UNROLL_LAYER_QUANT_PAIRS
#define KVR_UNROLL_LAYER_QUANT_PAIRS 4  // the same, pairs of units per access (2 pairs; 70B
                                        // with KVR_LAUNCH_NO_WAIT 5828 -> 6132, 8B layers
                                        // 6279 -> 6470, MLA 6618 -> 6726, Qwen 32K 6795 -> 6775)
#endif
#ifndef KVR_UNROLL_LAYER_QUANT_PF
#define KVR_UNROLL_LAYER_QUANT_PF 4 // the same, ordered one-wave launches (L2 prefetch)
#endif
#ifndef KVR_PREFETCH_CTAS_EIGHTHS
#define KVR_PREFETCH_CTAS_EIGHTHS 5  // single-layer ordered bit copies on the whole device:
                                     // eighths of the grid (the first CTAs) that prefetch
                                     // their rows to L2 (kvr_prefetch_ctas)
#endif
#ifndef KVR_ROW_WINDOW
#define KVR_ROW_WINDOW 1024      // rows whose pointers a CTA keeps in shared memory at once
#endif

// Units in flight per thread of the kernel instance for a conversion (KvrConv),
// a launch mode (KvrMode) and the access width (pairs: two units per access);
// a quantizing unit takes two loads, a dequantizing one two stores. The kernel's
// instances and the CPU emulation of its launches both read it. Measured on
// 70B layers (one GB300, GB/s), one unit per access: the prefetching quantizer
// with 4 units 5239, with 2 5075; the per-layer dequantizer with 2 units 4307
// (ordered) / 5620 (no wait), with 4 4163 / 5245, with 1 3755 / 4891, with 8
// (80 registers) 3805 / 4702, and 2 units also won on the multi-wave MLA, Qwen
// 32K and 8B layers; with pairs, 4 units (2 pairs) won in every per-layer
// instance (see the _PAIRS values above).
constexpr int kvr_units(int32_t conv, int32_t mode, bool pairs) {
    return conv == KVR_CONV_BF16_TO_E4M3
               ? (mode == KVR_MODE_LAYER_PREFETCH ? KVR_UNROLL_LAYER_QUANT_PF
                  : mode == KVR_MODE_WHOLE        ? KVR_UNROLL / 2
                  : pairs                         ? KVR_UNROLL_LAYER_QUANT_PAIRS
                                                  : KVR_UNROLL_LAYER_QUANT)
           : conv == KVR_CONV_E4M3_TO_BF16
               ? (mode == KVR_MODE_WHOLE ? KVR_UNROLL / 2
                  : pairs                ? KVR_UNROLL_LAYER_CONVERT_PAIRS
                                         : KVR_UNROLL_LAYER_CONVERT)
               : (mode == KVR_MODE_WHOLE ? KVR_UNROLL : KVR_UNROLL_LAYER);
}

// A whole-prompt launch aims at this many CTAs per SM; items are sliced until
// it does, but no slice gets fewer than KVR_MIN_SLICE_CHUNKS units. Per-layer
// launches are shaped by the kernel's occupancy (see choose_layer_slices);
// KVR_LAYER_CTAS_PER_SM stands in for it when it is unknown.
#ifndef KVR_TARGET_CTAS_PER_SM
#define KVR_TARGET_CTAS_PER_SM 8
#endif
#ifndef KVR_LAYER_CTAS_PER_SM
#define KVR_LAYER_CTAS_PER_SM 8
#endif
#ifndef KVR_MIN_SLICE_CHUNKS
#define KVR_MIN_SLICE_CHUNKS 512
#endif
// Whole-prompt (and multi-layer) bit-copy launches also slice items until no
// CTA reads more than this many bytes (items of large decode blocks).
#ifndef KVR_MAX_CTA_BYTES
#define KVR_MAX_CTA_BYTES (64 * 1024)
#endif
// Token tiles hold whole decode blocks and grow (in whole decode blocks)
// until a tile moves about this many bytes per layer.
#ifndef KVR_TARGET_ITEM_BYTES
#define KVR_TARGET_ITEM_BYTES (64 * 1024)
#endif

struct KvrHostPlan {
    KvrGeom g;
    int32_t num_layers = 0;
    int32_t src_tp = 0, dst_tp = 0;
    int32_t tile = 0;                  // tokens per work item (a multiple of Bd)
    std::vector<uint64_t> src_base;    // [Tp][L][C] addresses of the prefill views
    std::vector<uint64_t> dst_base;    // [Td][L][C] addresses of the decode views
    std::vector<uint64_t> src_regions; // merged [start, end) byte ranges the prefill views span
    std::vector<uint64_t> dst_regions; // the same for the decode side
    std::vector<KvrItem> items;        // (request, token tile) work items
    std::vector<int32_t> sbt;          // used prefill block ids, request after request
    std::vector<int32_t> dbt;          // used decode block ids, request after request
    std::vector<float> factors;        // conversion: 1/s (quantize) or s (dequantize)
    int64_t bytes_read = 0;            // bytes one full relayout reads
    int64_t bytes_written = 0;         // bytes one full relayout writes
    int32_t slices_all = 1;            // slices per item, whole-prompt launch
    int32_t slices_layer = 1;          // slices per item, per-layer launch
    int32_t slices_layer_pf = 0;       // the same for the prefetching instance (ordered
                                       // launches whose layer fits one wave of it; 0: none)
    int64_t avg_chunks = 0;            // average units of an item
    int32_t sm_count = 0;              // SMs of the device the plan was built for
    int32_t layer_resident = 0;        // CTAs of the per-layer kernel an SM holds (0: unknown)
    int32_t layer_resident_pf = 0;     // the same for its prefetching instance
    bool pairs = false;                // rows allow pairs of adjacent units per access
                                       // (32-byte accesses): see kvr_build_host_plan
};

// Whether a launch of mode `mode` (KvrMode) over `layers` layers of a plan moves
// pairs of units: every instance where the plan's rows allow it, except the bit
// copy's prefetching instance outside 2-layer ranges (its loads mostly hit L2;
// measured on 70B layers, single units against pairs: 1 layer 6190 / 6146 GB/s,
// 2 layers 6140 / 6457, 4 layers 6089 / 5485).
inline bool kvr_launch_pairs(bool plan_pairs, int32_t conv, int32_t mode, int32_t layers) {
    return plan_pairs &&
           !(conv == KVR_CONV_NONE && mode == KVR_MODE_LAYER_PREFETCH && layers != 2);
}

// Slices per item of a launch over `count` (>= 2) layers, shaped like a
// whole-prompt launch (count == num_layers gives slices_all). `stream_sms`:
// the SMs of the green context the launch's stream runs on (0: the whole
// device). On the whole device a bit copy's items are also cut to at most
// KVR_MAX_CTA_BYTES read per CTA (HBM-bound: balance pays); on fewer SMs the
// launch is latency-bound per SM and larger CTAs amortize their row-table
// prologue, so items are only sliced to fill those SMs.
int32_t kvr_range_slices(const KvrHostPlan &hp, int32_t count, int32_t stream_sms);

// Shape of a kv_relayout_layers() launch over `count` layers on a stream with
// `stream_sms` SMs (0 or the device's count: the whole device): slices per
// item, and the kernel instance (KvrMode). An ordered launch (no_wait false)
// whose (layer, item) tasks fit in one wave of the prefetching per-layer
// instance on those SMs runs that instance, shaped for it; otherwise one
// layer, or a range whose tasks fit in one wave of the per-layer instance
// (short and latency-bound like a single layer), runs the per-layer instance;
// longer ranges run the whole-prompt one. Per-layer grids on fewer SMs are
// shaped for those SMs (on 16-96 of 152 SMs, 80 ordered 70B layers ran 5-29 %
// faster than with the whole device's shape).
void kvr_range_launch(const KvrHostPlan &hp, int32_t count, int32_t stream_sms, bool no_wait,
                      int32_t *slices, int32_t *mode);

// SMs of the green context `stream` (a cudaStream_t) belongs to, or 0 when it
// belongs to none or the driver cannot say (sm_stream.cpp).
int32_t kvr_stream_green_sms(void *stream);

// Validate `d` with its layouts (NULL: the standard layout of d's pools) and
// the conversion `cv` (NULL: bit copy); when `hp` is non-NULL also build the
// host plan for a device with `sm_count` SMs. Never touches device memory.
// Either byte output may be NULL.
// `layer_resident` / `layer_resident_pf`: CTAs of the per-layer kernel and of
// its prefetching instance one SM holds at once (0 when unknown; 0 for the
// second: no prefetching launches), used to shape per-layer grids.
kvr_status kvr_build_host_plan(const kvr_desc *d, const kvr_layout *src_layout,
                               const kvr_layout *dst_layout, const kvr_convert *cv,
                               int sm_count, int layer_resident, int layer_resident_pf,
                               KvrHostPlan *hp, int64_t *bytes_read, int64_t *bytes_written);

// Per-layer and whole-prompt grid shapes of `hp` for per-layer kernel instances
// that hold `layer_resident` (and, prefetching, `layer_resident_pf`) CTAs per
// SM (kvr_build_host_plan calls it; a plan may reshape with the occupancy of
// the instances it will run).
void kvr_shape_launches(KvrHostPlan &hp, int layer_resident, int layer_resident_pf);

// KvrArgs::prefetch_ctas of a launch of `count` layers on a stream of
// `stream_sms` SMs (0: the whole device) that kvr_range_launch gave `mode` and
// `slices`: the first KVR_PREFETCH_CTAS_EIGHTHS / 8 of the grid for a
// single-layer launch of the prefetching instance on the whole device, every
// CTA otherwise (measured on 70B layers: whole device 6201 -> 6320 GB/s; on
// streams of 48-112 SMs the same cut lost up to 8 %, on 128 SMs it gained 4 %;
// ranges of 2-4 layers lost 1 %).
uint32_t kvr_prefetch_ctas(const KvrHostPlan &hp, int32_t count, int32_t stream_sms, int32_t mode,
                           int32_t slices);

// Kernel arguments of one launch starting at layer `layer0`.
KvrArgs kvr_launch_args(const KvrHostPlan &hp, const KvrItem *dev_items,
                        const int32_t *dev_sbt, const int32_t *dev_dbt,
                        const float *dev_factors, const uint64_t *dev_src_base,
                        const uint64_t *dev_dst_base, int32_t layer0, int32_t slices);

// The staging side of a pack or unpack plan (kv_relayout_plan_pack/_unpack): a
// contiguous [L][C][sum n][H][D] buffer seen as a single shard of one-token
// blocks, request r's tokens from sum(n[:r]) on, so a block id is the token's
// row in the buffer. `layout` points into `bases`.
struct KvrStaging {
    std::vector<const void *> bases;   // [L][C] view bases
    std::vector<int64_t> off;          // CSR offsets: prefix sums of the prompt lengths
    std::vector<int32_t> ids;          // 0 .. sum n - 1
    kvr_layout layout;
    int64_t total = 0;                 // tokens in the batch
};

// Tokens of d's batch and the bytes of its staging buffer for `es`-byte elements
// (host only; validates the fields it reads).
kvr_status kvr_staging_extent(const kvr_desc *d, int64_t es, int64_t *total, int64_t *bytes);

// *out = *desc with its decode side (pack) or prefill side (unpack) replaced by
// the staging buffer `staging`, whose layout *st receives (pass it as that side's
// kvr_layout). The staging buffer holds the decode dtype when packing, the
// prefill dtype (desc->elem_bytes) when unpacking.
kvr_status kvr_staging_desc(const kvr_desc *desc, const void *staging, const kvr_convert *cv,
                            bool pack, KvrStaging *st, kvr_desc *out);
