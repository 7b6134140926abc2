// plan.h -- host side of a relayout plan (no CUDA dependency).
#pragma once

#include <stdint.h>

#include <vector>

#include "kv_relayout.h"
#include "kvr_index.h"

// Launch shape of the relayout kernel.
#define KVR_THREADS 256          // threads per CTA
#define KVR_UNROLL 8             // 16-byte loads in flight per thread before its stores
// A launch aims at this many CTAs per SM; items are sliced until it does,
// but no slice gets fewer than KVR_MIN_SLICE_CHUNKS 16-byte chunks.
#define KVR_TARGET_CTAS_PER_SM 8
#define KVR_MIN_SLICE_CHUNKS 512

struct KvrHostPlan {
    KvrGeom g;
    int32_t num_layers = 0;
    int32_t src_tp = 0, dst_tp = 0;
    const void *src[KVR_MAX_TP] = {};
    void *dst[KVR_MAX_TP] = {};
    std::vector<KvrItem> items;        // (request, decode logical block) work items
    std::vector<int32_t> sbt;          // used prefill block ids, request after request
    int64_t bytes = 0;                 // bytes read (= bytes written) by one full relayout
    int32_t slices_all = 1;            // slices per item, whole-prompt launch
    int32_t slices_layer = 1;          // slices per item, per-layer launch
};

// Validate `d`; when `hp` is non-NULL also build the host plan for a device
// with `sm_count` SMs. Never touches device memory.
kvr_status kvr_build_host_plan(const kvr_desc *d, int sm_count, KvrHostPlan *hp,
                               int64_t *bytes);

// Kernel arguments of one launch: layers [layer0, layer0 + 1) or all layers.
KvrArgs kvr_launch_args(const KvrHostPlan &hp, const KvrItem *dev_items,
                        const int32_t *dev_sbt, int32_t layer0, int32_t slices);
