// relayout.cu -- fused gather -> head re-shard -> scatter of paged KV cache (sm_103a).
//
// One kernel does the whole hand-off of the page "PD 分离与 KV 传输"
// (ai-infra-handbooks, serving/distributed/pd-disagg; sections "实现" and
// "布局转换"): each 16-byte chunk of a head row is read from the prefill
// shard that holds the head, at the row the prefill block table gives for
// the token, and written to the decode shard that holds the head, at the row
// the decode block table gives. There is no intermediate buffer: the gather,
// the TP re-shard and the scatter are one load and one store per chunk.
//
// It is pure data movement (no arithmetic on the values, no tensor cores),
// bound by HBM bandwidth: every chunk is read once and written once, so the
// DRAM traffic floor is 2 x (KV bytes of the prompts). The kernel keeps
// KVR_UNROLL independent 16-byte loads in flight per thread before their
// stores, uses streaming cache hints on both sides (neither the prefill rows
// nor the decode rows are touched again by this kernel), and opts into
// programmatic dependent launch so back-to-back per-layer launches overlap
// their launch latency with the previous launch's tail.
#include <cuda_runtime.h>

#include <new>

#include "kv_relayout.h"
#include "kvr_index.h"
#include "plan.h"

struct kvr_plan {
    KvrHostPlan host;
    void *dev_meta = nullptr;       // items, then prefill and decode block ids
    const KvrItem *dev_items = nullptr;
    const int32_t *dev_sbt = nullptr;
    const int32_t *dev_dbt = nullptr;
    int device = 0;
};

namespace {

__device__ __forceinline__ uint4 load_stream(const unsigned char *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void store_stream(unsigned char *p, const uint4 &v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// U: 16-byte loads each thread keeps in flight before its stores.
template <int U>
__global__ void __launch_bounds__(KVR_THREADS)
    kvr_relayout_kernel(const __grid_constant__ KvrArgs a) {
    // (prefill row address, decode row address) of the rows this CTA copies
    __shared__ ulonglong2 rows[KVR_ROW_WINDOW];

    // Wait for the grid this launch follows in its stream (a no-op without
    // programmatic dependent launch), then let the next launch start early.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");

    int32_t layer;
    KvrItem it;
    uint32_t q0, q1;
    kvr_task(a, blockIdx.x, a.items, &layer, &it, &q0, &q1);
    if (q0 >= q1) return;
    const uint32_t rc = (uint32_t)a.g.row_chunks;
    const uint32_t r_end = a.g.div_rc.div(q1 - 1) + 1;

    for (uint32_t w0 = a.g.div_rc.div(q0); w0 < r_end; w0 += KVR_ROW_WINDOW) {
        const uint32_t w1 = min(w0 + (uint32_t)KVR_ROW_WINDOW, r_end);
        // 1. one thread per row: the row's two addresses (block tables read here)
        for (uint32_t r = w0 + threadIdx.x; r < w1; r += KVR_THREADS) {
            uint32_t sp, dp;
            int64_t soff, doff;
            kvr_row(a.g, layer, it, a.sbt, a.dbt, r, &sp, &soff, &dp, &doff);
            rows[r - w0] = make_ulonglong2((unsigned long long)(a.src[sp] + soff),
                                           (unsigned long long)(a.dst[dp] + doff));
        }
        __syncthreads();
        // 2. the 16-byte chunks of those rows: U loads in flight per thread
        const uint32_t qa = max(q0, w0 * rc), qb = min(q1, w1 * rc);
        for (uint32_t base = qa + threadIdx.x; base < qb; base += U * KVR_THREADS) {
            uint4 v[U];
            unsigned char *to[U];
#pragma unroll
            for (int k = 0; k < U; ++k) {
                const uint32_t q = base + (uint32_t)k * KVR_THREADS;
                to[k] = nullptr;
                if (q < qb) {
                    const uint32_t r = a.g.div_rc.div(q);
                    const uint32_t off = (q - r * rc) * 16u;
                    const ulonglong2 p = rows[r - w0];
                    v[k] = load_stream((const unsigned char *)p.x + off);
                    to[k] = (unsigned char *)p.y + off;
                }
            }
#pragma unroll
            for (int k = 0; k < U; ++k)
                if (to[k] != nullptr) store_stream(to[k], v[k]);
        }
        __syncthreads();
    }
}

kvr_status launch(const kvr_plan *p, int32_t layer0, int32_t layers, int32_t slices,
                  bool per_layer, void *stream) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVR_ERR_CUDA;
    if (dev != p->device) return KVR_ERR_INVALID_ARG;
    const KvrArgs a =
        kvr_launch_args(p->host, p->dev_items, p->dev_sbt, p->dev_dbt, layer0, slices);
    const uint64_t grid = (uint64_t)layers * a.tasks_per_layer;
    if (grid == 0) return KVR_OK;

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
    const cudaError_t e = per_layer
                              ? cudaLaunchKernelEx(&cfg, kvr_relayout_kernel<KVR_UNROLL_LAYER>, a)
                              : cudaLaunchKernelEx(&cfg, kvr_relayout_kernel<KVR_UNROLL>, a);
    return e == cudaSuccess ? KVR_OK : KVR_ERR_CUDA;
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
    const int64_t layers_comps = (int64_t)hp.num_layers * hp.g.C;
    for (int32_t s = 0; s < hp.src_tp; ++s) {
        const kvr_status st = check_pool(hp.src[s], hp.g.src_plane_bytes * layers_comps, dev);
        if (st != KVR_OK) return st;
    }
    for (int32_t s = 0; s < hp.dst_tp; ++s) {
        const kvr_status st = check_pool(hp.dst[s], hp.g.dst_plane_bytes * layers_comps, dev);
        if (st != KVR_OK) return st;
    }
    return KVR_OK;
}

}  // namespace

extern "C" kvr_status kv_relayout_plan(const kvr_desc *desc, kvr_plan **out) {
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
        st = kvr_build_host_plan(desc, sms, &p->host, nullptr);
    } catch (...) {
        st = KVR_ERR_NOMEM;
    }
    if (st == KVR_OK) st = check_pools(p->host, dev);
    if (st != KVR_OK) {
        delete p;
        return st;
    }
    p->device = dev;
    const size_t items_bytes = p->host.items.size() * sizeof(KvrItem);
    const size_t sbt_bytes = p->host.sbt.size() * sizeof(int32_t);
    const size_t dbt_bytes = p->host.dbt.size() * sizeof(int32_t);
    if (items_bytes > 0) {
        if (cudaMalloc(&p->dev_meta, items_bytes + sbt_bytes + dbt_bytes) != cudaSuccess) {
            cudaGetLastError();
            delete p;
            return KVR_ERR_NOMEM;
        }
        unsigned char *base = (unsigned char *)p->dev_meta;
        if (cudaMemcpy(base, p->host.items.data(), items_bytes, cudaMemcpyHostToDevice) !=
                cudaSuccess ||
            cudaMemcpy(base + items_bytes, p->host.sbt.data(), sbt_bytes,
                       cudaMemcpyHostToDevice) != cudaSuccess ||
            cudaMemcpy(base + items_bytes + sbt_bytes, p->host.dbt.data(), dbt_bytes,
                       cudaMemcpyHostToDevice) != cudaSuccess) {
            cudaFree(p->dev_meta);
            delete p;
            return KVR_ERR_CUDA;
        }
        p->dev_items = (const KvrItem *)base;
        p->dev_sbt = (const int32_t *)(base + items_bytes);
        p->dev_dbt = (const int32_t *)(base + items_bytes + sbt_bytes);
    }
    *out = p;
    return KVR_OK;
}

extern "C" kvr_status kv_relayout_layer(const kvr_plan *plan, int32_t layer, void *stream) {
    if (plan == nullptr) return KVR_ERR_INVALID_ARG;
    if (layer < 0 || layer >= plan->host.num_layers) return KVR_ERR_LAYER_RANGE;
    return launch(plan, layer, 1, plan->host.slices_layer, true, stream);
}

extern "C" kvr_status kv_relayout_all(const kvr_plan *plan, void *stream) {
    if (plan == nullptr) return KVR_ERR_INVALID_ARG;
    return launch(plan, 0, plan->host.num_layers, plan->host.slices_all, false, stream);
}

extern "C" kvr_status kv_relayout_plan_bytes(const kvr_plan *plan, int64_t *bytes_read,
                                             int64_t *bytes_written) {
    if (plan == nullptr) return KVR_ERR_INVALID_ARG;
    if (bytes_read) *bytes_read = plan->host.bytes;
    if (bytes_written) *bytes_written = plan->host.bytes;
    return KVR_OK;
}

extern "C" void kv_relayout_plan_destroy(kvr_plan *plan) {
    if (plan == nullptr) return;
    if (plan->dev_meta != nullptr) cudaFree(plan->dev_meta);
    delete plan;
}

// ---------------------------------------------------------------------------
// kv_relayout_all_prealloc: the whole-prompt relayout without any device
// allocation. The kernel's scratch (the work list and the used prefill block
// ids, normally in the plan's cudaMalloc'd buffer) lives in the file-scope
// array below instead. Every GPU that loads this library holds the array
// until the process exits.
// ---------------------------------------------------------------------------
#include <mutex>

#define KVR_PREALLOC_MAX_DEVICES 64

static __device__ __align__(256) unsigned char g_kvr_prealloc_scratch[KVR_PREALLOC_SCRATCH_BYTES];

namespace {

struct PreallocScratch {
    bool ready = false;
    unsigned char *addr = nullptr;   // device address of g_kvr_prealloc_scratch
    int sms = 0;
};

PreallocScratch g_prealloc[KVR_PREALLOC_MAX_DEVICES];
std::mutex g_prealloc_mu;

// Once per device, with that device current: the array's device address. In
// host code the array's name is only a host-side stand-in, so the kernel must
// be given this address, never the name.
kvr_status prealloc_setup(int dev, PreallocScratch *out) {
    std::lock_guard<std::mutex> lock(g_prealloc_mu);
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
    *out = s;
    return KVR_OK;
}

}  // namespace

extern "C" kvr_status kv_relayout_all_prealloc(const kvr_desc *desc, void *stream) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KVR_ERR_CUDA;
    if (dev < 0 || dev >= KVR_PREALLOC_MAX_DEVICES) return KVR_ERR_UNSUPPORTED;
    PreallocScratch sc;
    kvr_status st = prealloc_setup(dev, &sc);
    if (st != KVR_OK) return st;

    KvrHostPlan hp;
    try {
        st = kvr_build_host_plan(desc, sc.sms, &hp, nullptr);
    } catch (...) {
        st = KVR_ERR_NOMEM;
    }
    if (st == KVR_OK) st = check_pools(hp, dev);
    if (st != KVR_OK) return st;
    const size_t items_bytes = hp.items.size() * sizeof(KvrItem);
    const size_t sbt_bytes = hp.sbt.size() * sizeof(int32_t);
    const size_t dbt_bytes = hp.dbt.size() * sizeof(int32_t);
    if (items_bytes + sbt_bytes + dbt_bytes > KVR_PREALLOC_SCRATCH_BYTES)
        return KVR_ERR_SCRATCH_LIMIT;
    if (items_bytes == 0) return KVR_OK;

    // The whole array is overwritten up to what this call reads, so nothing
    // needs clearing; the copies are ordered before the launch on `stream`.
    cudaStream_t s = (cudaStream_t)stream;
    if (cudaMemcpyAsync(sc.addr, hp.items.data(), items_bytes, cudaMemcpyHostToDevice, s) !=
            cudaSuccess ||
        cudaMemcpyAsync(sc.addr + items_bytes, hp.sbt.data(), sbt_bytes,
                        cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(sc.addr + items_bytes + sbt_bytes, hp.dbt.data(), dbt_bytes,
                        cudaMemcpyHostToDevice, s) != cudaSuccess)
        return KVR_ERR_CUDA;

    const KvrArgs a = kvr_launch_args(hp, (const KvrItem *)sc.addr,
                                      (const int32_t *)(sc.addr + items_bytes),
                                      (const int32_t *)(sc.addr + items_bytes + sbt_bytes), 0,
                                      hp.slices_all);
    const uint64_t grid = (uint64_t)hp.num_layers * a.tasks_per_layer;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(KVR_THREADS, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kvr_relayout_kernel<KVR_UNROLL>, a) == cudaSuccess
               ? KVR_OK
               : KVR_ERR_CUDA;
}
