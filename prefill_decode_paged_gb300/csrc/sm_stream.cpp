// sm_stream.cpp -- a stream whose kernels run on a limited number of SMs.
//
// Page "PD multiplexing: splitting prefill and decode by SM on one GPU"
// (ai-infra-handbooks, en/serving/frontier/pd-multiplex), section "Green
// contexts: carving out SMs for a stream": a green context owns part of the
// device's SMs, and kernels submitted to a stream created on it run only on
// those SMs; memory-bound work such as decode gets near the bandwidth limit
// with a small share of SMs. The relayout is memory-bound too: handing it a
// stream with a few SMs leaves the rest to the model's compute, and sweeping
// the SM count measures how many SMs it needs to saturate HBM.
//
// The driver entry points are looked up through the runtime
// (cudaGetDriverEntryPointByVersion, at the ABI version of the CUDA headers
// this file is compiled with: cuGreenCtxStreamCreate has no 12.4 version), so
// the library does not link libcuda.
#include <cuda.h>
#include <cuda_runtime.h>

#include <new>

#include "kv_relayout.h"
#include "plan.h"

struct kvr_sm_stream {
    CUgreenCtx ctx = nullptr;
    CUstream stream = nullptr;
};

namespace {

using PFN_DeviceGet = CUresult (*)(CUdevice *, int);
using PFN_DeviceGetDevResource = CUresult (*)(CUdevice, CUdevResource *, CUdevResourceType);
using PFN_DevSmResourceSplitByCount = CUresult (*)(CUdevResource *, unsigned int *,
                                                   const CUdevResource *, CUdevResource *,
                                                   unsigned int, unsigned int);
using PFN_DevResourceGenerateDesc = CUresult (*)(CUdevResourceDesc *, CUdevResource *,
                                                 unsigned int);
using PFN_GreenCtxCreate = CUresult (*)(CUgreenCtx *, CUdevResourceDesc, CUdevice, unsigned int);
using PFN_GreenCtxStreamCreate = CUresult (*)(CUstream *, CUgreenCtx, unsigned int, int);
using PFN_GreenCtxDestroy = CUresult (*)(CUgreenCtx);
using PFN_StreamDestroy = CUresult (*)(CUstream);

struct Driver {
    PFN_DeviceGet device_get = nullptr;
    PFN_DeviceGetDevResource get_resource = nullptr;
    PFN_DevSmResourceSplitByCount split = nullptr;
    PFN_DevResourceGenerateDesc generate_desc = nullptr;
    PFN_GreenCtxCreate ctx_create = nullptr;
    PFN_GreenCtxStreamCreate stream_create = nullptr;
    PFN_GreenCtxDestroy ctx_destroy = nullptr;
    PFN_StreamDestroy stream_destroy = nullptr;
};

template <typename F>
bool entry(const char *name, F *fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &p, CUDART_VERSION, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || p == nullptr) {
        cudaGetLastError();
        return false;
    }
    *fn = reinterpret_cast<F>(p);
    return true;
}

bool load(Driver *d) {
    return entry("cuDeviceGet", &d->device_get) &&
           entry("cuDeviceGetDevResource", &d->get_resource) &&
           entry("cuDevSmResourceSplitByCount", &d->split) &&
           entry("cuDevResourceGenerateDesc", &d->generate_desc) &&
           entry("cuGreenCtxCreate", &d->ctx_create) &&
           entry("cuGreenCtxStreamCreate", &d->stream_create) &&
           entry("cuGreenCtxDestroy", &d->ctx_destroy) &&
           entry("cuStreamDestroy", &d->stream_destroy);
}

using PFN_StreamGetGreenCtx = CUresult (*)(CUstream, CUgreenCtx *);
using PFN_GreenCtxGetDevResource = CUresult (*)(CUgreenCtx, CUdevResource *, CUdevResourceType);

struct GreenQuery {
    PFN_StreamGetGreenCtx stream_green = nullptr;
    PFN_GreenCtxGetDevResource resource = nullptr;
    bool ok = false;
};

GreenQuery load_query() {
    GreenQuery q;
    q.ok = entry("cuStreamGetGreenCtx", &q.stream_green) &&
           entry("cuGreenCtxGetDevResource", &q.resource);
    return q;
}

}  // namespace

int32_t kvr_stream_green_sms(void *stream) {
    static const GreenQuery q = load_query();
    if (!q.ok || stream == nullptr) return 0;
    CUgreenCtx g = nullptr;
    if (q.stream_green((CUstream)stream, &g) != CUDA_SUCCESS || g == nullptr) return 0;
    CUdevResource r;
    if (q.resource(g, &r, CU_DEV_RESOURCE_TYPE_SM) != CUDA_SUCCESS) return 0;
    return (int32_t)r.sm.smCount;
}

extern "C" kvr_status kv_relayout_sm_stream_create(int32_t sm_count, kvr_sm_stream **out,
                                                   void **stream, int32_t *sms_granted) {
    if (out == nullptr || stream == nullptr) return KVR_ERR_INVALID_ARG;
    *out = nullptr;
    *stream = nullptr;
    if (sm_count < 1) return KVR_ERR_INVALID_ARG;
    int dev = 0, total = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&total, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return KVR_ERR_CUDA;
    if (sm_count > total) return KVR_ERR_INVALID_ARG;
    Driver d;
    if (!load(&d)) return KVR_ERR_UNSUPPORTED;

    CUdevice cudev;
    CUdevResource all, part, rest;
    if (d.device_get(&cudev, dev) != CUDA_SUCCESS ||
        d.get_resource(cudev, &all, CU_DEV_RESOURCE_TYPE_SM) != CUDA_SUCCESS)
        return KVR_ERR_CUDA;
    CUdevResource *use = &all;
    if (sm_count < total) {
        unsigned int groups = 1;
        if (d.split(&part, &groups, &all, &rest, 0, (unsigned int)sm_count) != CUDA_SUCCESS ||
            groups != 1)
            return KVR_ERR_UNSUPPORTED;
        use = &part;
    }
    CUdevResourceDesc desc;
    if (d.generate_desc(&desc, use, 1) != CUDA_SUCCESS) return KVR_ERR_CUDA;
    kvr_sm_stream *s = new (std::nothrow) kvr_sm_stream();
    if (s == nullptr) return KVR_ERR_NOMEM;
    if (d.ctx_create(&s->ctx, desc, cudev, CU_GREEN_CTX_DEFAULT_STREAM) != CUDA_SUCCESS) {
        delete s;
        return KVR_ERR_CUDA;
    }
    if (d.stream_create(&s->stream, s->ctx, CU_STREAM_NON_BLOCKING, 0) != CUDA_SUCCESS) {
        d.ctx_destroy(s->ctx);
        delete s;
        return KVR_ERR_CUDA;
    }
    if (sms_granted != nullptr) *sms_granted = (int32_t)use->sm.smCount;
    *out = s;
    *stream = (void *)s->stream;
    return KVR_OK;
}

extern "C" void kv_relayout_sm_stream_destroy(kvr_sm_stream *s) {
    if (s == nullptr) return;
    Driver d;
    if (load(&d)) {
        if (s->stream != nullptr) d.stream_destroy(s->stream);
        if (s->ctx != nullptr) d.ctx_destroy(s->ctx);
    }
    delete s;
}
