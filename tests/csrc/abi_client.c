/* abi_client.c -- a plain C99 client of the relayout's C ABI (test harness).
 *
 * Built with gcc -std=c99 against include/kv_relayout.h alone and linked to
 * the library, it shows that the ABI needs neither C++ nor Python nor torch.
 *
 *   abi_client host   validation and byte counts on fake pool addresses (no GPU)
 *   abi_client gpu    pools from cudaMalloc; whole-prompt, per-layer and layer
 *                     range launches checked byte for byte against the C oracle;
 *                     pack into a staging buffer (checked against the oracle's
 *                     gather into [L][C][sum n][H][D]) and unpack from it (checked
 *                     against the oracle's direct relayout)
 *
 * Exit status 0 on success; a message on stderr otherwise.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "kv_relayout.h"

/* The CPU oracle (oracle/kv_oracle.c), declared here: it has no header. */
int kvo_relayout(int32_t layer_begin, int32_t layer_end, int32_t num_layers,
                 int32_t num_components, int32_t kv_heads, int32_t head_dim, int32_t elem_bytes,
                 int32_t src_tp, int32_t dst_tp, int32_t src_block, int32_t dst_block,
                 int64_t src_num_blocks, int64_t dst_num_blocks,
                 const uint8_t *const *src_pools, uint8_t *const *dst_pools,
                 int32_t num_requests, const int32_t *seq_lens, const int64_t *src_off,
                 const int32_t *src_bt, const int64_t *dst_off, const int32_t *dst_bt);

/* The oracle on any layout (per-(shard, layer, component) view bases and strides). */
int kvo_relayout_general(int32_t layer_begin, int32_t layer_end, int32_t num_layers,
                         int32_t num_components, int32_t kv_heads, int32_t head_dim,
                         int32_t src_dtype, int32_t dst_dtype, int32_t elem_bytes,
                         int32_t per_head, const float *scales, int32_t src_tp, int32_t dst_tp,
                         int32_t src_block, int32_t dst_block, const uint64_t *src_base,
                         int64_t s_block_stride, int64_t s_token_stride, int64_t s_head_stride,
                         const uint64_t *dst_base, int64_t d_block_stride,
                         int64_t d_token_stride, int64_t d_head_stride, int32_t num_requests,
                         const int32_t *seq_lens, const int64_t *src_off, const int32_t *src_bt,
                         const int64_t *dst_off, const int32_t *dst_bt);

#include <cuda_runtime_api.h>
#define H2D cudaMemcpyHostToDevice
#define D2H cudaMemcpyDeviceToHost

#define FAIL(...)                                   \
    do {                                            \
        fprintf(stderr, "abi_client: " __VA_ARGS__); \
        fprintf(stderr, "\n");                      \
        return 1;                                   \
    } while (0)

/* Geometry: L2 C2 H8 D64 bf16-sized elements, prefill TP4 block 16, decode TP2
 * block 64, three prompts (one empty), tables from a fixed shuffle. */
enum { L = 3, C = 2, H = 8, D = 64, ES = 2, TP_S = 4, TP_D = 2, BP = 16, BD = 64, R = 3 };
static const int32_t lens[R] = {300, 0, 77};
#define NP 40
#define ND 12

static uint32_t lcg(uint32_t *s) {
    *s = *s * 1664525u + 1013904223u;
    return *s >> 8;
}

static void shuffle(int32_t *a, int n, uint32_t seed) {
    int i;
    for (i = 0; i < n; ++i) a[i] = i;
    for (i = n - 1; i > 0; --i) {
        int j = (int)(lcg(&seed) % (uint32_t)(i + 1));
        int32_t t = a[i];
        a[i] = a[j];
        a[j] = t;
    }
}

static int64_t src_off[R + 1], dst_off[R + 1];
static int32_t src_bt[NP], dst_bt[ND];

static void tables(void) {
    int32_t perm_s[NP], perm_d[ND];
    int r, k, ps = 0, pd = 0;
    shuffle(perm_s, NP, 7u);
    shuffle(perm_d, ND, 11u);
    src_off[0] = dst_off[0] = 0;
    for (r = 0; r < R; ++r) {
        int ns = (lens[r] + BP - 1) / BP, nd = (lens[r] + 1 + BD - 1) / BD; /* +1: reserve */
        if (lens[r] == 0) nd = 0;
        for (k = 0; k < ns; ++k) src_bt[ps + k] = perm_s[ps + k];
        for (k = 0; k < nd; ++k) dst_bt[pd + k] = perm_d[pd + k];
        ps += ns;
        pd += nd;
        src_off[r + 1] = ps;
        dst_off[r + 1] = pd;
    }
}

static void describe(kvr_desc *d, void *const *src, void *const *dst) {
    memset(d, 0, sizeof(*d));
    d->num_layers = L;
    d->num_components = C;
    d->kv_heads = H;
    d->head_dim = D;
    d->elem_bytes = ES;
    d->src_tp = TP_S;
    d->dst_tp = TP_D;
    d->src_block_size = BP;
    d->dst_block_size = BD;
    d->src_num_blocks = NP;
    d->dst_num_blocks = ND;
    d->src_pools = (const void *const *)src;
    d->dst_pools = dst;
    d->num_requests = R;
    d->seq_lens = lens;
    d->src_bt_offsets = src_off;
    d->src_bt = src_bt;
    d->dst_bt_offsets = dst_off;
    d->dst_bt = dst_bt;
}

static const int64_t src_pool_bytes = (int64_t)L * C * NP * BP * (H / TP_S) * D * ES;
static const int64_t dst_pool_bytes = (int64_t)L * C * ND * BD * (H / TP_D) * D * ES;

static int host_mode(void) {
    void *src[TP_S], *dst[TP_D];
    kvr_desc d;
    int64_t r = -1, w = -1;
    int s;
    kvr_status st;
    for (s = 0; s < TP_S; ++s) src[s] = (void *)(uintptr_t)(((uint64_t)1 << 40) + s * ((uint64_t)1 << 30));
    for (s = 0; s < TP_D; ++s) dst[s] = (void *)(uintptr_t)(((uint64_t)1 << 41) + s * ((uint64_t)1 << 30));
    describe(&d, src, dst);
    st = kv_relayout_desc_bytes(&d, &r, &w);
    if (st != KVR_OK) FAIL("desc_bytes: %s", kv_relayout_strerror(st));
    if (r != (int64_t)(300 + 77) * L * C * H * D * ES || w != r)
        FAIL("byte count %lld/%lld", (long long)r, (long long)w);
    /* documented errors */
    d.dst_tp = 3;
    if (kv_relayout_desc_bytes(&d, &r, &w) != KVR_ERR_UNSUPPORTED) FAIL("H %% Td accepted");
    d.dst_tp = TP_D;
    src[1] = (void *)((uintptr_t)src[1] + 8);
    if (kv_relayout_desc_bytes(&d, &r, &w) != KVR_ERR_ALIGNMENT) FAIL("misaligned pool accepted");
    src[1] = (void *)((uintptr_t)src[1] - 8);
    dst_bt[1] = dst_bt[0];
    if (kv_relayout_desc_bytes(&d, &r, &w) != KVR_ERR_DST_ALIAS) FAIL("decode alias accepted");
    tables();
    dst_bt[0] = ND;
    if (kv_relayout_desc_bytes(&d, &r, &w) != KVR_ERR_BLOCK_RANGE) FAIL("block id accepted");
    tables();
    dst[1] = (void *)((uintptr_t)dst[0] + 64);
    if (kv_relayout_desc_bytes(&d, &r, &w) != KVR_ERR_POOL_OVERLAP) FAIL("overlap accepted");
    if (kv_relayout_desc_bytes(NULL, &r, &w) != KVR_ERR_INVALID_ARG) FAIL("NULL accepted");
    if (strcmp(kv_relayout_strerror((kvr_status)12345), "unknown status") != 0)
        FAIL("strerror of an unknown status");
    describe(&d, src, dst);
    if (kv_relayout_staging_bytes(&d, ES, &r) != KVR_OK ||
        r != (int64_t)(300 + 77) * L * C * H * D * ES)
        FAIL("staging bytes %lld", (long long)r);
    if (kv_relayout_staging_bytes(&d, 3, &r) != KVR_ERR_INVALID_ARG) FAIL("3-byte staging");
    printf("abi_client host: ok\n");
    return 0;
}

/* one run of the given launch mode into fresh decode pools; compares with the oracle */
static int gpu_run(int mode, uint8_t *const *h_src, uint8_t *const *h_ref, void *const *d_src) {
    void *d_dst[TP_D];
    uint8_t *got;
    kvr_desc d;
    kvr_plan *plan = NULL;
    kvr_status st = KVR_OK;
    int s, l;
    got = (uint8_t *)malloc((size_t)dst_pool_bytes);
    if (got == NULL) FAIL("host allocation");
    for (s = 0; s < TP_D; ++s) {
        if (cudaMalloc(&d_dst[s], (size_t)dst_pool_bytes) != 0) FAIL("cudaMalloc");
        memset(got, 0xEE, (size_t)dst_pool_bytes);
        cudaMemcpy(d_dst[s], got, (size_t)dst_pool_bytes, H2D);
    }
    (void)h_src;
    describe(&d, d_src, d_dst);
    st = kv_relayout_plan(&d, &plan);
    if (st != KVR_OK) FAIL("plan: %s", kv_relayout_strerror(st));
    if (mode == 0) {
        st = kv_relayout_all(plan, NULL);
    } else if (mode == 1) {
        for (l = 0; l < L && st == KVR_OK; ++l) st = kv_relayout_layer(plan, l, NULL);
    } else {
        st = kv_relayout_layers(plan, 0, 2, NULL);
        if (st == KVR_OK) st = kv_relayout_layers_ex(plan, 2, 1, KVR_LAUNCH_NO_WAIT, NULL);
    }
    if (st != KVR_OK) FAIL("launch (mode %d): %s", mode, kv_relayout_strerror(st));
    if (cudaDeviceSynchronize() != 0) FAIL("synchronize");
    kv_relayout_plan_destroy(plan);
    for (s = 0; s < TP_D; ++s) {
        cudaMemcpy(got, d_dst[s], (size_t)dst_pool_bytes, D2H);
        if (memcmp(got, h_ref[s], (size_t)dst_pool_bytes) != 0)
            FAIL("mode %d: decode shard %d differs from the oracle", mode, s);
        cudaFree(d_dst[s]);
    }
    free(got);
    return 0;
}

/* pack into a staging buffer [L][C][sum n][H][D], then unpack it into fresh decode
 * pools layer by layer: the staging bytes against the oracle's gather into that
 * buffer, the decode bytes against the oracle's direct relayout */
#define TOTAL (300 + 0 + 77)
static int gpu_staging(uint8_t *const *h_src, uint8_t *const *h_ref, void *const *d_src) {
    const int64_t row = (int64_t)D * ES, tok = row * H, plane = tok * TOTAL;
    const int64_t stage_bytes = plane * L * C;
    const int64_t hs = (H / TP_S) * row, sblk = BP * hs;          /* standard prefill strides */
    int64_t stage_off[R + 1], got_bytes = -1;
    int32_t stage_ids[TOTAL];
    uint64_t sbase[TP_S * L * C], dbase[L * C];
    uint8_t *want, *got;
    void *d_stage, *d_dst[TP_D];
    kvr_desc d;
    kvr_plan *plan = NULL;
    kvr_status st = KVR_OK;
    const float one = 1.0f;
    int r, s, v, l;
    stage_off[0] = 0;
    for (r = 0; r < R; ++r) stage_off[r + 1] = stage_off[r] + lens[r];
    for (v = 0; v < TOTAL; ++v) stage_ids[v] = v;
    want = (uint8_t *)calloc((size_t)stage_bytes, 1);
    got = (uint8_t *)malloc((size_t)(stage_bytes > dst_pool_bytes ? stage_bytes : dst_pool_bytes));
    if (want == NULL || got == NULL) FAIL("host allocation");
    for (s = 0; s < TP_S; ++s)
        for (v = 0; v < L * C; ++v)
            sbase[s * L * C + v] = (uint64_t)(uintptr_t)(h_src[s] + (int64_t)v * NP * sblk);
    for (v = 0; v < L * C; ++v) dbase[v] = (uint64_t)(uintptr_t)(want + (int64_t)v * plane);
    if (kvo_relayout_general(0, L, L, C, H, D, 0, 0, ES, 0, &one, TP_S, 1, BP, 1, sbase, sblk,
                             hs, row, dbase, tok, tok, row, R, lens, src_off, src_bt,
                             stage_off, stage_ids) != 0)
        FAIL("oracle (staging)");
    describe(&d, d_src, NULL);
    if (kv_relayout_staging_bytes(&d, ES, &got_bytes) != KVR_OK || got_bytes != stage_bytes)
        FAIL("staging bytes %lld", (long long)got_bytes);
    if (cudaMalloc(&d_stage, (size_t)stage_bytes) != 0) FAIL("cudaMalloc");
    cudaMemset(d_stage, 0, (size_t)stage_bytes);
    st = kv_relayout_plan_pack(&d, d_stage, NULL, &plan);
    if (st != KVR_OK) FAIL("plan_pack: %s", kv_relayout_strerror(st));
    st = kv_relayout_all(plan, NULL);
    if (st != KVR_OK) FAIL("pack launch: %s", kv_relayout_strerror(st));
    if (cudaDeviceSynchronize() != 0) FAIL("synchronize");
    kv_relayout_plan_destroy(plan);
    cudaMemcpy(got, d_stage, (size_t)stage_bytes, D2H);
    if (memcmp(got, want, (size_t)stage_bytes) != 0) FAIL("packed staging differs from the oracle");
    for (s = 0; s < TP_D; ++s) {
        if (cudaMalloc(&d_dst[s], (size_t)dst_pool_bytes) != 0) FAIL("cudaMalloc");
        cudaMemset(d_dst[s], 0xEE, (size_t)dst_pool_bytes);
    }
    describe(&d, NULL, d_dst);
    st = kv_relayout_plan_unpack(&d, d_stage, NULL, &plan);
    if (st != KVR_OK) FAIL("plan_unpack: %s", kv_relayout_strerror(st));
    for (l = 0; l < L && st == KVR_OK; ++l) st = kv_relayout_layer(plan, l, NULL);
    if (st != KVR_OK) FAIL("unpack launch: %s", kv_relayout_strerror(st));
    if (cudaDeviceSynchronize() != 0) FAIL("synchronize");
    kv_relayout_plan_destroy(plan);
    for (s = 0; s < TP_D; ++s) {
        cudaMemcpy(got, d_dst[s], (size_t)dst_pool_bytes, D2H);
        if (memcmp(got, h_ref[s], (size_t)dst_pool_bytes) != 0)
            FAIL("unpacked decode shard %d differs from the oracle", s);
        cudaFree(d_dst[s]);
    }
    cudaFree(d_stage);
    free(want);
    free(got);
    return 0;
}

static int gpu_mode(void) {
    uint8_t *h_src[TP_S], *h_ref[TP_D];
    void *d_src[TP_S];
    uint32_t seed = 12345u;
    int s, mode;
    int64_t i;
    for (s = 0; s < TP_S; ++s) {
        h_src[s] = (uint8_t *)malloc((size_t)src_pool_bytes);
        if (h_src[s] == NULL) FAIL("host allocation");
        for (i = 0; i < src_pool_bytes; ++i) h_src[s][i] = (uint8_t)lcg(&seed);
        if (cudaMalloc(&d_src[s], (size_t)src_pool_bytes) != 0) FAIL("cudaMalloc");
        cudaMemcpy(d_src[s], h_src[s], (size_t)src_pool_bytes, H2D);
    }
    for (s = 0; s < TP_D; ++s) {
        h_ref[s] = (uint8_t *)malloc((size_t)dst_pool_bytes);
        if (h_ref[s] == NULL) FAIL("host allocation");
        memset(h_ref[s], 0xEE, (size_t)dst_pool_bytes);
    }
    if (kvo_relayout(0, L, L, C, H, D, ES, TP_S, TP_D, BP, BD, NP, ND,
                     (const uint8_t *const *)h_src, h_ref, R, lens, src_off, src_bt, dst_off,
                     dst_bt) != 0)
        FAIL("oracle");
    for (mode = 0; mode < 3; ++mode)
        if (gpu_run(mode, h_src, h_ref, d_src) != 0) return 1;
    if (gpu_staging(h_src, h_ref, d_src) != 0) return 1;
    for (s = 0; s < TP_S; ++s) {
        cudaFree(d_src[s]);
        free(h_src[s]);
    }
    for (s = 0; s < TP_D; ++s) free(h_ref[s]);
    printf("abi_client gpu: ok (whole-prompt, per-layer, layer ranges, pack, unpack)\n");
    return 0;
}

int main(int argc, char **argv) {
    tables();
    if (argc > 1 && strcmp(argv[1], "gpu") == 0) return gpu_mode();
    return host_mode();
}
