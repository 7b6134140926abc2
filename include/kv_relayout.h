/*
 * kv_relayout.h -- C ABI of the prefill -> decode KV-cache relayout on one GPU.
 *
 * What it computes. Page "PD 分离与 KV 传输" (ai-infra-handbooks,
 * serving/distributed/pd-disagg):
 *   - section "实现" (pd.py prefill()/admit()): the prefill instance's K/V of
 *     a prompt is gathered through the prefill block table (block size Bp) and
 *     written through the decode block table (block size Bd): token p goes to
 *     decode slot block_ids[p / Bd] * Bd + p % Bd, for p < n only;
 *   - section "布局转换": when the TP degrees differ, a KV head moves from the
 *     prefill card that holds it to the decode card that holds it (a split
 *     for Tp < Td, a merge for Tp > Td);
 *   - section "流程" and the "KV-Cache 传输:方案与时延" section of
 *     "推理 INFRA 方法论（6）": the decode side allocates its blocks first and
 *     the prefill side writes straight into them, whole prompt or layer by
 *     layer as layers finish.
 * All shard pools live in the HBM of the current GPU; there is no second
 * device, collective or network. Elements are moved as raw bits (no dtype
 * conversion; NaN payloads and -0 are preserved).
 *
 * Pool memory. A pool may live in this GPU's HBM, in managed memory, or in
 * pinned host memory mapped into the device address space (cudaHostAlloc,
 * cudaHostRegister): on Grace-based GB300 systems the kernel then reads or
 * writes host memory directly over NVLink-C2C, with no staging copy. Launch
 * calls that build a plan check that the first and last byte of every pool is
 * such memory (KVR_ERR_POOL_ADDRESS otherwise).
 *
 * Pool layout. Each TP shard of each side is ONE contiguous buffer of
 *   [num_layers][num_components][num_blocks][block_size][H_local][head_dim]
 * elements of elem_bytes bytes. Components: 2 = K then V planes, 1 = a single
 * latent plane (MLA). A TP degree tp that divides H: H_local = H / tp and
 * shard s holds the contiguous head range [s * H / tp, (s + 1) * H / tp).
 * A TP degree that is a multiple of H (more cards than KV heads, as when GQA
 * heads or an MLA latent are replicated across TP ranks): H_local = 1 and
 * head h is held whole by the tp / H consecutive shards h * tp / H ..
 * (h + 1) * tp / H - 1. The relayout reads such a head from the first prefill
 * shard that holds it and writes it to every decode shard that holds it
 * (every copy counts in the bytes written). Any other tp is refused.
 *
 * Block tables. CSR over requests: request r owns table entries
 * bt[off[r]] .. bt[off[r + 1] - 1]; entry k is the physical block holding the
 * request's tokens [k * B, (k + 1) * B). Only the first ceil(n_r / B) entries
 * of each request are used (a decode table may reserve more, e.g. for the
 * first generated token; those are never touched). One table per side, shared
 * by all shard pools of that side. Prefill block ids may repeat (a shared
 * prefix); used decode block ids may not.
 *
 * Ownership. The caller owns the pools, the streams and all host arrays; host
 * arrays may be freed as soon as kv_relayout_plan() returns. The library
 * owns a plan and its small device metadata buffer (work list and prefill
 * block ids), freed by kv_relayout_plan_destroy(). The library never
 * allocates, frees or chooses pool blocks.
 *
 * Errors. Every call returns a status; no C++ exception crosses this ABI.
 * Launch calls are asynchronous, never synchronize, and report only launch
 * errors (KVR_ERR_CUDA). A plan is immutable: launches of one plan from
 * several threads are safe, but launches that overlap in time on different
 * streams must not write the same decode blocks (the caller orders them).
 */
#ifndef KV_RELAYOUT_H_
#define KV_RELAYOUT_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Largest TP degree (number of shard pools) on either side. */
#define KVR_MAX_TP 16

typedef enum kvr_status {
    KVR_OK = 0,
    KVR_ERR_INVALID_ARG = -1,   /* NULL pointer, non-positive size, bad offsets, negative length */
    KVR_ERR_UNSUPPORTED = -2,   /* elem_bytes not 1/2/4, tp neither divides nor is a multiple
                                   of H, tp > KVR_MAX_TP, too large */
    KVR_ERR_ALIGNMENT = -3,     /* a pool not 16-byte aligned, or head_dim * elem_bytes % 16 != 0 */
    KVR_ERR_BLOCK_RANGE = -4,   /* a used block id outside [0, num_blocks) */
    KVR_ERR_TABLE_SHORT = -5,   /* a request has fewer than ceil(n / B) table entries */
    KVR_ERR_DST_ALIAS = -6,     /* a decode block id used twice */
    KVR_ERR_LAYER_RANGE = -7,   /* layer outside [0, num_layers) */
    KVR_ERR_CUDA = -8,          /* a CUDA runtime call failed (no device, launch error, ...) */
    KVR_ERR_NOMEM = -9,         /* host or device allocation of the plan failed */
    KVR_ERR_POOL_OVERLAP = -10, /* a decode pool overlaps another decode pool or a prefill pool */
    KVR_ERR_SCRATCH_LIMIT = -11, /* kv_relayout_all_prealloc: work list larger than its scratch */
    KVR_ERR_POOL_ADDRESS = -12, /* a pool's first or last byte is not memory this GPU can access */
    KVR_ERR_DEVICE_BOUNDS = -13 /* checked builds: a launch computed a row outside its pools */
} kvr_status;

typedef struct kvr_desc {
    int32_t num_layers;        /* L >= 1 */
    int32_t num_components;    /* C: 2 (K, V) or 1 (MLA latent) */
    int32_t kv_heads;          /* H >= 1: global KV heads (1 for an MLA latent) */
    int32_t head_dim;          /* D >= 1: elements per head row */
    int32_t elem_bytes;        /* es: 1, 2 or 4 */
    int32_t src_tp;            /* Tp: prefill shard pools, 1..KVR_MAX_TP, divides H or a multiple of it */
    int32_t dst_tp;            /* Td: decode shard pools, 1..KVR_MAX_TP, divides H or a multiple of it */
    int32_t src_block_size;    /* Bp >= 1 tokens per prefill block */
    int32_t dst_block_size;    /* Bd >= 1 tokens per decode block */
    int64_t src_num_blocks;    /* Np >= 1 blocks in each prefill shard pool */
    int64_t dst_num_blocks;    /* Nd >= 1 blocks in each decode shard pool */
    const void *const *src_pools;   /* host array [Tp] of device pointers, 16-B aligned */
    void *const *dst_pools;         /* host array [Td] of device pointers, 16-B aligned */
    int32_t num_requests;           /* R >= 0 */
    const int32_t *seq_lens;        /* host [R], n_r >= 0 (0 = nothing to move) */
    const int64_t *src_bt_offsets;  /* host [R + 1], non-decreasing, >= 0 */
    const int32_t *src_bt;          /* host, prefill block ids */
    const int64_t *dst_bt_offsets;  /* host [R + 1], non-decreasing, >= 0 */
    const int32_t *dst_bt;          /* host, decode block ids */
} kvr_desc;

typedef struct kvr_plan kvr_plan;

/*
 * Element types for a relayout that changes the KV dtype on the way (page
 * "PD 分离与 KV 传输", section "布局转换": one side keeps BF16 KV, the other
 * FP8 KV, and the conversion is best done on the GPU around the transfer).
 * FP8 is E4M3 of the OCP 8-bit floating point format (bias 7, subnormals, no
 * infinities, S.1111.111 = NaN, largest finite 448). With scale s:
 *   BF16 -> E4M3:  q = E4M3(x * fl32(1 / s)), nearest with ties to even; values
 *                  beyond +-448 and infinities saturate to +-448; a NaN x gives
 *                  S.1111.111 with the sign of x;
 *   E4M3 -> BF16:  y = BF16(float(q) * s), nearest with ties to even; a NaN
 *                  code gives sign | 0x7FC0 with the sign of the code.
 * Products are single fp32 multiplications; 1/s is rounded to fp32 once.
 */
typedef enum kvr_dtype {
    KVR_DTYPE_BF16 = 1,
    KVR_DTYPE_FP8_E4M3 = 2
} kvr_dtype;

typedef struct kvr_convert {
    int32_t src_dtype;     /* kvr_dtype of the prefill pools; desc->elem_bytes is its size */
    int32_t dst_dtype;     /* kvr_dtype of the decode pools: the other of the two */
    int32_t per_head;      /* 0: one scale per (layer, component); 1: per (layer, component, head) */
    const float *scales;   /* host [L][C] or [L][C][H]: positive, finite; copied by the plan */
} kvr_convert;

/*
 * Validate *desc on the host and compute the bytes one full relayout reads
 * and writes (each = sum_r n_r * L * C * H * D * es, the page's "KV per token
 * times prompt length", section "传输的代价"; writes times Td / H when the
 * decode side replicates heads). Makes no CUDA call and
 * dereferences no device pointer. Either output pointer may be NULL.
 */
kvr_status kv_relayout_desc_bytes(const kvr_desc *desc, int64_t *bytes_read,
                                  int64_t *bytes_written);

/*
 * Validate *desc (as above), check that every pool is memory the current
 * device can access, build the work list on the host and upload it with the
 * used block ids to the current device (one allocation, synchronous copies).
 * *out is set to the new plan, or to NULL on failure.
 */
kvr_status kv_relayout_plan(const kvr_desc *desc, kvr_plan **out);

/*
 * A physical layout of one side (page "PD 分离与 KV 传输", section "布局转换":
 * attention backends differ in whether K and V are stored together and in
 * the order of the head and token dimensions). Per (TP shard s, layer l,
 * component c) the side is a strided view [block][token][local head][dim]:
 * element [b][t][h][e] of that view is at
 *   bases[(s * L + l) * C + c] + b * block_stride + t * token_stride
 *                              + h * head_stride + e * element size,
 * i.e. head rows (dim) are contiguous and the three strides are shared by all
 * views of the side (H_local local heads, as above). Examples: the standard
 * layout [L][C][N][B][H_local][D]; one K and one V tensor per layer; K and V
 * interleaved per block
 * ([N][C][B][H][D]); head-major blocks ([N][H][B][D]); a contiguous
 * [tokens][heads][dim] staging buffer seen as blocks of one token.
 * Requirements: every base 16-byte aligned and non-NULL; strides >= 0 and
 * multiples of 16 (a stride whose dimension has extent 1 is ignored).
 * Performance (not a requirement): when every base and stride of both sides is
 * a multiple of 32 bytes and the row moves an even number of 16-byte units (16
 * elements each when converting), the kernel moves 32 bytes per access, which
 * is the faster path; pools from the CUDA
 * allocator (256-byte aligned) in the standard layout take it whenever the row
 * allows. On the
 * decode side the views must not alias: sorted by stride, each dimension
 * (of extent > 1) must step over the whole extent of the smaller ones, the
 * smallest over one head row; no two decode views may share a byte (views
 * may interleave, as K and V blocks do) and no decode view's span may meet a
 * prefill view's span (else KVR_ERR_POOL_OVERLAP).
 */
typedef struct kvr_layout {
    const void *const *bases;   /* host [tp * num_layers * num_components] device addresses */
    int64_t block_stride;       /* bytes between consecutive blocks */
    int64_t token_stride;       /* bytes between consecutive token slots of a block */
    int64_t head_stride;        /* bytes between consecutive local heads of a token */
} kvr_layout;

/*
 * As kv_relayout_desc_bytes() / kv_relayout_plan(), for a relayout that also
 * converts the element type (kvr_convert above; cv == NULL is a plain bit
 * copy). Decode pools then hold dst_dtype elements: their layout is the same
 * with dst_dtype's element size, and head_dim times each side's element size
 * must be a multiple of 16 bytes (KVR_ERR_ALIGNMENT). Bytes read and written
 * differ (e.g. 2 and 1 per element for BF16 -> E4M3). The plan's launches are
 * kv_relayout_layer() / kv_relayout_all() as for any plan.
 * Errors: KVR_ERR_UNSUPPORTED for a dtype pair other than BF16 <-> E4M3;
 * KVR_ERR_INVALID_ARG if desc->elem_bytes is not src_dtype's size, per_head
 * is not 0/1, or a scale is missing, not finite or not positive.
 */
kvr_status kv_relayout_desc_convert_bytes(const kvr_desc *desc, const kvr_convert *cv,
                                          int64_t *bytes_read, int64_t *bytes_written);
kvr_status kv_relayout_plan_convert(const kvr_desc *desc, const kvr_convert *cv,
                                    kvr_plan **out);

/*
 * The general form: any layout on either side (kvr_layout above) and an
 * optional conversion. src_layout / dst_layout NULL: that side is
 * desc->src_pools / desc->dst_pools in the standard layout; non-NULL: the
 * layout replaces the pools (desc->src_pools / dst_pools are then ignored and
 * may be NULL; num_blocks still bounds the block ids). cv NULL: bit copy.
 * kv_relayout_desc_bytes_ex() validates on the host only (no CUDA call).
 */
kvr_status kv_relayout_desc_bytes_ex(const kvr_desc *desc, const kvr_layout *src_layout,
                                     const kvr_layout *dst_layout, const kvr_convert *cv,
                                     int64_t *bytes_read, int64_t *bytes_written);
kvr_status kv_relayout_plan_ex(const kvr_desc *desc, const kvr_layout *src_layout,
                               const kvr_layout *dst_layout, const kvr_convert *cv,
                               kvr_plan **out);

/*
 * The two halves of the hand-off through a contiguous staging buffer (page
 * "PD 分离与 KV 传输", section "实现": pd.py's prefill() gathers each layer's K
 * and V of a prompt into a contiguous [seq, kv_heads, head_dim] array, and
 * admit() writes that array through the decode block table; the page
 * "推理 INFRA 方法论（6）", section "KV-Cache 传输:方案与时延", stages the KV
 * this way when the two sides' TP degrees differ and a link sits between them).
 *
 * The staging buffer is ONE contiguous buffer of
 *   [num_layers][num_components][sum of n_r][kv_heads][head_dim]
 * elements: every global head side by side (the prefill shards' head ranges
 * merged, a replicated head once), request r's tokens at rows
 * sum(n[:r]) .. sum(n[:r + 1]) - 1. It must be 16-byte aligned, memory the
 * current device can access, and hold kv_relayout_staging_bytes() bytes.
 *
 * kv_relayout_plan_pack(): a plan that gathers the prefill pools of *desc into
 * `staging` (the desc's decode-side fields dst_tp, dst_block_size,
 * dst_num_blocks, dst_pools, dst_bt_offsets and dst_bt are ignored). With a
 * conversion `cv`, the staging buffer holds cv->dst_dtype elements.
 * kv_relayout_plan_unpack(): a plan that writes `staging` into the decode
 * pools of *desc (its prefill-side fields src_tp, src_block_size,
 * src_num_blocks, src_pools, src_bt_offsets and src_bt are ignored); the
 * staging buffer holds desc->elem_bytes elements (cv->src_dtype with a
 * conversion). Either plan is launched with kv_relayout_all() /
 * kv_relayout_layer() / kv_relayout_layers() like any plan; packing and then
 * unpacking gives the same decode bytes as one kv_relayout_plan() relayout.
 * Errors: those of kv_relayout_plan_ex() (the staging buffer is one side's
 * view: KVR_ERR_POOL_OVERLAP if it meets the other side's pools), and
 * KVR_ERR_INVALID_ARG for a NULL staging buffer or a batch of zero tokens.
 *
 * kv_relayout_staging_bytes(): the staging buffer's size for elements of
 * `elem_bytes` bytes (1, 2 or 4): L * C * (sum of n_r) * H * D * elem_bytes.
 * Host only (no CUDA call); reads num_layers, num_components, kv_heads,
 * head_dim, num_requests and seq_lens of *desc.
 */
kvr_status kv_relayout_staging_bytes(const kvr_desc *desc, int32_t elem_bytes, int64_t *bytes);
kvr_status kv_relayout_plan_pack(const kvr_desc *desc, void *staging, const kvr_convert *cv,
                                 kvr_plan **out);
kvr_status kv_relayout_plan_unpack(const kvr_desc *desc, const void *staging,
                                   const kvr_convert *cv, kvr_plan **out);

/*
 * Move layer `layer` of every request: one kernel launch on `stream`
 * (a cudaStream_t; NULL = the legacy default stream). Asynchronous. Calling
 * it for every layer gives the same bytes as kv_relayout_all(). The current
 * device must be the plan's device.
 */
kvr_status kv_relayout_layer(const kvr_plan *plan, int32_t layer, void *stream);

/* Move all layers of every request: one kernel launch on `stream`. */
kvr_status kv_relayout_all(const kvr_plan *plan, void *stream);

/*
 * Move layers [first, first + count) of every request: one kernel launch on
 * `stream`. Asynchronous. For an engine that computes prefill a group of
 * layers at a time (page "PD multiplexing: splitting prefill and decode by SM
 * on one GPU", section "SGLang's PD multiplexing": a round computes
 * split_forward_token_budget // prompt tokens layers) and hands each group
 * over as it finishes. count == 1 is kv_relayout_layer(); first == 0 with
 * count == L is kv_relayout_all(); any split of [0, L) into ranges gives the
 * same bytes as kv_relayout_all(). KVR_ERR_LAYER_RANGE unless
 * 0 <= first, 1 <= count and first + count <= L.
 */
kvr_status kv_relayout_layers(const kvr_plan *plan, int32_t first, int32_t count,
                              void *stream);

/* Launch flags of kv_relayout_layers_ex(). */
#define KVR_LAUNCH_NO_WAIT 1u

/*
 * kv_relayout_layers() with launch flags (0: identical to it; unknown bits:
 * KVR_ERR_INVALID_ARG).
 *
 * Every launch is ordered after the kernel launched before it on `stream`:
 * the kernel may start early (programmatic dependent launch) and build its
 * work tables, but it waits for that kernel to finish before it loads from
 * or stores to a pool, which is what orders a hand-off after the kernel that
 * wrote its prefill rows. (A per-layer launch may ask L2 to prefetch its
 * prefill rows before that wait; the prefetch is only a cache hint, and the
 * loads after the wait see everything the previous kernel wrote.) KVR_LAUNCH_NO_WAIT moves that wait to the end of the launch,
 * after its copies: the launch reads and writes the pools while the kernel
 * before it may still run, and still completes only after that kernel (work
 * queued after it on the stream sees both), so back-to-back hand-off
 * launches stream into each other instead of draining between launches (on
 * the 70B workload, 80 single-layer launches: 5.3 -> 6.7 TB/s).
 * Pass it only when the work just before this launch on `stream` is another
 * hand-off launch (of this plan, or of a plan whose decode views do not meet
 * this one's), and every prefill row this launch reads and every decode block
 * it writes was last written by work queued on `stream` before the latest
 * hand-off launch made without the flag (such a launch lets later launches
 * start only after it has waited for everything before it). For example: the
 * layers that are already computed, handed over one launch each, the first
 * without the flag. A launch right after any other kernel or copy must not
 * pass it.
 */
kvr_status kv_relayout_layers_ex(const kvr_plan *plan, int32_t first, int32_t count,
                                 uint32_t flags, void *stream);

/* Bytes one kv_relayout_all() reads and writes (per layer: divide by L). */
kvr_status kv_relayout_plan_bytes(const kvr_plan *plan, int64_t *bytes_read,
                                  int64_t *bytes_written);

/*
 * The launch shape the plan chose: CTAs of one kv_relayout_all() launch
 * (`grid_all`), of one kv_relayout_layer() launch (`grid_layer`), and the
 * decode-side tokens one work item covers (`tile_tokens`). Any output pointer
 * may be NULL. Per-layer grids are sized from the kernel's occupancy on the
 * plan's device: a layer whose tiles fit in one wave of resident CTAs is
 * split to fill that wave, a larger one to about three waves.
 */
kvr_status kv_relayout_plan_launch_shape(const kvr_plan *plan, int64_t *grid_all,
                                         int64_t *grid_layer, int32_t *tile_tokens);

/* Free the plan and its device buffer (NULL is a no-op). Synchronizes the
 * device buffer's release like cudaFree: call it after the launches that use
 * the plan have been ordered before any reuse of that memory. */
void kv_relayout_plan_destroy(kvr_plan *plan);

/* Static, human-readable name of a status. */
const char *kv_relayout_strerror(kvr_status status);

/*
 * A stream whose kernels run on at most about `sm_count` SMs of the current
 * device (a CUDA green context). Page "PD multiplexing: splitting prefill and
 * decode by SM on one GPU", section "Green contexts: carving out SMs for a
 * stream": memory-bound work reaches the bandwidth limit on a share of the
 * SMs, leaving the rest to compute; launching the relayout on such a stream
 * hands the KV over beside the model's kernels. The count is rounded up to
 * the device's split granularity (8 SMs on this GPU generation);
 * *sms_granted receives the SMs the stream got. The stream is a cudaStream_t
 * for kv_relayout_layer() / kv_relayout_all() and any other launch; it shares
 * memory with the rest of the process. Relayout launches on such a stream
 * shape their grids for its SMs (they ask the driver which green context the
 * stream belongs to at each launch). Errors: KVR_ERR_INVALID_ARG for a
 * count outside [1, SMs], KVR_ERR_UNSUPPORTED when the driver has no green
 * contexts or cannot split, KVR_ERR_CUDA for other driver failures.
 * Destroy it (after its work is done) with kv_relayout_sm_stream_destroy().
 */
typedef struct kvr_sm_stream kvr_sm_stream;
kvr_status kv_relayout_sm_stream_create(int32_t sm_count, kvr_sm_stream **out, void **stream,
                                        int32_t *sms_granted);
void kv_relayout_sm_stream_destroy(kvr_sm_stream *s);

/* Size of the device scratch array kv_relayout_all_prealloc() works in. */
#define KVR_PREALLOC_SCRATCH_BYTES (1u << 20)

/*
 * kv_relayout_all(), for callers that cannot allocate device memory.
 *
 * The pages have no counterpart of this call; it exists for integration.
 * Some callers cannot call cudaMalloc when they hand KV over: a serving
 * engine that has carved (nearly) all of HBM into its KV block pools up front
 * has no room left for a new allocation, and a latency-critical loop cannot
 * afford cudaMalloc/cudaFree, which may synchronize the whole device and so
 * stall the other streams. kv_relayout_plan() allocates a small device buffer
 * for the work list; this call allocates nothing: it validates *desc exactly
 * like kv_relayout_plan(), copies the work list (16 bytes per token tile of
 * a request, 8 bytes per (shard, layer, component) view of each side, 4 bytes
 * per used prefill and decode block id) with one cudaMemcpyAsync into a
 * fixed device array of KVR_PREALLOC_SCRATCH_BYTES (1 MiB) that the library
 * reserves on every GPU that loads it, until the process exits, and launches
 * the same kernel as kv_relayout_all() on `stream`, with the grid shaped for
 * the stream's green context as kv_relayout_all() does. The pool memory
 * checks of kv_relayout_plan() apply.
 *
 *  - A work list larger than the array is rejected with
 *    KVR_ERR_SCRATCH_LIMIT before anything is copied or launched; use
 *    kv_relayout_plan() for such batches.
 *  - The first call on a device looks up the array's device address on that
 *    device (with the device current) and caches it; make that first call
 *    before any stream capture begins.
 *  - The work list is copied from pageable host memory that the call frees
 *    before it returns: the call returns once the CUDA runtime has taken the
 *    copy, which may wait for work already queued on `stream`. While `stream`
 *    is being captured, the call returns KVR_ERR_UNSUPPORTED and enqueues
 *    nothing.
 *  - Every call on a device shares the one array. Calls from several host
 *    threads enqueue their copy and their kernel under one lock per device,
 *    so calls on one stream run one after another. Calls whose copies and
 *    kernels overlap on the GPU (different streams not ordered by the caller)
 *    race on the array and may move the wrong rows: issue them on one stream
 *    or order them with events.
 *  - The host arrays of *desc may be freed when the call returns.
 */
kvr_status kv_relayout_all_prealloc(const kvr_desc *desc, void *stream);

/*
 * Device-side address checks (test builds). The library can be compiled with
 * KVR_DEVICE_CHECKS defined (prefill_decode_paged_gb300.build.build_checked()):
 * its kernels then check, for every row of every launch of a plan made by
 * kv_relayout_plan*(), that the row's prefill bytes lie inside the prefill
 * pools (views) and its decode bytes inside the decode pools, as the plan
 * validated them; a row that does not is counted in an error word and not
 * read, prefetched or written. The checks catch a disagreement between the
 * plan's validation and the kernel's address arithmetic on the GPU itself,
 * without ever touching memory outside the pools. Product builds skip them.
 *
 * kv_relayout_debug_status(): waits for the device (cudaDeviceSynchronize),
 * reads and clears the plan's error word into *flags (may be NULL); returns
 * KVR_ERR_DEVICE_BOUNDS if a row was dropped since the last call, KVR_OK if
 * not, KVR_ERR_UNSUPPORTED in a product build.
 * kv_relayout_debug_narrow(): makes the checks treat the last `bytes` bytes of
 * every pool region as outside it (to test that the checks fire; those rows
 * are then dropped, the others still move); KVR_ERR_UNSUPPORTED in a product
 * build. kv_relayout_all_prealloc() launches are not checked.
 */
kvr_status kv_relayout_debug_status(const kvr_plan *plan, uint32_t *flags);
kvr_status kv_relayout_debug_narrow(kvr_plan *plan, int64_t bytes);

#ifdef __cplusplus
}
#endif

#endif /* KV_RELAYOUT_H_ */
