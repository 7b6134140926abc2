/*
 * kv_oracle.c -- plain, slow, obviously correct CPU definition of the
 * prefill -> decode KV-cache relayout.
 *
 * TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and the CPU
 * baseline / reference legs of bench.py may build, load or call this file.
 * The CUDA library never links, includes or calls it, and this file shares
 * no header, helper or constant with the CUDA library.
 *
 * What it follows (page "PD 分离与 KV 传输", ai-infra-handbooks,
 * serving/distributed/pd-disagg):
 *   - section "实现", pd.py prefill(): the prefill instance gathers every
 *     layer's K/V of the prompt, token by token, through its own block table,
 *     into a [seq, kv_heads, head_dim] array;
 *   - section "实现", pd.py admit(): the decode instance writes token p of
 *     the prompt to slot  block_ids[p // block_size] * block_size
 *     + p % block_size  of its own pool, for p < n only (so the slots of a
 *     partial last block past the prompt are never touched);
 *   - section "布局转换", item "TP 不同": the prefill side holds 1/Tp of the
 *     KV heads per card and the decode side 1/Td; a head moves from one
 *     card's shard to another's;
 *   - section "传输的代价": KV per token times prompt length is the amount
 *     of data moved.
 *
 * Readings taken where the page is silent (each is listed in the design doc):
 *   - pool layout, one buffer per TP shard: [L][C][N][B][H_local][D] of
 *     es-byte elements (C = 2 for K and V, C = 1 for an MLA latent);
 *   - TP shard s holds the contiguous head range [s*H/T, (s+1)*H/T);
 *   - one block table per side, shared by all shards of that side;
 *   - elements are copied as es raw bytes: no conversion, NaN payloads kept.
 *
 * Every function here is a plain loop nest; there is no blocking, fusion or
 * reordering beyond the definition.
 */
#include <stdint.h>
#include <stddef.h>

/* Bytes of KV cache one token occupies, summed over layers, components,
 * heads and head dimension ("KV/token", section "传输的代价"). */
int64_t kvo_bytes_per_token(int32_t num_layers, int32_t num_components,
                            int32_t kv_heads, int32_t head_dim,
                            int32_t elem_bytes)
{
    return (int64_t)num_layers * num_components * kv_heads * head_dim * elem_bytes;
}

/* Bytes one hand-off moves for a batch of prompts: KV/token times the
 * prompt lengths (section "传输的代价"; pd.py's own counter sums the
 * gathered K and V of every layer). */
int64_t kvo_transfer_bytes(int32_t num_layers, int32_t num_components,
                           int32_t kv_heads, int32_t head_dim,
                           int32_t elem_bytes, int32_t num_requests,
                           const int32_t *seq_lens)
{
    int64_t tokens = 0;
    for (int32_t r = 0; r < num_requests; ++r)
        tokens += seq_lens[r];
    return tokens * kvo_bytes_per_token(num_layers, num_components, kv_heads,
                                        head_dim, elem_bytes);
}

/*
 * The relayout itself, for layers [layer_begin, layer_end).
 *
 * src_pools[sp] is the prefill shard sp (of src_tp), layout
 *   [num_layers][num_components][src_num_blocks][src_block][H/src_tp][head_dim];
 * dst_pools[dp] is the decode shard dp (of dst_tp), layout
 *   [num_layers][num_components][dst_num_blocks][dst_block][H/dst_tp][head_dim].
 * Request r owns src_bt[src_off[r] ...] and dst_bt[dst_off[r] ...]; entry k
 * of a table is the physical block that holds tokens [k*B, (k+1)*B).
 *
 * Returns 0, or -1 when the head count is not divisible by a TP degree.
 */
int kvo_relayout(int32_t layer_begin, int32_t layer_end,
                 int32_t num_layers, int32_t num_components,
                 int32_t kv_heads, int32_t head_dim, int32_t elem_bytes,
                 int32_t src_tp, int32_t dst_tp,
                 int32_t src_block, int32_t dst_block,
                 int64_t src_num_blocks, int64_t dst_num_blocks,
                 const uint8_t *const *src_pools, uint8_t *const *dst_pools,
                 int32_t num_requests, const int32_t *seq_lens,
                 const int64_t *src_off, const int32_t *src_bt,
                 const int64_t *dst_off, const int32_t *dst_bt)
{
    if (kv_heads % src_tp != 0 || kv_heads % dst_tp != 0)
        return -1;
    (void)num_layers;
    const int64_t src_heads = kv_heads / src_tp; /* heads per prefill card */
    const int64_t dst_heads = kv_heads / dst_tp; /* heads per decode card */
    const int64_t C = num_components;
    const int64_t D = head_dim;

    for (int32_t r = 0; r < num_requests; ++r) {
        const int64_t n = seq_lens[r];
        for (int64_t l = layer_begin; l < layer_end; ++l) {
            for (int64_t c = 0; c < C; ++c) {
                for (int64_t t = 0; t < n; ++t) {
                    /* prefill side: block table entry t / Bp, offset t % Bp */
                    const int64_t sblk = src_bt[src_off[r] + t / src_block];
                    const int64_t soff = t % src_block;
                    /* decode side: slot = block_ids[t // Bd] * Bd + t % Bd */
                    const int64_t dblk = dst_bt[dst_off[r] + t / dst_block];
                    const int64_t doff = t % dst_block;
                    for (int64_t h = 0; h < kv_heads; ++h) {
                        /* head h lives on prefill card h / (H/Tp) ... */
                        const int64_t sp = h / src_heads;
                        const int64_t sh = h % src_heads;
                        /* ... and goes to decode card h / (H/Td) */
                        const int64_t dp = h / dst_heads;
                        const int64_t dh = h % dst_heads;
                        for (int64_t e = 0; e < D; ++e) {
                            const int64_t s_elem =
                                ((((l * C + c) * src_num_blocks + sblk) * src_block + soff)
                                     * src_heads + sh) * D + e;
                            const int64_t d_elem =
                                ((((l * C + c) * dst_num_blocks + dblk) * dst_block + doff)
                                     * dst_heads + dh) * D + e;
                            const uint8_t *from = src_pools[sp] + s_elem * elem_bytes;
                            uint8_t *to = dst_pools[dp] + d_elem * elem_bytes;
                            for (int32_t b = 0; b < elem_bytes; ++b)
                                to[b] = from[b];
                        }
                    }
                }
            }
        }
    }
    return 0;
}
