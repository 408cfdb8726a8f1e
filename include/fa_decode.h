/*
 * fa_decode.h -- C ABI of the GB300 (sm_103a) decode-step attention library.
 *
 * One call computes, for every sequence b and query head h of a decode step,
 *
 *     out[b][h][:] = softmax(scale * q[b][h] . K_b[kv][t] for t in [lo_b, L_b)) @ V_b[kv]
 *
 * with kv = h / (n_q_heads / n_kv_heads), L_b = seq_lens[b] and
 * lo_b = (window[b] > 0 && L_b > window[b]) ? L_b - window[b] : 0.
 * Sources (mlx-native page "flash_attn_vec_hybrid.metal", kernel
 * flash_attn_vec_hybrid_impl and its batched / GQA siblings):
 *   - GQA head map: the "map query head to KV head" step;
 *   - length and sliding-window rule: the per-chunk mask block (keys with
 *     logical index < kv_seq_len - sliding_window are masked, window 0 =
 *     global, the tessl page "nn.rs" flash_attn_decode: "window == 0 selects
 *     the global rule");
 *   - online softmax over KV blocks and the split-K partial (O, S, M) with a
 *     log-sum-exp merge: the "Online softmax" block, the cross-simdgroup
 *     reduce and the NWG > 1 partial write, and the separate reduce pass
 *     (flash_attn_vec_reduce, tessl flash_attn_decode_reduce);
 *   - an empty attended range gives a zero row ("S == 0 ? 0").
 * The int8 V variant stores V as int8 codes times one fp16 scale per 32
 * consecutive head_dim elements (dequantisation as ggml block_q8_0 on the
 * DS4Server page "dsv4_hc.metal").
 *
 * All pointers passed to fa_decode are DEVICE pointers unless stated, owned
 * by the caller; the library allocates nothing, keeps no pointer after
 * return, and enqueues all work on `stream` (a cudaStream_t; NULL = legacy
 * default stream) without synchronising.  Every function returns 0 on success
 * or a negative FA_ERR_* code; nothing is launched when a check fails, and
 * fa_decode_last_error() returns a message for the calling thread's last
 * failure.
 */
#ifndef FA_DECODE_H
#define FA_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FA_API __attribute__((visibility("default")))

/* Error codes. */
#define FA_OK 0
#define FA_ERR_NULL (-1)        /* a required pointer is NULL */
#define FA_ERR_HEAD_DIM (-2)    /* head_dim not 128 or 256 */
#define FA_ERR_HEADS (-3)       /* heads <= 0, or n_q_heads % n_kv_heads != 0, or group > 64 */
#define FA_ERR_WORKSPACE (-4)   /* workspace smaller than fa_decode_workspace_size() */
#define FA_ERR_SCALE (-5)       /* scale not finite */
#define FA_ERR_LAYOUT (-6)      /* bad batch / page_size / block counts / capacity */
#define FA_ERR_ALIAS (-7)       /* out overlaps an input or the workspace */
#define FA_ERR_CUDA (-8)        /* a CUDA call or kernel launch failed */
#define FA_ERR_ALIGN (-9)       /* a pointer is not aligned as its entry point requires */

/* Device-side status bits, reported by fa_decode_device_status(). */
#define FA_STATUS_LEN_CLAMPED 1u   /* a seq_lens entry was < 0 or > capacity and was clamped */
#define FA_STATUS_BAD_BLOCK 2u     /* a block-table entry was outside [0, num_blocks); tile skipped */
#define FA_STATUS_WAIT_TIMEOUT 4u  /* a copy wait passed its ~1 s limit; that split's result is void */
#define FA_STATUS_POS_RANGE 8u     /* fa_append_kv: a position outside [0, capacity); store skipped */
#define FA_STATUS_BAD_SLOT 16u     /* a slot id outside [0, n_slots): zero row / store skipped */

/*
 * fa_decode -- one decode step of attention for `batch` sequences.
 *
 * q          [batch][n_q_heads][head_dim] fp16.
 * k_cache    fp16 keys.  Paged (block_table != NULL):
 *              [num_blocks][n_kv_heads][page_size][head_dim];
 *            contiguous (block_table == NULL):
 *              [batch][n_kv_heads][capacity][head_dim], capacity = max_blocks_per_seq.
 * v_cache    values, same layout as k_cache: fp16 when v_scales == NULL, else int8.
 * v_scales   NULL (fp16 V) or the fp16 scales of int8 V, one per 32 head_dim
 *            elements: [...same leading dims as v_cache...][head_dim / 32].
 * block_table int32 [batch][max_blocks_per_seq]: logical page p of sequence b
 *            lives in physical block block_table[b][p]; only the pages that
 *            hold keys in the attended range are read.  NULL = contiguous.
 * seq_lens   int32 [batch]: keys in each sequence's cache (the current token
 *            included).  Values outside [0, capacity] are clamped on the
 *            device and flagged (FA_STATUS_LEN_CLAMPED).
 * window     int32 [batch] sliding-window sizes (0 = global), or NULL (all global).
 * scale      softmax scale applied to q.k (e.g. 1/sqrt(head_dim)).
 * out        [batch][n_q_heads][head_dim] fp32, written in full (zero rows
 *            for empty ranges).  Must not overlap any input or the workspace.
 * batch      number of sequences (0 is a no-op).
 * page_size  tokens per physical block, a positive multiple of 16 (ignored
 *            when contiguous).
 * max_blocks_per_seq  block-table row length (paged), or the per-sequence
 *            capacity in tokens (contiguous; a multiple of 16 for int8 V).
 * num_blocks physical blocks in the paged caches (bounds for block ids;
 *            ignored when contiguous).
 * workspace  device scratch of at least fa_decode_workspace_size() bytes,
 *            16-byte aligned; contents need no initialisation and are not
 *            preserved.  May be NULL when that size is 0.  Calls that may
 *            overlap on the GPU must not share a workspace.
 * stream     cudaStream_t to enqueue on.  A call does all its work in its
 *            launches on `stream`, and the split plan is made on the device
 *            from seq_lens and window, so after a first call outside any
 *            capture (which sets the kernels' shared-memory limits) a call
 *            may be captured in a CUDA graph and replayed with new
 *            device-side lengths.
 *
 * q, k_cache, v_cache, v_scales and out must be 16-byte aligned, and
 * seq_lens, block_table and window 4-byte aligned (else FA_ERR_ALIGN).
 *
 * Plans.  A step normally runs two kernels: a persistent split kernel that
 * gives every warp an equal share of the step's tiles, then a log-sum-exp
 * merge.  A small step -- one column group per KV head, and few and short
 * enough (sequence, KV head) units that a thread-block cluster of 8, 4, 2 or 1
 * CTAs per unit fits on the GPU at once with at most 4 tiles of 16 tokens per
 * warp at head_dim 128 (1 at 256) -- instead runs one kernel: each unit's
 * cluster splits its tiles over its warps and folds their partials in
 * distributed shared memory, so the workspace is not written.
 * Setting FA_DECODE_PLAN=streamk in the environment keeps every step on the
 * two-kernel plan.  Both plans compute the same result within the stated
 * tolerances.
 */
FA_API int fa_decode(const void *q, const void *k_cache, const void *v_cache,
                     const void *v_scales, const int32_t *block_table,
                     const int32_t *seq_lens, int n_q_heads, int n_kv_heads, int head_dim,
                     float scale, const int32_t *window, void *out, int batch, int page_size,
                     int max_blocks_per_seq, int num_blocks, void *workspace,
                     size_t workspace_bytes, void *stream);

/*
 * fa_decode_batch_invariant -- fa_decode whose result for a sequence does not
 * depend on the rest of the batch, bit for bit: a sequence decoded alone,
 * or in any batch, in any position, gives the same bytes.  The hf2q page
 * "batched_body.rs" holds its batched multi-slot decode to this rule against
 * serial single-slot runs (its slot-aware parity tests).
 *
 * fa_decode's split plan gives every worker an equal share of the whole
 * batch's tiles, so where a sequence's KV range is cut, and so the rounding
 * of its merged result, depends on the batch.  Here each (sequence, KV head
 * [, head group]) range is cut into splits of split_tokens keys counted from
 * its first attended key, whatever the batch.  Each split is computed from
 * scratch by one worker.  The splits' partials are merged in split order.
 * Workers take equal runs of whole splits, so the balance is coarser than
 * fa_decode's; a sequence of at most split_tokens keys is not split at all.
 *
 * split_tokens  a positive multiple of 16: keys per split (e.g. 512).
 * workspace     fa_decode_batch_invariant_workspace_size() bytes; contents
 *               need no initialisation.
 * Other arguments, layouts, rules and errors as fa_decode, plus
 * FA_ERR_LAYOUT for a bad split_tokens.  The result equals fa_decode's
 * within the same tolerances.
 */
FA_API int fa_decode_batch_invariant(const void *q, const void *k_cache, const void *v_cache,
                                     const void *v_scales, const int32_t *block_table,
                                     const int32_t *seq_lens, int n_q_heads, int n_kv_heads,
                                     int head_dim, float scale, const int32_t *window, void *out,
                                     int batch, int page_size, int max_blocks_per_seq,
                                     int num_blocks, int split_tokens, void *workspace,
                                     size_t workspace_bytes, void *stream);

/* Scratch bytes for fa_decode_batch_invariant: one partial (D floats of O
 * plus max and sum) per query head and split of every sequence at
 * max_kv_len keys.  Host-only; 0 for invalid sizes, and for sizes whose
 * scratch would not fit in a size_t (the decode call then fails with
 * FA_ERR_WORKSPACE whatever buffer it is given). */
FA_API size_t fa_decode_batch_invariant_workspace_size(int batch, int n_q_heads, int n_kv_heads,
                                                       int head_dim, int max_kv_len,
                                                       int split_tokens);

/*
 * The batch-invariant plan for the other two decode forms, with the same
 * guarantee (a sequence's bytes do not depend on the rest of the batch):
 *   fa_decode_multi_batch_invariant -- fa_decode_multi's arguments plus
 *     split_tokens; workspace of
 *     fa_decode_multi_batch_invariant_workspace_size() bytes;
 *   fa_decode_ring_batch_invariant -- fa_decode_ring's arguments plus
 *     split_tokens; workspace of fa_decode_batch_invariant_workspace_size(
 *     batch, n_q_heads, n_kv_heads, head_dim, capacity + 16, split_tokens)
 *     bytes (a ring's attended range can straddle one more tile).
 * Rules and errors as the forms they extend and as fa_decode_batch_invariant.
 */
FA_API int fa_decode_multi_batch_invariant(const void *q, const void *k_cache,
                                           const void *v_cache, const void *v_scales,
                                           const int32_t *block_table, const int32_t *seq_lens,
                                           int n_queries, int n_q_heads, int n_kv_heads,
                                           int head_dim, float scale, const int32_t *window,
                                           void *out, int batch, int page_size,
                                           int max_blocks_per_seq, int num_blocks,
                                           int split_tokens, void *workspace,
                                           size_t workspace_bytes, void *stream);
FA_API size_t fa_decode_multi_batch_invariant_workspace_size(int batch, int n_queries,
                                                             int n_q_heads, int n_kv_heads,
                                                             int head_dim, int max_kv_len,
                                                             int split_tokens);
FA_API int fa_decode_ring_batch_invariant(const void *q, const void *k_cache,
                                          const void *v_cache, const void *v_scales,
                                          const int32_t *seq_lens, int n_q_heads, int n_kv_heads,
                                          int head_dim, float scale, const int32_t *window,
                                          void *out, int batch, int capacity, int split_tokens,
                                          void *workspace, size_t workspace_bytes, void *stream);

/*
 * fa_decode_multi -- several query tokens per sequence in one call: the
 * speculative-verify form of the decode step (the n_queries field of the
 * pages' params; causal rule of tessl's flash_attn_rows on the "nn.rs" page).
 *
 * q   [batch][n_queries][n_q_heads][head_dim] fp16: each sequence's last
 *     n_queries tokens, all already in the cache (seq_lens counts them).
 * out [batch][n_queries][n_q_heads][head_dim] fp32.
 * Query j of sequence b sits at position L_b - n_queries + j and attends the
 * keys up to and including itself; a window W > 0 keeps its last W keys.  A
 * query whose position is negative gets a zero row.  n_queries = 1 is
 * fa_decode.  The workspace must hold fa_decode_multi_workspace_size() bytes.
 * Layouts, other arguments and errors as fa_decode; n_queries in [1, 256].
 */
FA_API int fa_decode_multi(const void *q, const void *k_cache, const void *v_cache,
                           const void *v_scales, const int32_t *block_table,
                           const int32_t *seq_lens, int n_queries, int n_q_heads, int n_kv_heads,
                           int head_dim, float scale, const int32_t *window, void *out, int batch,
                           int page_size, int max_blocks_per_seq, int num_blocks,
                           void *workspace, size_t workspace_bytes, void *stream);

/* Scratch bytes for fa_decode_multi (host-only; arguments as
 * fa_decode_workspace_size plus n_queries). */
FA_API size_t fa_decode_multi_workspace_size(int batch, int n_queries, int n_q_heads,
                                             int n_kv_heads, int head_dim, int max_kv_len,
                                             int num_sms);

/*
 * fa_decode_ring -- fa_decode over a ring cache: the storage mode of a
 * sliding-window layer on the mlx-native page (flash_attn_vec_hybrid_batched,
 * "sliding ring storage"): each sequence's contiguous [capacity] rows are
 * reused round-robin, token t living at row t % capacity, and the live
 * length is min(tokens seen, capacity).
 *
 * k_cache, v_cache (and v_scales) [batch][n_kv_heads][capacity][...] as the
 * contiguous layout of fa_decode; capacity a positive multiple of 16.
 * seq_lens[b] = tokens sequence b has seen (may exceed capacity); the keys
 * attended are the last min(seq_lens[b], capacity) tokens, further cut to the
 * last window[b] when window[b] > 0.  The workspace must hold
 * fa_decode_workspace_size(batch, n_q_heads, n_kv_heads, head_dim,
 * capacity + 16, 0) bytes.  Other arguments, rules and errors as fa_decode.
 */
FA_API int fa_decode_ring(const void *q, const void *k_cache, const void *v_cache,
                          const void *v_scales, const int32_t *seq_lens, int n_q_heads,
                          int n_kv_heads, int head_dim, float scale, const int32_t *window,
                          void *out, int batch, int capacity, void *workspace,
                          size_t workspace_bytes, void *stream);

/*
 * fa_decode_slots -- fa_decode over a pool of per-slot contiguous (ring = 0)
 * or ring (ring = 1) caches, each batch row reading the slot a device-side
 * slot map names.  The batched kernels of the mlx-native page
 * (flash_attn_vec_hybrid_batched and its GQA / per-slot-bucket sibling) read
 * per query row the row's slot (slot_id_arr) and position (seq_pos_arr) on
 * the device and address that slot's [n_kv_heads][capacity][head_dim] rows;
 * this is that indirection, so a server decodes only its active slots (any
 * subset of the pool, in any order) without copying caches.
 *
 * k_cache, v_cache (and v_scales) [n_slots][n_kv_heads][capacity][...], the
 *            contiguous layout of fa_decode (fa_decode_ring's when ring = 1).
 * slot_ids   int32 [batch] (device): row b uses slot slot_ids[b].  A slot id
 *            outside [0, n_slots) gives row b a zero output and sets
 *            FA_STATUS_BAD_SLOT.  Rows may share a slot (read-only).
 * q, out, seq_lens, window  per row, as fa_decode: seq_lens[b] is the length
 *            of row b's slot (the page's seq_pos + 1; for a ring the tokens
 *            the slot has seen, as fa_decode_ring).
 * n_slots    slots in the pool; capacity  tokens per slot (a multiple of 16
 *            for a ring or for int8 V).
 * workspace  fa_decode_workspace_size(batch, n_q_heads, n_kv_heads, head_dim,
 *            ring ? capacity + 16 : capacity, 0) bytes.
 * Other arguments, rules and errors as fa_decode; slot_ids is 4-byte aligned
 * (else FA_ERR_ALIGN).  The split plan covers the batch rows only, so idle
 * slots cost nothing.
 */
FA_API int fa_decode_slots(const void *q, const void *k_cache, const void *v_cache,
                           const void *v_scales, const int32_t *slot_ids,
                           const int32_t *seq_lens, int n_q_heads, int n_kv_heads, int head_dim,
                           float scale, const int32_t *window, void *out, int batch, int n_slots,
                           int capacity, int ring, void *workspace, size_t workspace_bytes,
                           void *stream);

/*
 * fa_decode_workspace_size -- bytes of scratch fa_decode needs for these
 * sizes: the split-K partials (unnormalised O plus running max and sum per
 * query head and split; the "partial scratch B*H*chunks*(D+2)" of tessl's
 * flash_attn_decode).  max_kv_len is the per-sequence capacity in tokens
 * (max_blocks_per_seq * page_size when paged).  num_sms <= 0 queries the
 * current device; pass the same value fa_decode will see (it uses the
 * current device's SM count).  Host-only; never launches.  Returns 0 for
 * invalid sizes.
 */
FA_API size_t fa_decode_workspace_size(int batch, int n_q_heads, int n_kv_heads, int head_dim,
                                       int max_kv_len, int num_sms);

/*
 * fa_quantize_v_int8 -- pack fp32 values into the int8 V cache format.
 * x [n_rows][head_dim] fp32 (device) -> codes [n_rows][head_dim] int8 and
 * scales [n_rows][head_dim/32] fp16 (device).  Per block of 32 elements:
 * s = fp16 round-to-nearest-even(max|x| / 127); code = clamp(round-half-even(
 * x / s), -127, 127), all zero when s == 0.  (The pages print only the
 * dequantisation, ggml block_q8_0 on the DS4Server page "dsv4_hc.metal";
 * this quantiser is the plain symmetric reading.)  head_dim % 32 == 0; x is
 * 4-byte and scales 2-byte aligned (else FA_ERR_ALIGN).
 */
FA_API int fa_quantize_v_int8(const float *x, long long n_rows, int head_dim, int8_t *codes,
                              void *scales, void *stream);

/*
 * fa_append_kv -- write one decode step's K and V rows into the cache, the
 * step before attention on every decode (the hf2q page "batched_body.rs"
 * copies the step's K row f32 -> f16 into the cache at cache_pos; tessl's
 * kv_store_timestep on the "nn.rs" page stores at a device-side offset and
 * makes an out-of-range store a no-op).
 *
 * k_new, v_new [batch][n_kv_heads][head_dim] fp32 (device).
 * positions    int32 [batch] (device): the token index t each sequence writes.
 * For every (b, kv): K row (b, kv, t) <- fp16 round-to-nearest-even of
 * k_new[b][kv]; V row <- the same for an fp16 V cache (v_scales == NULL), or
 * the int8 codec of fa_quantize_v_int8 (codes + one fp16 scale per 32).
 * Cache layouts, block_table, page_size, max_blocks_per_seq and num_blocks
 * are those of fa_decode.  A position outside [0, capacity) leaves the
 * sequence's rows untouched and sets FA_STATUS_POS_RANGE; an unmapped block
 * id (outside [0, num_blocks)) skips that store and sets FA_STATUS_BAD_BLOCK.
 * head_dim must be a positive multiple of 32.  The caches must not overlap
 * k_new, v_new or positions.  Every pointer is aligned to its element type
 * (4 bytes for fp32 and int32, 2 for fp16), else FA_ERR_ALIGN.
 */
FA_API int fa_append_kv(const float *k_new, const float *v_new, void *k_cache, void *v_cache,
                        void *v_scales, const int32_t *block_table, const int32_t *positions,
                        int batch, int n_kv_heads, int head_dim, int page_size,
                        int max_blocks_per_seq, int num_blocks, void *stream);

/*
 * fa_append_kv_ring -- fa_append_kv into a ring cache of fa_decode_ring:
 * token positions[b] >= 0 goes to row positions[b] % capacity (a negative
 * position stores nothing and sets FA_STATUS_POS_RANGE).
 */
FA_API int fa_append_kv_ring(const float *k_new, const float *v_new, void *k_cache, void *v_cache,
                             void *v_scales, const int32_t *positions, int batch, int n_kv_heads,
                             int head_dim, int capacity, void *stream);

/*
 * fa_append_kv_slots -- fa_append_kv (ring = 0) or fa_append_kv_ring
 * (ring = 1) into the pool of fa_decode_slots: row b of k_new, v_new and
 * positions writes slot slot_ids[b] (int32 [batch], device) at token
 * positions[b].  A slot id outside [0, n_slots) stores nothing and sets
 * FA_STATUS_BAD_SLOT.  Two rows naming the same slot and row race; give each
 * row its own slot.  Other rules and errors as the append it extends.
 */
FA_API int fa_append_kv_slots(const float *k_new, const float *v_new, void *k_cache,
                              void *v_cache, void *v_scales, const int32_t *slot_ids,
                              const int32_t *positions, int batch, int n_kv_heads, int head_dim,
                              int n_slots, int capacity, int ring, void *stream);

/*
 * fa_gather_kv_debug -- copy sequence b's first n_tokens cache rows, through
 * the same page-address path fa_decode's loader uses, into dense
 * [n_kv_heads][n_tokens][row_bytes] (device).  row_bytes = 2*head_dim for K
 * or fp16 V, head_dim for int8 V, head_dim/16 for the scales.  A byte copy;
 * exists so the block-table indirection can be checked bit for bit.
 * Block ids are range-checked against num_blocks (FA_ERR_LAYOUT on the host
 * is impossible for device tables; bad ids leave zero rows and set
 * FA_STATUS_BAD_BLOCK).  block_table is 4-byte aligned (else FA_ERR_ALIGN).
 */
FA_API int fa_gather_kv_debug(const void *cache, int row_bytes, const int32_t *block_table,
                              int b, int n_kv_heads, int page_size, int max_blocks_per_seq,
                              int num_blocks, int n_tokens, void *dense, void *stream);

/*
 * fa_selftest_wait_timeout -- failure-path self-test (no counterpart on the
 * pages).  Launches one warp that arms a shared-memory barrier nothing will
 * complete and waits on it with the same bounded wait the decode kernels use
 * for their copies.  After about one second the wait gives up, the warp exits
 * and FA_STATUS_WAIT_TIMEOUT is set, showing that a copy that never lands
 * surfaces as a status bit (read with fa_decode_device_status) rather than a
 * hang, with the context still usable.
 */
FA_API int fa_selftest_wait_timeout(void *stream);

/*
 * fa_decode_device_status -- wait for `stream`, then read and clear the
 * device-side FA_STATUS_* bits accumulated since the last call.
 */
FA_API int fa_decode_device_status(unsigned int *status, void *stream);

/*
 * fa_decode_noalloc -- fa_decode for callers that cannot allocate device
 * memory.  The pages have no counterpart; this is a deployment convenience.
 *
 * Some callers cannot call cudaMalloc (or any allocator) at the point where
 * they run attention: for example a plugin inside a host framework that owns
 * every device allocation through its own pool and forbids side allocations,
 * or code on a latency-critical path where an allocation's implicit device
 * synchronisation is not acceptable.  Such a caller still owns and passes
 * every input and the output, but has no workspace to give.
 *
 * This entry point takes the same arguments as fa_decode minus the
 * workspace, and runs the same kernels with their split-K scratch placed in a
 * fixed array compiled into the library (FA_NOALLOC_SCRATCH_BYTES, 8 MiB).
 * Every GPU that loads the library holds that array until the process exits.
 * It allocates nothing and calls no allocating routine.
 *
 * Limits and rules:
 *   - a call whose own scratch need (the workspace fa_decode takes for these
 *     sizes and this V type; fa_decode_workspace_size, which covers both V
 *     types, bounds it) exceeds FA_NOALLOC_SCRATCH_BYTES is rejected with
 *     FA_ERR_WORKSPACE and a message stating both sizes; nothing is launched;
 *   - the first call in a CUDA context (for runtime-API callers: the first
 *     call on a device) looks up the array's device address in that context,
 *     with it current, and caches it under the context's id; make that
 *     first call before any stream capture begins;
 *   - all calls share the one array: calls whose kernels overlap on the GPU
 *     (different streams, or different host threads on one device) race on
 *     it and give wrong results.  Serialise them, e.g. on one stream.  The
 *     scratch needs no clearing between calls (every value read in a call is
 *     written earlier in that call).
 */
#define FA_NOALLOC_SCRATCH_BYTES (8u << 20)
FA_API int fa_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                             const void *v_scales, const int32_t *block_table,
                             const int32_t *seq_lens, int n_q_heads, int n_kv_heads,
                             int head_dim, float scale, const int32_t *window, void *out,
                             int batch, int page_size, int max_blocks_per_seq, int num_blocks,
                             void *stream);

/*
 * fa_decode_profile_next -- instrumentation for timing.  The next fa_decode
 * call made on this host thread records the cudaEvent_t `split_start` on its
 * stream just before its split-K kernel and `split_end` just after it (the
 * merge kernel follows), then forgets both.  Either may be NULL.  No work is
 * skipped or changed.
 */
FA_API int fa_decode_profile_next(void *split_start, void *split_end);

/* Message for the calling thread's last failed call ("" if none). */
FA_API const char *fa_decode_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_DECODE_H */
