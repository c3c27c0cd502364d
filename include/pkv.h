/*
 * pkv.h -- attention over a paged KV cache on NVIDIA GB300 (sm_103a).
 *
 * Three operations make up one attention layer of a paged-KV inference step:
 *
 *   pkv_kv_store            write this step's new K/V rows into their pool slots
 *   pkv_paged_decode_attn   one query token per sequence over its cached keys
 *   pkv_paged_decode_attn_store  kv_store of the decode rows fused into the
 *                           decode attention (one launch instead of two)
 *   pkv_paged_prefill_attn  ragged causal attention of new tokens over a
 *                           cached prefix plus themselves
 *   pkv_paged_prefill_attn_shared  the same, for requests that share a cached
 *                           prefix: each shared key tile is read once for
 *                           all of a group's new tokens
 *
 * Sources of the operations' meaning:
 *   - mini-sglang "Engine Class": forward_batch takes a batch whose phase is
 *     prefill or decode and which carries out_loc (the cache slot of every new
 *     token); the engine's page_table maps logical to physical KV locations;
 *     its KV pool is paged (page_size 16 in the example config).
 *   - miniVLLM "Engine Architecture": prepare_prefill builds cu_seqlens_q
 *     (cumulative new-token counts, e.g. [0, 5, 8, 12]), slot_mapping and
 *     block_tables, skipping the num_cached_tokens of each sequence;
 *     prepare_decode builds context_lens, slot_mapping and block_tables;
 *     allocate_kv_cache lays each layer's K and V out as
 *     [num_blocks, block_size, num_kv_heads, head_dim].
 *   - miniVLLM "LLMEngine": model shapes with num_heads query heads sharing
 *     num_kv_heads KV heads (grouped-query attention), block_size 256.
 *
 * Conventions shared by every call:
 *   - bf16 tensors are passed as raw 16-bit patterns (pkv_bf16); all tensor
 *     pointers are DEVICE pointers owned by the caller, dense and C-contiguous
 *     in the layouts stated below, and 16-byte aligned.  The library never
 *     allocates, frees or keeps device memory.
 *   - The KV pool of one layer is k_cache and v_cache, each
 *     [num_pages, page_size, num_kv_heads, head_dim]; pool slot s is row s of
 *     the pool viewed as [num_pages * page_size, num_kv_heads, head_dim].
 *     Token position j of request r lives in slot
 *         page_table[r * page_table_stride + j / page_size] * page_size + j % page_size.
 *   - Query head h reads KV head h / (num_q_heads / num_kv_heads).
 *   - seq_lens[r] counts ALL keys request r attends to after this step's new
 *     tokens were stored: its cached prefix plus its new tokens.  kv_store must
 *     therefore run before the attention call that reads those tokens.
 *   - Pool slots holding no token of the request are never read, so their
 *     contents (even NaN) do not matter.
 *   - stream is a cudaStream_t (NULL = the legacy default stream).  Every call
 *     is asynchronous on that stream and does no host synchronisation; the
 *     launch configuration depends only on host arguments, never on device
 *     data, so the calls can be captured in a CUDA graph.
 *   - Errors the host can see (null pointers, bad sizes, unsupported shapes,
 *     misalignment, workspace too small) return a pkv_status at once and launch
 *     nothing.  Errors only the device can see (a page id outside the pool, a
 *     seq_len beyond the page-table row, a slot beyond the pool, bad
 *     cu_seqlens_q) are OR-ed as PKV_DEV_* bits into *dev_status when
 *     dev_status is not NULL; the affected rows are then skipped (kv_store) or
 *     written as NaN (attention), and nothing outside the caller's buffers is
 *     ever touched.  The kernels never trap.
 *   - Supported: head_dim 64 or 128; num_q_heads / num_kv_heads in {1, 2, 4, 8};
 *     page_size a power of two from 1 to 256.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t pkv_bf16;

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_EINVAL = 1,        /* bad argument: null pointer, size, alignment, workspace */
    PKV_EUNSUPPORTED = 2,  /* valid but not built: head_dim, GQA ratio, page_size, batch */
    PKV_ECUDA = 3,         /* a CUDA runtime call failed (launch, attribute, device query) */
} pkv_status;

/* Bits OR-ed into *dev_status by the kernels. */
#define PKV_DEV_BAD_SLOT    1  /* out_loc[t] >= num_pages * page_size: row not stored */
#define PKV_DEV_BAD_PAGE    2  /* a page id outside [0, num_pages): rows written as NaN */
#define PKV_DEV_BAD_SEQLEN  4  /* seq_len < 0, > page_table_stride * page_size, or < new tokens */
#define PKV_DEV_BAD_CUSEQ   8  /* cu_seqlens_q not monotone, not starting at 0, or new
                                  tokens beyond max_q_len / total_q_tokens */
#define PKV_DEV_TIMEOUT    16  /* an internal pipeline wait gave up (should never happen) */
#define PKV_DEV_BAD_WORKSPACE 32  /* prefill: the workspace counters were not zero when the
                                     call started (never cleared, or in use by another call
                                     at the same time); work may have been skipped */
#define PKV_DEV_BAD_SHARED 64  /* shared-prefix prefill: groups that do not partition the
                                  batch in order, a shared length that is negative, not a
                                  whole number of pages or longer than a member's cached
                                  prefix (the rows concerned written as NaN), or a member
                                  whose page-table row does not list the shared pages */

/* Human-readable name of a pkv_status value. */
const char *pkv_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int pkv_version(void);

/*
 * kv_store: copy each new token's K and V rows into its pool slot.
 *
 * mini-sglang "Engine Class" (forward_batch, out_loc) and miniVLLM "Engine
 * Architecture" (slot_mapping: the physical cache slot each new token is
 * written to; allocate_kv_cache: the pool layout).
 *
 *   k_new, v_new  [num_tokens, num_kv_heads, head_dim] bf16, read
 *   out_loc       [num_tokens] int32: destination slot, or < 0 to skip the
 *                 token (padding).  Two tokens with the same slot are a
 *                 caller error: which one lands is unspecified.
 *   k_cache, v_cache  the pool, [num_pages, page_size, num_kv_heads, head_dim],
 *                 written only at the listed slots, bit for bit.
 *   dev_status    optional device int32: PKV_DEV_BAD_SLOT when a slot is
 *                 >= num_pages * page_size (that token is skipped).
 * num_tokens == 0 is a no-op.
 */
pkv_status pkv_kv_store(const pkv_bf16 *k_new, const pkv_bf16 *v_new,
                        const int32_t *out_loc, int64_t num_tokens,
                        pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                        int64_t num_pages, int page_size, int num_kv_heads,
                        int head_dim, int32_t *dev_status, void *stream);

/*
 * Bytes of device workspace pkv_paged_decode_attn needs for these sizes on
 * the current device (partial softmax results of sequences whose keys are
 * split over several thread blocks, and the per-batch tile offsets).
 * Returns 0 for invalid sizes.
 */
size_t pkv_decode_workspace_size(int batch, int num_q_heads, int num_kv_heads,
                                 int head_dim);

/*
 * paged_decode_attn: one new query token per sequence attends to all
 * seq_lens[b] keys of its sequence (including its own, stored by kv_store).
 *
 * miniVLLM "Engine Architecture", prepare_decode: each sequence contributes
 * one token; context_lens holds the tokens processed so far; block_tables
 * give the physical block of each logical block.
 *
 *   q             [batch, num_q_heads, head_dim] bf16
 *   k_cache, v_cache  pool as above
 *   page_table    int32 rows of page_table_stride entries, row b for sequence b;
 *                 entries past ceil(seq_lens[b] / page_size) are never read
 *   seq_lens      [batch] int32, keys per sequence; 0 gives a zero output row
 *   softmax_scale multiplies q.k before the softmax (1/sqrt(head_dim) usually)
 *   workspace     device buffer of at least
 *                 pkv_decode_workspace_size(batch, num_q_heads, num_kv_heads,
 *                 head_dim) bytes, 16-byte aligned, no initial contents needed;
 *                 two calls in flight at once need two workspaces
 *   out           [batch, num_q_heads, head_dim] bf16:
 *                 out[b,h] = sum_j softmax_j(scale * q[b,h].k_j) v_j
 *                 accumulated in fp32 and rounded to bf16
 * batch must be <= 4096.
 */
pkv_status pkv_paged_decode_attn(const pkv_bf16 *q, const pkv_bf16 *k_cache,
                                 const pkv_bf16 *v_cache, const int32_t *page_table,
                                 int64_t page_table_stride, const int32_t *seq_lens,
                                 int batch, int num_q_heads, int num_kv_heads,
                                 int head_dim, int page_size, int64_t num_pages,
                                 float softmax_scale, void *workspace,
                                 size_t workspace_bytes, int32_t *dev_status,
                                 pkv_bf16 *out, void *stream);

/*
 * paged_decode_attn_store: pkv_kv_store of each sequence's one new K/V row
 * followed by pkv_paged_decode_attn, in one call (two kernels instead of
 * three).
 *
 * mini-sglang "Engine Class": in a decode batch each request brings one new
 * token whose K/V row is written to the cache slot out_loc names and which
 * its own query attends to; miniVLLM "Engine Architecture", prepare_decode:
 * slot_mapping holds the slot of each sequence's last position.
 *
 *   k_new, v_new  [batch, num_kv_heads, head_dim] bf16, read: the new rows
 *   out_loc       [batch] int32: the pool slot of sequence b's new row, which
 *                 must be the slot position seq_lens[b] - 1 maps to; < 0
 *                 skips the store (that position is then read from the pool
 *                 as it is)
 *   k_cache, v_cache  the pool, written at the out_loc slots bit for bit as
 *                 pkv_kv_store writes them, then read as by
 *                 pkv_paged_decode_attn
 *   out           exactly as kv_store followed by pkv_paged_decode_attn
 *   other arguments, workspace and limits as for pkv_paged_decode_attn.
 * Each row is stored by the thread block that reads the tile holding position
 * seq_lens[b] - 1 of that sequence, before it reads that tile.  Device errors
 * add to those of pkv_paged_decode_attn: PKV_DEV_BAD_SLOT when out_loc[b] is
 * >= num_pages * page_size (row not stored), or is not the slot of position
 * seq_lens[b] - 1 (row stored; blocks that read that slot in the same call may
 * see either value, so the outputs are unspecified).  A sequence with
 * seq_lens[b] == 0 still has its row stored and gets a zero output.
 */
pkv_status pkv_paged_decode_attn_store(const pkv_bf16 *q, const pkv_bf16 *k_new,
                                       const pkv_bf16 *v_new, const int32_t *out_loc,
                                       pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                                       const int32_t *page_table, int64_t page_table_stride,
                                       const int32_t *seq_lens, int batch, int num_q_heads,
                                       int num_kv_heads, int head_dim, int page_size,
                                       int64_t num_pages, float softmax_scale,
                                       void *workspace, size_t workspace_bytes,
                                       int32_t *dev_status, pkv_bf16 *out, void *stream);

/*
 * paged_prefill_attn: causal attention of each request's new tokens over its
 * cached prefix and themselves.
 *
 * miniVLLM "Engine Architecture", prepare_prefill: the new tokens of all
 * requests are concatenated (cached prefix tokens excluded) with offsets
 * cu_seqlens_q; block_tables map logical to physical blocks.  zero-to-sglang
 * "Chapter 1 mini-sglang: What an Inference Engine Looks Like", section on
 * Req: a request's extend length is its current length minus its cached
 * length.
 *
 *   q             [total_q_tokens, num_q_heads, head_dim] bf16
 *   cu_seqlens_q  [batch + 1] int32, cu_seqlens_q[0] = 0, non-decreasing;
 *                 request r owns new tokens cu_seqlens_q[r] .. cu_seqlens_q[r+1]-1
 *   seq_lens      [batch] int32: cached prefix c_r plus new tokens n_r
 *   max_q_len     host upper bound on every n_r (sizes the launch grid)
 *   workspace     device buffer of at least pkv_prefill_workspace_size() bytes,
 *                 16-byte aligned, holding the call's work-queue counters.  It
 *                 must be zero-filled once before its first use (cudaMemset);
 *                 every call returns it to zero when its last thread block
 *                 finishes, so it can be reused by later calls, graph replays
 *                 included.  Calls that may run at the same time (different
 *                 streams, or several captured calls in flight) need
 *                 workspaces of their own.  A call that finds the counters
 *                 not zero (a workspace never cleared, or in use by another
 *                 call at the same time) may skip work: it raises
 *                 PKV_DEV_BAD_WORKSPACE and its output is unspecified.
 *   out           [total_q_tokens, num_q_heads, head_dim] bf16: new token i of
 *                 request r (absolute position c_r + i) attends keys
 *                 0 .. c_r + i; accumulated in fp32, rounded to bf16
 * Other arguments as for pkv_paged_decode_attn.
 * The kernel is persistent (one thread block per SM); its blocks take their
 * first work item by block index and the rest from the workspace counters.
 */
pkv_status pkv_paged_prefill_attn(const pkv_bf16 *q, const int32_t *cu_seqlens_q,
                                  const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                                  const int32_t *page_table, int64_t page_table_stride,
                                  const int32_t *seq_lens, int batch,
                                  int64_t total_q_tokens, int max_q_len,
                                  int num_q_heads, int num_kv_heads, int head_dim,
                                  int page_size, int64_t num_pages, float softmax_scale,
                                  void *workspace, size_t workspace_bytes,
                                  int32_t *dev_status, pkv_bf16 *out, void *stream);

/* Bytes of device workspace pkv_paged_prefill_attn needs (a small constant). */
size_t pkv_prefill_workspace_size(void);

/*
 * paged_prefill_attn_shared: pkv_paged_prefill_attn for a batch in which
 * groups of requests share their leading cached keys (prefix caching: the
 * requests' page-table rows list the same physical pages for a common prefix,
 * which the pool holds once).
 *
 * zero-to-sglang "Chapter 1 mini-sglang: What an Inference Engine Looks
 * Like", the roadmap on prefix caching and RadixAttention: requests that
 * begin with the same tokens reuse one cached copy of that prefix's KV.
 * miniVLLM "Engine Architecture", prepare_prefill: block_tables map each
 * sequence's logical blocks to physical blocks, so several sequences can list
 * the same blocks.
 *
 * The result is that of pkv_paged_prefill_attn on the same arguments (every
 * new token attends keys 0 .. c_r + i of its own request); only the order of
 * work differs.  A work item is a block of a group's new tokens, packed back
 * to back across the group's requests: it runs over the group's shared keys
 * once for all its rows (no mask: every new token comes after the prefix),
 * then over each of its requests' own keys from the shared length on, that
 * request's rows causal and the others masked, with one online softmax per
 * row over both ranges.  So each shared K/V tile is loaded once per 256
 * packed query rows rather than once per request, and short requests no
 * longer leave their query tiles mostly empty.
 *
 *   prefix_group_start  [num_prefix_groups + 1] int32: group g is requests
 *                 prefix_group_start[g] .. prefix_group_start[g+1]-1; the
 *                 groups partition the batch in order (first entry 0, last
 *                 entry batch, strictly increasing); a request that shares
 *                 nothing is a group of one with prefix_len 0
 *   prefix_len    [num_prefix_groups] int32: keys 0 .. prefix_len[g]-1 are
 *                 shared by the group's requests: a whole number of pages,
 *                 listed first in each member's page-table row (the first
 *                 member's row is the one read), and within every member's
 *                 cached prefix.  0 = nothing shared.
 *   num_prefix_groups  groups; 0 makes the call pkv_paged_prefill_attn
 *   max_group_tokens   host upper bound on the new tokens of any one group
 *                 (sizes the grid); 0 makes the call pkv_paged_prefill_attn
 *   workspace     as for pkv_paged_prefill_attn (pkv_prefill_workspace_size()
 *                 bytes of work-queue counters, zero-filled once)
 * Other arguments as for pkv_paged_prefill_attn.  Device-detected errors add
 * PKV_DEV_BAD_SHARED (see above) to those of pkv_paged_prefill_attn.
 */
pkv_status pkv_paged_prefill_attn_shared(const pkv_bf16 *q, const int32_t *cu_seqlens_q,
                                         const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                                         const int32_t *page_table, int64_t page_table_stride,
                                         const int32_t *seq_lens, int batch,
                                         int64_t total_q_tokens, int max_q_len,
                                         int num_q_heads, int num_kv_heads, int head_dim,
                                         int page_size, int64_t num_pages, float softmax_scale,
                                         const int32_t *prefix_group_start,
                                         const int32_t *prefix_len, int num_prefix_groups,
                                         int max_group_tokens, void *workspace,
                                         size_t workspace_bytes, int32_t *dev_status,
                                         pkv_bf16 *out, void *stream);

/*
 * Size of the fixed scratch area that pkv_paged_decode_attn_noalloc uses in
 * place of a caller-provided workspace (4 MiB, enough for head_dim 128 with
 * 8 query heads per KV head on GPUs of up to 240 SMs).
 */
#define PKV_NOALLOC_SCRATCH_BYTES 4194304

/*
 * pkv_paged_decode_attn_noalloc: the same decode attention as
 * pkv_paged_decode_attn, for callers that cannot hand the library a workspace.
 *
 * The pages this library follows have no counterpart of this call; it exists
 * for callers that are not able to allocate device memory when they call
 * attention: an inference runtime that plans every byte of device memory up
 * front and forbids allocation on its hot path, a plugin inside another
 * framework that is given only its inputs and outputs, or code that must not
 * touch the allocator at all.  Instead of a workspace argument, the call uses
 * one scratch array of PKV_NOALLOC_SCRATCH_BYTES that the library declares in
 * device memory; every GPU that loads the library holds that array until the
 * process exits.  The call itself never allocates or frees memory (no
 * cudaMalloc, cudaFree or allocating library routine).
 *
 *   - Arguments, layouts, results and device error bits are those of
 *     pkv_paged_decode_attn without workspace / workspace_bytes.
 *   - Sizes whose workspace (pkv_decode_workspace_size) would exceed
 *     PKV_NOALLOC_SCRATCH_BYTES are rejected with PKV_EUNSUPPORTED and nothing
 *     is launched.
 *   - The first call on each device looks up the device address of the
 *     scratch array for that device (a host-side query, made once per device
 *     with that device current).  Make that first call before any stream
 *     capture.
 *   - All calls share the one scratch array and it keeps whatever the last
 *     call left there; the kernels write every scratch word they read, so
 *     nothing needs clearing between calls.  Two calls whose kernels overlap
 *     on the GPU (different streams, no ordering between them) race on the
 *     scratch array and may return wrong results: order them on one stream or
 *     with events.
 */
pkv_status pkv_paged_decode_attn_noalloc(const pkv_bf16 *q, const pkv_bf16 *k_cache,
                                         const pkv_bf16 *v_cache, const int32_t *page_table,
                                         int64_t page_table_stride, const int32_t *seq_lens,
                                         int batch, int num_q_heads, int num_kv_heads,
                                         int head_dim, int page_size, int64_t num_pages,
                                         float softmax_scale, int32_t *dev_status,
                                         pkv_bf16 *out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
