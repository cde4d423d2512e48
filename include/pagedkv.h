/*
 * pagedkv.h -- C ABI of the GB300 (sm_103a) paged KV-cache decode path.
 *
 * The method is PagedAttention as the vLLM pages describe it:
 *   - vLLM concept page (compassingai.com), "15 分钟专家深入" item 2: the KV
 *     cache is cut into fixed-size blocks of 16 tokens, each sequence owns a
 *     page table (block table) of physical block ids, new blocks are filled
 *     on demand, and a GPU kernel gathers the blocks through the table;
 *   - same page, "技术原理": gather the blocks named by the table, then
 *     scores = Q K^T / sqrt(head_dim), softmax, times V;
 *   - vLLM v0.17.1 notes (admirer.cn), "修复方案": blocks freshly handed to
 *     attention are zeroed on the GPU before first use, with the block ids
 *     sent from host memory together with the launch;
 *   - vLLM internals (naphjohn.github.io), §1.1 and Figure 1: blocks lie
 *     anywhere in the pool and shared prefixes point at the same block.
 *
 * Conventions for every entry point:
 *   - Pointers are DEVICE pointers unless a parameter says otherwise.  The
 *     caller owns all memory; the library allocates nothing per call.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *     Every call is asynchronous on that stream.
 *   - The return value reports errors the host can see before launching
 *     (null pointers, bad sizes or dtypes, CUDA launch failures).  Errors
 *     only the device can see (a slot, block id or sequence length out of
 *     range, an internal wait that timed out) skip the offending item and
 *     are recorded in a device error word that pkv_check() reads and clears.
 *     No kernel traps.
 *   - Layout of both caches: [num_blocks, block_size, num_kv_heads,
 *     head_dim], row-major and contiguous; block_size must be 16, head_dim
 *     64 or 128.  Elements are bf16, or OCP E4M3 bytes with one fp32 scale
 *     per cache (value = decode(byte) * scale).
 *   - Entry points are thread-safe; calls on the same stream are ordered.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_OK = 0,
    PKV_ERR_ARG = 1,       /* null pointer, negative size, bad partition  */
    PKV_ERR_DTYPE = 2,     /* unknown cache dtype                          */
    PKV_ERR_SHAPE = 3,     /* block_size != 16, head_dim not 64/128,
                              num_heads not a multiple of num_kv_heads     */
    PKV_ERR_CUDA = 4,      /* a CUDA runtime/driver call failed            */
    PKV_ERR_RANGE = 5,     /* device: slot / block id / seq_len out of range */
    PKV_ERR_TIMEOUT = 6,   /* device: a bounded wait gave up               */
    PKV_ERR_WORKSPACE = 7  /* workspace missing or too small               */
} pkv_status;

typedef enum { PKV_BF16 = 0, PKV_FP8_E4M3 = 1 } pkv_dtype;

/* A paged KV cache.  The struct is read during the call only; the buffers
 * it points at stay owned by the caller. */
typedef struct {
    void *key_cache;       /* [num_blocks, block_size, num_kv_heads, head_dim] */
    void *value_cache;     /* same shape and dtype as key_cache             */
    int32_t num_blocks;
    int32_t block_size;    /* must be 16                                    */
    int32_t num_kv_heads;
    int32_t head_dim;      /* 64 or 128                                     */
    int32_t dtype;         /* pkv_dtype                                     */
    float k_scale;         /* fp8 only: value = decode(byte) * k_scale      */
    float v_scale;         /* fp8 only                                      */
} pkv_cache;

/* Slot-mapped KV write.  Source: vLLM concept page (compassingai.com),
 * "15 分钟专家深入" item 2 (blocks filled on demand as tokens arrive) and its
 * mention of high-bandwidth KV pack/unpack kernels.
 *   k, v          bf16 [num_tokens, num_kv_heads, head_dim], contiguous.
 *   slot_mapping  int64 [num_tokens]; slot s >= 0 writes row s % 16 of
 *                 block s / 16; s < 0 skips the token (padding);
 *                 s >= num_blocks * 16 is a device range error (skipped).
 * bf16 caches receive the bits unchanged.  fp8 caches receive
 * E4M3(round-to-nearest-even, saturate to +-448)(x / scale) where the
 * division is IEEE binary32 and scale is k_scale or v_scale.
 * Tokens must not share a slot (the order between them is unspecified). */
pkv_status paged_kv_write(const void *k, const void *v,
                          const int64_t *slot_mapping, int64_t num_tokens,
                          const pkv_cache *cache, void *stream);

/* Zero freshly allocated blocks.  Source: vLLM v0.17.1 notes (admirer.cn),
 * "修复方案": only the newly allocated blocks are cleared, every byte of
 * their K and V segments, before attention first reads them; the ids travel
 * from host memory with the launch.
 *   block_ids     int32 [n]; on the host when ids_on_host != 0 (any host
 *                 memory: the ids are copied into the launch parameters, so
 *                 the buffer may be reused as soon as the call returns),
 *                 otherwise on the device.
 * Ids outside [0, num_blocks) are device range errors (skipped).  No other
 * block is touched. */
pkv_status paged_kv_zero_blocks(const pkv_cache *cache,
                                const int32_t *block_ids, int64_t n,
                                int ids_on_host, void *stream);

/* Zeroing of freshly allocated blocks and the slot-mapped write of new
 * tokens in one launch: the result is that of paged_kv_zero_blocks(cache,
 * block_ids, n, ids_on_host) followed by paged_kv_write(k, v, slot_mapping,
 * num_tokens, cache).  Sources: those of the two calls (vLLM v0.17.1 notes,
 * "修复方案"; vLLM concept page, "15 分钟专家深入" item 2).  Arguments and
 * device range errors are those of the two calls; either count may be 0.
 * A zeroing CTA clears only the rows of its block that no token of this
 * call writes, and the writing CTAs write every token, so the two never
 * touch the same bytes.  More than 4096 host ids take several launches, the
 * first of which also writes the tokens. */
pkv_status paged_kv_zero_and_write(const void *k, const void *v,
                                   const int64_t *slot_mapping, int64_t num_tokens,
                                   const pkv_cache *cache, const int32_t *block_ids,
                                   int64_t n, int ids_on_host, void *stream);

/* Copy whole blocks: for each i, every byte of key_cache[dst_ids[i]] and
 * value_cache[dst_ids[i]] becomes the byte of block src_ids[i].  Source:
 * vLLM internals (naphjohn.github.io), §1.1 (copy-on-write of a shared
 * prefix block that one sequence must modify).
 *   src_ids, dst_ids  int32 [n]; on the host when ids_on_host != 0 (copied
 *                 into the launch parameters), otherwise on the device.
 * Pairs are applied concurrently: no block may appear twice among the
 * destinations, nor as both a source and a destination.  Out-of-range ids
 * are device range errors (the pair is skipped). */
pkv_status paged_kv_copy_blocks(const pkv_cache *cache, const int32_t *src_ids,
                                const int32_t *dst_ids, int64_t n,
                                int ids_on_host, void *stream);

/* Swap blocks out to host memory: host_k[i] / host_v[i] (block_bytes =
 * 16 * num_kv_heads * head_dim * elt each, packed in list order) receive
 * block block_ids[i] of each cache.  Source: vLLM concept page
 * (compassingai.com), "15 分钟专家深入" item 1 (preempted sequences' KV
 * swapped out to CPU memory, swapped back in later).
 *   host_k, host_v  PINNED host memory (cudaHostAlloc / cudaHostRegister),
 *                 n * block_bytes each; the GPU writes them directly.
 *                 Pageable memory is rejected with PKV_ERR_ARG.
 * Ids as for paged_kv_copy_blocks; out-of-range ids are device range
 * errors (their slots are left untouched).  The host buffers are complete
 * once the stream reaches this point (e.g. after pkv_check). */
pkv_status paged_kv_swap_out(const pkv_cache *cache, const int32_t *block_ids,
                             int64_t n, int ids_on_host, void *host_k,
                             void *host_v, void *stream);

/* Swap blocks in from pinned host memory: block block_ids[i] of each cache
 * receives host_k[i] / host_v[i].  Same conventions as paged_kv_swap_out. */
pkv_status paged_kv_swap_in(const pkv_cache *cache, const int32_t *block_ids,
                            int64_t n, int ids_on_host, const void *host_k,
                            const void *host_v, void *stream);

/* Build one step's attention inputs on the GPU from a persistent request
 * state table.  Source: Model Runner V2 summary (papercache.org), Figure 2
 * and its section on GPU-native input preparation: each active request
 * keeps a stable row; every step gathers the scheduled rows, in batch
 * order, into the step's inputs, without CPU-side tensor work.
 *   idx_mapping        int32 [batch]: state row of each batch entry.
 *   num_scheduled      int32 [batch]: new tokens of each entry this step
 *                      (1 for decode, a chunk length for chunked prefill).
 *   state_block_table  int32 [num_rows, max_blocks].
 *   state_num_computed int32 [num_rows]: tokens already in the cache.
 *   state_token_ids    int32 [num_rows, max_model_len].
 *   total_tokens       host bound: capacity of the per-token outputs.
 * Outputs (device):
 *   block_tables    int32 [batch, max_blocks] = state rows, gathered;
 *   seq_lens        int32 [batch] = num_computed + num_scheduled;
 *   query_start_loc int32 [batch + 1] = exclusive prefix sum of
 *                   num_scheduled (last entry = total);
 *   positions, input_ids  int32 [total_tokens];
 *   slot_mapping    int64 [total_tokens]: the cache slot of each new token.
 * Device range errors (row out of range, position past the table or the
 * token buffer, more tokens than total_tokens, negative counts) skip the
 * affected outputs (slots become -1) and are reported by pkv_check(). */
pkv_status paged_prepare_inputs(const int32_t *idx_mapping,
                                const int32_t *num_scheduled, int32_t batch,
                                const int32_t *state_block_table,
                                int32_t max_blocks,
                                const int32_t *state_num_computed,
                                const int32_t *state_token_ids,
                                int32_t max_model_len, int32_t num_rows,
                                int64_t total_tokens, int32_t *block_tables,
                                int32_t *seq_lens, int32_t *query_start_loc,
                                int32_t *positions, int32_t *input_ids,
                                int64_t *slot_mapping, void *stream);

/* Decode attention over a paged cache, one query token per sequence.
 * Source: vLLM concept page (compassingai.com), "技术原理" pseudocode
 * (gather by page table, Q K^T / sqrt(d), softmax, times V) and its note on
 * GQA (fewer KV heads than Q heads); the gather happens inside the kernel
 * (vLLM internals, naphjohn.github.io, §4.1).
 *   q             bf16 [batch, num_heads, head_dim].
 *   block_tables  int32 [batch, max_blocks]; entry j of row b is the
 *                 physical block of tokens 16j..16j+15 of sequence b.
 *                 Only entries j < ceil(seq_lens[b] / 16) are read.
 *   seq_lens      int32 [batch] (device); 0 gives an all-zero output row.
 *   scale         multiplies Q.K (1/sqrt(head_dim) in the pages).
 *   out           bf16 [batch, num_heads, head_dim].
 *   max_seq_len   host upper bound of seq_lens (sizes the grid); a longer
 *                 sequence is clamped and reported as a range error.
 *   partition_tokens  0 = automatic (see paged_attention_partition_tokens);
 *                 otherwise a multiple of 16: every sequence is split into
 *                 partitions of that many tokens, each attended by one CTA
 *                 per kv head (by one warp when partitions hold at most 512
 *                 tokens); a second kernel merges the partitions of split
 *                 sequences with a log-sum-exp reduce.
 *   workspace     device scratch of workspace_bytes, at least
 *                 paged_attention_workspace_bytes(...) for the same
 *                 arguments; may be NULL when that function returns 0.
 * q head h reads kv head h / (num_heads / num_kv_heads).  Positions past
 * seq_lens[b] are excluded by selection, so stale bits (NaN/Inf) in unused
 * slots never reach the output.  The result is bitwise deterministic and
 * independent of where the blocks lie in the pool. */
pkv_status paged_attention_decode(const void *q, const pkv_cache *cache,
                                  const int32_t *block_tables,
                                  int32_t max_blocks, const int32_t *seq_lens,
                                  int32_t batch, int32_t num_heads,
                                  float scale, void *out, int32_t max_seq_len,
                                  int32_t partition_tokens, void *workspace,
                                  size_t workspace_bytes, void *stream);

/* One decode step in one call: each sequence's new tokens are written into
 * the cache, then every sequence is attended as by paged_attention_decode.
 * Source: vLLM concept page (compassingai.com), "15 分钟专家深入" item 2
 * (a new token's K/V goes to the block its table names, allocated on
 * demand), vLLM v0.17.1 notes (admirer.cn), "修复方案" (a freshly allocated
 * block is zeroed before attention reads it), and the "技术原理" pseudocode
 * for the attention; the fusion is this library's.
 *   k_new, v_new  bf16 [num_new_tokens, num_kv_heads, head_dim] (device,
 *                 16-byte aligned): the new tokens' K and V.
 *   new_start_loc int32 [batch + 1] (device) or NULL: sequence b's new
 *                 tokens are rows new_start_loc[b] .. new_start_loc[b+1] - 1,
 *                 at its last n_b positions L - n_b .. L - 1 (L =
 *                 seq_lens[b], which counts them).  NULL: one new token per
 *                 sequence, row b (num_new_tokens must equal batch).
 *   Other arguments, the workspace and the result as for
 *   paged_attention_decode.
 * Position t of sequence b goes to row t % 16 of block
 * block_tables[b][t / 16], E4M3-encoded as by paged_kv_write for an fp8
 * cache.  A block whose first position is one of the new tokens is a block
 * allocated for this step: its rows past L are zeroed (rows of earlier
 * positions in the block holding L - n_b are left as they are).  The cache
 * then holds the bytes that paged_kv_zero_and_write would leave with those
 * blocks listed as fresh and the new tokens' slots in slot_mapping, and the
 * output equals that of paged_attention_decode on that cache bit for bit.
 * A table entry outside the pool writes nothing for that block; a length
 * above max_seq_len or the table's width (attended clamped, as by
 * paged_attention_decode), n_b < 0, n_b > L or rows past num_new_tokens
 * write nothing for the sequence; each is reported by pkv_check().  The
 * writes are done inside the decode kernel, by the warps that read the
 * blocks, so no separate write launch precedes the attention.  Stale rows
 * of blocks the new tokens do not reach need paged_kv_zero_and_write. */
pkv_status paged_attention_decode_step(const void *q, const void *k_new,
                                       const void *v_new,
                                       const int32_t *new_start_loc,
                                       int64_t num_new_tokens,
                                       const pkv_cache *cache,
                                       const int32_t *block_tables,
                                       int32_t max_blocks,
                                       const int32_t *seq_lens, int32_t batch,
                                       int32_t num_heads, float scale,
                                       void *out, int32_t max_seq_len,
                                       int32_t partition_tokens,
                                       void *workspace, size_t workspace_bytes,
                                       void *stream);

/* Prefill / chunked-prefill attention over a paged cache: several query
 * tokens per sequence, causal within the sequence.  Source: vLLM concept
 * page (compassingai.com), "Continuous Batching" (chunked prefill: a long
 * prompt is cut into chunks that are interleaved with decode steps) and the
 * "技术原理" pseudocode (gather, Q K^T scaled, softmax, times V).
 *   q             bf16 [num_tokens, num_heads, head_dim], the query tokens
 *                 of all sequences back to back.
 *   query_start_loc int32 [batch + 1] (device): sequence b owns rows
 *                 query_start_loc[b] .. query_start_loc[b+1] - 1 of q and
 *                 out; n_b = that count (the output of
 *                 paged_prepare_inputs has this layout).
 *   seq_lens      int32 [batch] (device): c_b + n_b, where c_b tokens were
 *                 cached by earlier steps; the chunk's own K/V must already
 *                 be in the cache (paged_kv_write) as its last n_b tokens.
 *   block_tables, max_blocks: as for paged_attention_decode.
 *   scale         multiplies Q.K; must be positive (1/sqrt(head_dim)).
 *   out           bf16 [num_tokens, num_heads, head_dim].
 *   max_query_len host upper bound of every n_b (sizes the grid); rows of
 *                 tokens past it are not computed.
 * Query row i of sequence b is at position c_b + i and attends to the key
 * positions 0 .. c_b + i; a one-token chunk is a decode step.  With an
 * E4M3 cache the products run in f16 (the cache values are exact there; q
 * is rounded from bf16 to f16, so it must lie inside the f16 range) with
 * k_scale and v_scale applied as in paged_attention_decode.
 * num_heads / num_kv_heads must be at most 128.  Device-detected errors (n_b < 0, c_b < 0, a needed block id
 * outside the pool, seq_lens[b] > 16 * max_blocks) are reported by
 * pkv_check(); the affected rows are zeroed where they lie inside q. */
pkv_status paged_attention_prefill(const void *q, const pkv_cache *cache,
                                   const int32_t *block_tables,
                                   int32_t max_blocks, const int32_t *seq_lens,
                                   const int32_t *query_start_loc,
                                   int32_t batch, int32_t num_heads,
                                   int64_t num_tokens, float scale, void *out,
                                   int32_t max_query_len, void *stream);

/* Cascade (shared-prefix) decode: the same result as
 * paged_attention_decode, computed with each group's shared prefix read
 * once for all of the group's sequences.  Source: vLLM internals
 * (naphjohn.github.io), §1.1-1.2 and Figure 1 (sequences whose prompts
 * share a prefix point at the same physical blocks, refcounted) and the
 * vLLM concept page's PagedAttention pseudocode; the two-pass evaluation is
 * this library's (the pages describe the sharing, not a kernel for it).
 *   group_start   int32 [num_groups + 1] (device): group G is sequences
 *                 group_start[G] .. group_start[G+1] - 1 (consecutive rows
 *                 of q, block_tables, seq_lens); groups must not overlap
 *                 (group_start never decreases);
 *                 sequences outside every group are attended in full.
 *   prefix_len    int32 [num_groups] (device): tokens of G's shared prefix,
 *                 a multiple of 16, at most max_prefix_len; every member's
 *                 table must start with the same prefix_len / 16 block ids
 *                 and every member must be at least that long.
 *   max_group_size, max_prefix_len  host bounds (size the prefix grid).
 *   workspace     at least paged_attention_cascade_workspace_bytes(...),
 *                 256-byte aligned.
 *   Other arguments as for paged_attention_decode; scale must be positive.
 *   Both bf16 and E4M3 caches are accepted (the prefix pass of an E4M3
 *   cache runs on f16 operands, as in paged_attention_prefill).
 * Pass 1 (tensor cores) attends each group's member queries to its prefix,
 * in partitions of at least 512 tokens (longer when that still fills one
 * wave of CTAs); pass 2 attends each sequence to its own
 * tokens; a log-sum-exp merge combines the partials.  A group whose
 * members' tables or lengths break the contract is reported by pkv_check()
 * and its members are attended in full, so the output stays correct.
 * All three launches go on `stream`, in that order, with programmatic
 * dependent launch: pass 2 starts while pass 1 runs (the passes do not
 * depend on each other), and the merge waits for both.  The call keeps no
 * state between calls and shares nothing across streams. */
pkv_status paged_attention_decode_cascade(
    const void *q, const pkv_cache *cache, const int32_t *block_tables,
    int32_t max_blocks, const int32_t *seq_lens, int32_t batch,
    int32_t num_heads, const int32_t *group_start, const int32_t *prefix_len,
    int32_t num_groups, int32_t max_group_size, int32_t max_prefix_len,
    float scale, void *out, int32_t max_seq_len, int32_t partition_tokens,
    void *workspace, size_t workspace_bytes, void *stream);

/* Bytes of workspace paged_attention_decode_cascade needs (0 on invalid
 * arguments).  Host-only. */
size_t paged_attention_cascade_workspace_bytes(int32_t batch,
                                               int32_t num_heads,
                                               int32_t num_kv_heads,
                                               int32_t head_dim,
                                               int32_t max_seq_len,
                                               int32_t max_prefix_len,
                                               int32_t partition_tokens);

/* Bytes of workspace paged_attention_decode needs for these arguments
 * (0 when no sequence can be split).  Host-only; never fails. */
size_t paged_attention_workspace_bytes(int32_t batch, int32_t num_heads,
                                       int32_t num_kv_heads, int32_t head_dim,
                                       int32_t max_seq_len,
                                       int32_t partition_tokens);

/* The partition length (tokens) paged_attention_decode uses for these
 * arguments: partition_tokens itself when it is positive, otherwise the
 * automatic choice (a power-of-two multiple of 256 tokens, or the whole
 * max_seq_len when the sequences alone fill the GPU).  Returns -1 on
 * invalid arguments (partition_tokens negative or not a multiple of 16,
 * num_heads not a multiple of num_kv_heads). */
int32_t paged_attention_partition_tokens(int32_t batch, int32_t num_heads,
                                         int32_t num_kv_heads,
                                         int32_t max_seq_len,
                                         int32_t partition_tokens);

/* Size of the fixed device scratch area used by
 * paged_attention_decode_noalloc (16 MiB). */
#define PKV_NOALLOC_SCRATCH_BYTES (16u << 20)

/* paged_attention_decode for callers that cannot allocate device memory
 * (code running where cudaMalloc is forbidden or unavailable: inside an
 * allocator or allocation callback, under a device-memory budget already
 * fully handed out, or in a runtime without its own device allocator).
 * The paper has no counterpart to this entry point; it exists for such
 * callers only.
 *   Arguments are those of paged_attention_decode without the workspace:
 *   the split-KV partials go to a library-owned __device__ array of
 *   PKV_NOALLOC_SCRATCH_BYTES.  Invalid arguments get the answer
 *   paged_attention_decode would give (PKV_ERR_ARG / PKV_ERR_SHAPE, e.g.
 *   more than 65535 partitions per sequence); valid calls whose scratch
 *   need (paged_attention_workspace_bytes for the same arguments) exceeds
 *   the array return PKV_ERR_WORKSPACE without launching anything.
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) and caches it: make that first call before any
 *   stream capture.  That look-up is also when the CUDA driver loads the
 *   array (lazy module loading, the default) and takes its 16 MiB from the
 *   device, so a caller that cannot allocate later should make one call at
 *   set-up, while memory is available; after it, calls allocate nothing and
 *   the device holds the array until the process exits.  The cached
 *   address does not survive cudaDeviceReset.  All calls share the array
 *   and it keeps the last call's contents (nothing in it needs to start at
 *   zero); calls whose kernels overlap on the GPU race on it, so order them
 *   on one stream or with events. */
pkv_status paged_attention_decode_noalloc(const void *q, const pkv_cache *cache,
                                          const int32_t *block_tables,
                                          int32_t max_blocks,
                                          const int32_t *seq_lens,
                                          int32_t batch, int32_t num_heads,
                                          float scale, void *out,
                                          int32_t max_seq_len,
                                          int32_t partition_tokens,
                                          void *stream);

/* Synchronise `stream`, then read and clear the device error records of
 * the current device.  Returns PKV_OK, PKV_ERR_RANGE or PKV_ERR_TIMEOUT
 * (the first error recorded since the last check, by the GPU's global
 * timer, whichever kernel recorded it), or PKV_ERR_CUDA.  When `detail` is
 * not NULL it receives the offending index (slot, block id or sequence) of
 * that first error, or -1.  Every record is cleared, so errors recorded
 * after the first one are not reported. */
pkv_status pkv_check(void *stream, int64_t *detail);

/* Static description of a status code. */
const char *pkv_status_str(pkv_status status);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
