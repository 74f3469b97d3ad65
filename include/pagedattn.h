/*
 * pagedattn.h -- C ABI of libpagedattn.so: attention over a paged KV cache on
 * NVIDIA GB300 (sm_103a).
 *
 * The cache is a pool of fixed-size physical blocks; each request reaches its
 * tokens through a Block Table row that maps logical block b (tokens
 * b*block_size .. b*block_size + block_size - 1) to a physical block id
 * ("PagedAttention 显存分页与连续批处理(Continuous Batching)实战",
 * "PagedAttention 核心机理" part 1; "连续批处理：推理吞吐的范式革命",
 * section 2.2).
 *
 * Conventions for every call:
 *  - pa_bf16 is a raw bfloat16 bit pattern.  Every array pointer is a DEVICE
 *    pointer owned by the caller, C-contiguous, 16-byte aligned; the library
 *    never frees or keeps it.
 *  - KV cache layout: [num_blocks, block_size, num_kv_heads, head_dim].
 *  - Calls are asynchronous on `stream` (0 = legacy default stream).  The
 *    returned status covers argument checks and launch errors only.  Index
 *    errors found on the device (a slot, block id or length out of range)
 *    make the kernel skip that work item and set a device error word, which
 *    pa_check_device_errors() reads back.
 *  - The library allocates no device memory at run time.  pa_paged_attention
 *    takes a caller-provided workspace of pa_workspace_size() bytes (the
 *    allocation-free variant at the end of this header uses a fixed array
 *    built into the library instead).
 *  - Supported: block_size 16 or 32 for attention (the cache writes, block
 *    copies and swaps take any positive block_size); head_dim 64 or 128;
 *    num_q_heads a multiple of num_kv_heads with group size num_q_heads /
 *    num_kv_heads in {1, 2, 4, 8}; num_kv_heads in {1, 2, 4, 8}.  Anything
 *    else returns PA_ERR_UNSUPPORTED.
 *  - On error the call returns a non-zero status and pa_get_last_error()
 *    returns a message (per thread, valid until the next call on the thread).
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t pa_bf16;

enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,   /* bad size, null or misaligned pointer         */
  PA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (shape, block size) */
  PA_ERR_CUDA = 3,          /* a CUDA runtime call or a launch failed       */
  PA_ERR_DEVICE_BOUNDS = 4, /* a kernel found an index out of range         */
  PA_ERR_TIMEOUT = 5,       /* a kernel gave up a bounded wait              */
  PA_ERR_WORKSPACE = 6      /* workspace missing, too small or misaligned   */
};

/* Library version, major * 10000 + minor * 100 + patch. */
int pa_version(void);

/* Message for the last non-zero status returned on this thread. */
const char *pa_get_last_error(void);

/*
 * Slot scatter.  For each new token t in [0, num_tokens) with
 * s = slot_mapping[t] >= 0, copy k[t, :, :] to k_cache[s / block_size,
 * s % block_size, :, :] and v[t] to v_cache likewise (a bit copy).  A negative
 * slot skips the token.  Slots must be distinct within one call.  This is how
 * a step's new tokens reach their on-demand allocated physical slots
 * ("PagedAttention 显存分页与连续批处理实战", comparison table: blocks are
 * allocated on demand as a block fills; TypeScript Block Manager appendToken).
 *
 *   k, v          [num_tokens, num_kv_heads, head_dim]  bf16, read
 *   k_cache, v_cache  [num_blocks, block_size, num_kv_heads, head_dim], written
 *   slot_mapping  [num_tokens] int32, read
 * A slot >= num_blocks * block_size is skipped and flags PA_ERR_DEVICE_BOUNDS.
 */
int pa_reshape_and_cache(const pa_bf16 *k, const pa_bf16 *v, int32_t num_tokens,
                         pa_bf16 *k_cache, pa_bf16 *v_cache, int32_t num_blocks,
                         int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                         const int32_t *slot_mapping, cudaStream_t stream);

/*
 * Workspace bytes for pa_paged_attention on the current device: enough for
 * every call whose num_seqs, num_tokens, max_q_len and max_seq_len are at
 * most these (so one buffer sized for a serving loop's largest step serves
 * all its steps).  The size depends only on the arguments and the device's SM
 * count.  A call needs at least its split-KV decode scratch; the prefill
 * kernel splits keys only as far as the rest of the workspace allows, so a
 * smaller workspace is never an error past that, only fewer key pieces.
 * Returns 0 if an argument is invalid.
 */
size_t pa_workspace_size(int32_t num_seqs, int32_t num_tokens, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t max_q_len,
                         int32_t max_seq_len);

/*
 * Number of pieces the tensor-core prefill kernel splits each request's keys
 * into for a pa_paged_attention call with these sizes on the current device
 * (informational; 1 means no split).  With more than one piece, every prefill
 * row is written as per-piece partial results into the workspace and a second
 * kernel combines them with log-sum-exp weights, so the call launches one
 * kernel more.  Returns 0 if an argument is invalid.
 */
int pa_prefill_splits(int32_t num_tokens, int32_t num_q_heads, int32_t num_kv_heads,
                      int32_t head_dim, int32_t max_q_len, int32_t max_seq_len);

/*
 * Causal, GQA-aware, variable-length attention over the paged cache
 * ("连续批处理：推理吞吐的范式革命", section 4.1: walk the request's Block
 * Table, score q.k scaled, softmax, weighted sum of v, normalise; chunked
 * prefill mixes prompt slices and decode tokens in one batch:
 * "PagedAttention 显存分页与连续批处理实战", Chunked Prefill section).
 *
 * Request s owns query tokens query_start_loc[s] .. query_start_loc[s+1]-1
 * (q_len = their count, 0 allowed) and seq_lens[s] cached tokens, which
 * include those q_len tokens (write them with pa_reshape_and_cache first).
 * Query row i of request s is at position p = seq_lens[s] - q_len + i and
 * attends to positions 0..p; q head h reads kv head h / (num_q_heads /
 * num_kv_heads):
 *   out[t, h, :] = sum_j softmax_j(scale * q[t,h,:] . K[s,j,g,:]) V[s,j,g,:]
 * where K[s, j] = k_cache[block_tables[s, j / block_size], j % block_size].
 *
 *   q             [num_tokens, num_q_heads, head_dim] bf16, read
 *   k_cache, v_cache  [num_blocks, block_size, num_kv_heads, head_dim], read
 *   block_tables  [num_seqs, max_blocks] int32, read; only entries
 *                 0 .. ceil(seq_lens[s] / block_size) - 1 are read
 *   seq_lens      [num_seqs] int32, read
 *   query_start_loc [num_seqs + 1] int32, read, non-decreasing, last entry
 *                 <= num_tokens
 *   max_q_len, max_seq_len  host-side upper bounds of q_len and seq_lens
 *                 (size the launch; a request beyond them flags
 *                 PA_ERR_DEVICE_BOUNDS and its rows are not written)
 *   out           [num_tokens, num_q_heads, head_dim] bf16, written for every
 *                 token that belongs to a request; other rows are untouched
 *   workspace     device buffer of >= pa_workspace_size(...) bytes,
 *                 256-byte aligned; its contents on entry do not matter and
 *                 it must not be used by another call running concurrently
 * Accumulation is fp32; out is rounded to nearest even.  Rows with q_len == 1
 * run on the split-KV decode kernel, rows of requests with q_len >= 2 on the
 * tensor-core prefill kernel.  Where p . V runs on the tensor cores (prefill
 * rows, and decode rows when num_q_heads / num_kv_heads is 8) the softmax
 * weights enter it rounded to bf16, and the normalising sum adds the same
 * rounded weights, so every output row is an exact convex combination of V
 * rows with those weights.  A request with q_len > seq_len, seq_len >
 * max_blocks * block_size or a block id outside [0, num_blocks) flags
 * PA_ERR_DEVICE_BOUNDS.
 */
int pa_paged_attention(const pa_bf16 *q, const pa_bf16 *k_cache, const pa_bf16 *v_cache,
                       int32_t num_blocks, int32_t block_size, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_dim, const int32_t *block_tables,
                       int32_t max_blocks, const int32_t *seq_lens,
                       const int32_t *query_start_loc, int32_t num_seqs, int32_t num_tokens,
                       int32_t max_q_len, int32_t max_seq_len, float scale, pa_bf16 *out,
                       void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * pa_paged_attention with a host-side lower bound on the requests' query
 * rows as well: min_q_len <= q_len for every request with at least one row
 * (0 or 1: no bound).  With min_q_len >= 2 the call has no decode rows, so
 * only the prefill kernel runs (no empty decode launch after it); a request
 * with exactly one row then flags PA_ERR_DEVICE_BOUNDS and its row is not
 * written.  min_q_len > max_q_len is PA_ERR_INVALID_ARG.  Everything else is
 * pa_paged_attention.
 */
int pa_paged_attention_qrange(const pa_bf16 *q, const pa_bf16 *k_cache, const pa_bf16 *v_cache,
                              int32_t num_blocks, int32_t block_size, int32_t num_q_heads,
                              int32_t num_kv_heads, int32_t head_dim, const int32_t *block_tables,
                              int32_t max_blocks, const int32_t *seq_lens,
                              const int32_t *query_start_loc, int32_t num_seqs,
                              int32_t num_tokens, int32_t min_q_len, int32_t max_q_len,
                              int32_t max_seq_len, float scale, pa_bf16 *out, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/*
 * One decode step in one kernel: pa_reshape_and_cache followed by
 * pa_paged_attention, for a step whose requests all have q_len <= 1 (every
 * row a decode row; max_q_len is 1).  The decode kernel takes each request's
 * new key and value rows (token t = query_start_loc[s]) from k_new / v_new
 * straight into its copy of the request's last page, and stores them to
 * slot_mapping[t] from there, so no separate scatter runs and the new rows
 * are read from HBM once.  Precondition: slot_mapping[t] is the slot of the
 * request's position seq_lens[s] - 1 (its block table entry), or negative (the
 * row is not written and the cache's row is read, as with a separate
 * scatter); any other slot flags PA_ERR_DEVICE_BOUNDS.  Tokens outside every
 * request are not written.  bf16 cache only; arguments, workspace and errors
 * otherwise as pa_reshape_and_cache and pa_paged_attention.
 */
int pa_decode_step(const pa_bf16 *q, const pa_bf16 *k_new, const pa_bf16 *v_new,
                   pa_bf16 *k_cache, pa_bf16 *v_cache, int32_t num_blocks, int32_t block_size,
                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                   const int32_t *block_tables, int32_t max_blocks, const int32_t *seq_lens,
                   const int32_t *query_start_loc, int32_t num_seqs, int32_t num_tokens,
                   int32_t max_seq_len, const int32_t *slot_mapping, float scale, pa_bf16 *out,
                   void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * One serving step's slot scatter and attention, for any mix of decode rows
 * and chunked-prefill rows ("PagedAttention 显存分页与连续批处理(Continuous
 * Batching)实战", Chunked Prefill section: each iteration mixes prompt
 * slices with the running decodes), without a separate scatter kernel:
 * pa_reshape_and_cache followed by pa_paged_attention, in the attention
 * kernels themselves.  The tensor-core kernel takes a prefill request's new
 * key and value rows (tokens query_start_loc[s] ..) from k_new / v_new rather
 * than from the cache, and stores them to their slots while it runs; the
 * decode kernel does the same for decode rows (as pa_decode_step).  Outputs
 * and the cache afterwards are bit-identical to the two separate calls.
 * Precondition: slot_mapping[t] of query row i of request s is the slot of
 * its position seq_lens[s] - q_len + i (its block table entry).  A prefill
 * row with any other slot is not stored and flags PA_ERR_DEVICE_BOUNDS (its
 * attention still uses its k_new / v_new row); a decode row follows
 * pa_decode_step (a negative slot reads the cache's row, any other slot
 * flags).  Tokens outside every request are not written.  bf16 cache only;
 * arguments, workspace and errors otherwise as pa_reshape_and_cache and
 * pa_paged_attention.  Cost: every later query tile of a chunk reads the
 * chunk's new rows from k_new / v_new, and on a GB300 that measured slower
 * than one scatter launch (a 512-token chunk with 128 decode rows: 150 us
 * against 141 us for the two calls), so the step graph does not use it.
 */
int pa_paged_attention_step(const pa_bf16 *q, const pa_bf16 *k_new, const pa_bf16 *v_new,
                            pa_bf16 *k_cache, pa_bf16 *v_cache, int32_t num_blocks,
                            int32_t block_size, int32_t num_q_heads, int32_t num_kv_heads,
                            int32_t head_dim, const int32_t *block_tables, int32_t max_blocks,
                            const int32_t *seq_lens, const int32_t *query_start_loc,
                            int32_t num_seqs, int32_t num_tokens, int32_t max_q_len,
                            int32_t max_seq_len, const int32_t *slot_mapping, float scale,
                            pa_bf16 *out, void *workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/*
 * Copy-on-write block copy: for each pair i, physical block
 * src_dst_pairs[2i+1] of both caches becomes a bit copy of block
 * src_dst_pairs[2i] ("PagedAttention 显存分页与连续批处理实战", comparison
 * table, Copy-on-Write sharing of prompt blocks; "连续批处理：推理吞吐的范式革命",
 * section 4.2, prefix sharing).  Destinations must be distinct and no
 * destination may be a source of the same call (pairs are then independent
 * and run in parallel).  A pair whose source is -1 is padding and is skipped
 * (a fixed-size pair list, as a captured step graph uses); any other id
 * outside [0, num_blocks) skips the pair and flags PA_ERR_DEVICE_BOUNDS.
 *
 *   src_dst_pairs [num_pairs, 2] int32 device array, read
 */
int pa_copy_blocks(pa_bf16 *k_cache, pa_bf16 *v_cache, int32_t num_blocks, int32_t block_size,
                   int32_t num_kv_heads, int32_t head_dim, const int32_t *src_dst_pairs,
                   int32_t num_pairs, cudaStream_t stream);

/*
 * Block swap for preemption by swapping instead of recomputing
 * ("连续批处理：推理吞吐的范式革命", section 3.3: a preempted request's KV
 * cache moves to CPU memory and comes back without recomputation;
 * "vLLM中的PagedAttention机制与显存优化实践", section 2.1: swap is
 * block-grained and runs asynchronously on its own CUDA streams, so pass a
 * side stream to overlap it with attention on another).
 *
 * pa_swap_out copies blocks block_ids[0..n) of both caches to the host:
 * host_k[i] and host_v[i] ([n, block_size, num_kv_heads, head_dim] bf16
 * each, in list order) become bit copies of block block_ids[i].  A kernel
 * first packs the blocks into `staging`, then two cudaMemcpyAsync calls copy
 * it to the host (use pinned host memory for the copies to be asynchronous).
 * pa_swap_in is the reverse: block block_ids[i] of both caches becomes a bit
 * copy of host_k[i] / host_v[i]; ids must then be distinct.
 *
 *   block_ids  [n] int32 device array, read; an id outside [0, num_blocks)
 *              skips that block and flags PA_ERR_DEVICE_BOUNDS
 *   staging    device buffer of pa_swap_staging_bytes(n, ...) bytes,
 *              16-byte aligned, owned by the caller, not used by another call
 *              meanwhile; its contents on entry do not matter
 *   host_k/v   host buffers of n * block_size * num_kv_heads * head_dim bf16
 * Asynchronous on `stream`: host_k / host_v hold the blocks after the stream
 * has synchronised (swap-out), and may be reused once it has (swap-in).
 */
size_t pa_swap_staging_bytes(int32_t n, int32_t block_size, int32_t num_kv_heads,
                             int32_t head_dim);
int pa_swap_out(const pa_bf16 *k_cache, const pa_bf16 *v_cache, int32_t num_blocks,
                int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                const int32_t *block_ids, int32_t n, pa_bf16 *staging, pa_bf16 *host_k,
                pa_bf16 *host_v, cudaStream_t stream);
int pa_swap_in(pa_bf16 *k_cache, pa_bf16 *v_cache, int32_t num_blocks, int32_t block_size,
               int32_t num_kv_heads, int32_t head_dim, const int32_t *block_ids, int32_t n,
               pa_bf16 *staging, const pa_bf16 *host_k, const pa_bf16 *host_v,
               cudaStream_t stream);

/*
 * 8-bit KV cache.  The pages have no counterpart: every cache they describe
 * holds the model's own precision.  This variant stores FP8 E4M3 codes (1
 * sign, 4 exponent bits of bias 7, 3 mantissa bits, no infinities, largest
 * magnitude 448) and one fp32 scale per cached (token, kv head) row, so
 * decode attention reads about half the bytes.  Each 16-token page of a
 * block holds its codes, then their scales, so one copy brings both:
 *
 *   page               [16, num_kv_heads, head_dim] uint8 codes, then
 *                      [16, num_kv_heads] fp32 scales:
 *                      pa_fp8_page_bytes(num_kv_heads, head_dim)
 *                      = 16 * num_kv_heads * (head_dim + 4) bytes
 *   k_cache, v_cache   [num_blocks, block_size / 16] pages
 *
 * The slot of token row r of page p of block b is b * block_size + 16 p + r.
 * block_size is a multiple of 16 (16 or 32 for attention).
 *
 * A row x (head_dim bf16 values) is stored as scale = max |x| / 448 (1 when
 * the row is all zero) and codes e4m3(x_c / scale), rounding to nearest with
 * ties to even and saturating; both divisions are fp32, round to nearest.
 * Attention uses code * scale in place of each cached value.  The decode
 * kernel (q_len 1) runs q . k and p . V on the tensor cores with
 * q * scale * log2(e) and p * value scale * 2^9 rounded to f16 (codes
 * convert to f16 exactly; the 2^9 is removed exactly).  The prefill kernel
 * (q_len >= 2, the chunked-prefill rows) turns each cached row into
 * f16(code * f16(scale)) in shared memory (codes exact in f16, one rounding
 * of the scale and one of the product), and runs
 * its tcgen05 products on f16 operands: q * scale * log2(e) and p rounded
 * to f16.  head_dim is 64 or 128; the same shapes as the bf16 cache.
 *
 * pa_fp8_page_bytes: the page size above (0 for a non-positive argument).
 *
 * pa_reshape_and_cache_fp8: pa_reshape_and_cache, quantising each new row
 * (codes and scale written to the new token's slot).  Alignment: k, v and
 * both caches 16 bytes, slot_mapping 4 bytes.
 */
size_t pa_fp8_page_bytes(int32_t num_kv_heads, int32_t head_dim);

int pa_reshape_and_cache_fp8(const pa_bf16 *k, const pa_bf16 *v, int32_t num_tokens,
                             uint8_t *k_cache, uint8_t *v_cache, int32_t num_blocks,
                             int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                             const int32_t *slot_mapping, cudaStream_t stream);

/*
 * pa_paged_attention over the 8-bit cache (same arguments, meaning, errors
 * and workspace as pa_paged_attention, with the caches in the page format
 * above).  Decode and prefill rows, mixed in one call, as
 * pa_paged_attention (see above for the arithmetic).
 */
int pa_paged_attention_fp8(const pa_bf16 *q, const uint8_t *k_cache, const uint8_t *v_cache,
                           int32_t num_blocks, int32_t block_size, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim, const int32_t *block_tables,
                           int32_t max_blocks, const int32_t *seq_lens,
                           const int32_t *query_start_loc, int32_t num_seqs, int32_t num_tokens,
                           int32_t max_q_len, int32_t max_seq_len, float scale, pa_bf16 *out,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * pa_copy_blocks over the 8-bit cache: each pair copies the destination
 * block's pages (codes and scales) from the source block (same pair rules,
 * padding and errors).  Both caches 16-byte aligned.
 */
int pa_copy_blocks_fp8(uint8_t *k_cache, uint8_t *v_cache, int32_t num_blocks,
                       int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                       const int32_t *src_dst_pairs, int32_t num_pairs, cudaStream_t stream);

/*
 * Synchronises `stream`, then reads and clears the device error word that
 * the kernels of this library set on the current device.  Returns PA_OK,
 * PA_ERR_DEVICE_BOUNDS, PA_ERR_TIMEOUT or PA_ERR_CUDA.
 */
int pa_check_device_errors(cudaStream_t stream);

/*
 * Failure-detection self-test.  Every wait inside the library's kernels (on
 * a copy landing, on a tensor-core product, on another warp's hand-off) is
 * bounded: past its limit (2 s) the kernel sets PA_ERR_TIMEOUT's bit in the
 * device error word, stops waiting and returns, so the context stays usable.
 * This call runs that same wait, with limit_ns (at most 1 s), on a barrier
 * that nothing completes; pa_check_device_errors afterwards returns
 * PA_ERR_TIMEOUT.  It faults nothing and hangs nothing.  limit_ns of 0 or
 * above 1 s is PA_ERR_INVALID_ARG.
 */
int pa_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream);

/*
 * Allocation-free form of pa_paged_attention.  The pages have no counterpart
 * for it; it exists for callers that cannot allocate device memory where they
 * run attention: code running while a stream is captured into a CUDA graph,
 * plugins whose host owns all device memory, serving loops that must not
 * allocate after start-up.
 *
 * Same arguments, layout and results as pa_paged_attention, minus the
 * workspace: scratch comes from an array built into the library
 * (pa_noalloc_scratch_bytes() bytes, 8 MiB, held on every device that loads
 * the library until the process exits).  A call needing more scratch than
 * that (see pa_workspace_size) returns PA_ERR_WORKSPACE.  Allocates nothing.
 * The first call on a device looks up the array's device address and keeps
 * it for the life of the process: make that first call before any stream
 * capture (a call with num_seqs = 0 and a valid cache geometry does only
 * this set-up and launches nothing), and do not use the library across a
 * cudaDeviceReset, after which the kept address is stale.  Calls share the
 * array, so calls whose executions overlap on the GPU race and must be
 * serialised by the caller.
 */
size_t pa_noalloc_scratch_bytes(void);

int pa_paged_attention_noalloc(const pa_bf16 *q, const pa_bf16 *k_cache,
                               const pa_bf16 *v_cache, int32_t num_blocks, int32_t block_size,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                               const int32_t *block_tables, int32_t max_blocks,
                               const int32_t *seq_lens, const int32_t *query_start_loc,
                               int32_t num_seqs, int32_t num_tokens, int32_t max_q_len,
                               int32_t max_seq_len, float scale, pa_bf16 *out,
                               cudaStream_t stream);

/*
 * One serving step captured as a CUDA graph: block copies (pa_copy_blocks),
 * slot scatter (pa_reshape_and_cache) and attention (pa_paged_attention) of
 * the iteration-level schedule ("PagedAttention 显存分页与连续批处理
 * (Continuous Batching)实战", continuous batching and Chunked Prefill
 * sections: every step runs the same sequence of operations over whichever
 * requests the scheduler picked), launched with one call instead of three to
 * five kernel launches.  The pages have no counterpart for the graph itself.
 *
 * The graph is built once over fixed device buffers sized for the largest
 * step (the pa_step_buffers maxima); before each launch the caller writes the
 * step's inputs into those buffers, padded to the maxima:
 *   - tokens t >= the step's count: slot_mapping[t] = -1 (not written);
 *   - sequences s >= the step's count: query_start_loc[s + 1] =
 *     query_start_loc[s] (no rows) and seq_lens[s] = 0;
 *   - copy pairs i >= the step's count: copy_pairs[2i] = -1 (skipped).
 * A step's sizes must stay within the maxima (max_q_len and max_seq_len
 * included: a request beyond them flags PA_ERR_DEVICE_BOUNDS at run time).
 * The graph runs scatter + attention as pa_decode_step (max_q_len 1: one
 * kernel, whose slot precondition applies) or as pa_reshape_and_cache then
 * pa_paged_attention.
 * Rows of out that belong to no request are left as they were.
 *
 * If host_meta is not NULL, every launch first copies meta_bytes from
 * host_meta (pinned host memory) to dev_meta, so that the step's inputs (the
 * integer arrays, and q / k_new / v_new too if the caller places them there)
 * can live in one region of dev_meta and reach the GPU in one copy inside the
 * graph.  If host_out is not NULL, every launch ends by copying the first
 * out_copy_bytes of out to host_out (pinned host memory).  The copies read
 * and write host memory when the launch executes on the GPU, not when it is
 * issued: do not touch those buffers until then (for example, alternate two
 * graphs over two sets of host buffers).
 *
 * Buffers stay owned by the caller and must outlive the graph.  Launches of
 * one graph, and of graphs sharing buffers, must not overlap on the GPU.
 */
typedef struct pa_step_buffers {
  pa_bf16 *k_cache, *v_cache;   /* [num_blocks, block_size, num_kv_heads, head_dim] */
  int32_t num_blocks, block_size, num_q_heads, num_kv_heads, head_dim;
  int32_t max_tokens;           /* rows of q, k_new, v_new, out, slot_mapping */
  int32_t max_seqs;             /* rows of block_tables and seq_lens (+1: query_start_loc) */
  int32_t max_blocks;           /* columns of block_tables */
  int32_t max_pairs;            /* rows of copy_pairs; 0: the graph has no copy step */
  int32_t max_q_len, max_seq_len;
  float scale;
  const pa_bf16 *q;             /* [max_tokens, num_q_heads, head_dim] */
  const pa_bf16 *k_new, *v_new; /* [max_tokens, num_kv_heads, head_dim] */
  pa_bf16 *out;                 /* [max_tokens, num_q_heads, head_dim] */
  const int32_t *slot_mapping;  /* [max_tokens] */
  const int32_t *block_tables;  /* [max_seqs, max_blocks] */
  const int32_t *seq_lens;      /* [max_seqs] */
  const int32_t *query_start_loc; /* [max_seqs + 1] */
  const int32_t *copy_pairs;    /* [max_pairs, 2] or NULL when max_pairs == 0 */
  void *workspace;              /* >= pa_workspace_size(max_seqs, max_tokens, ...) bytes */
  size_t workspace_bytes;
  const void *host_meta;        /* optional pinned host source of a per-launch copy */
  void *dev_meta;
  size_t meta_bytes;
  void *host_out;               /* optional pinned host destination of out */
  size_t out_copy_bytes;        /* <= max_tokens * num_q_heads * head_dim * 2 */
} pa_step_buffers;

typedef struct pa_step_graph pa_step_graph;

/*
 * Validates the buffers (the same checks as the three calls), captures the
 * step on the current device and instantiates it.  On success *graph owns
 * the graph; destroy it with pa_step_graph_destroy.  Nothing runs on the GPU.
 */
int pa_step_graph_create(const pa_step_buffers *buffers, pa_step_graph **graph);

/* Launches the captured step on `stream` (asynchronous). */
int pa_step_graph_launch(pa_step_graph *graph, cudaStream_t stream);

/* Frees the graph (NULL is a no-op).  Launches in flight may finish first. */
int pa_step_graph_destroy(pa_step_graph *graph);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
