// pa_internal.h -- host-side interfaces between the C-ABI layer (pa_api.cu)
// and the kernel translation units.  Not installed; not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

namespace pa {

// A named NVTX range over a scope of host code (the launches of one call), so
// that a profiler groups each kernel under the library call that issued it.
// NVTX is header-only: with no tool attached a push or pop is a test of a
// function pointer and nothing else.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Bits of the device error word (read back by pa_check_device_errors).
enum : unsigned {
  DEVERR_BOUNDS = 1u,   // an index / length was out of range; work skipped
  DEVERR_TIMEOUT = 2u,  // a bounded wait gave up
};

// 8-bit cache page: the codes of 16 token rows ([16, n_kv, head_dim] bytes),
// then their fp32 scales ([16, n_kv]); a block holds block_size / 16 pages.
constexpr int kFp8PageTokens = 16;
__host__ __device__ constexpr int64_t fp8_page_bytes(int n_kv, int head_dim) {
  return (int64_t)kFp8PageTokens * n_kv * (head_dim + 4);
}
__host__ __device__ constexpr int64_t fp8_scales_offset(int n_kv, int head_dim) {
  return (int64_t)kFp8PageTokens * n_kv * head_dim;
}

// Geometry and pointers of one paged-attention call, already validated.
struct AttnArgs {
  const uint16_t* q;
  const void* k_cache;     // bf16 values, or (fp8) pages of E4M3 codes and row scales
  const void* v_cache;
  bool fp8;
  // Fused scatter (decode-only steps over the bf16 cache): the decode kernel
  // takes each decode request's new row from these and stores it to its
  // slot; all null when the scatter ran as its own kernel.
  const uint16_t* fuse_k_new;
  const uint16_t* fuse_v_new;
  const int32_t* fuse_slot_mapping;
  int32_t num_blocks;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  const int32_t* block_tables;
  int32_t max_blocks;
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  int32_t num_seqs;
  int32_t num_tokens;
  int32_t max_q_len;
  int32_t max_seq_len;
  // log2(block_size / 16): the kernels walk 16-token pages, and page j of a
  // request lives in block block_tables[j >> block_shift], 16-token half
  // (j & ((1 << block_shift) - 1)) of it
  int32_t block_shift;
  float scale;
  uint16_t* out;
  unsigned* err;  // device error word
  // The kernel launched just before on the stream is the prefill kernel
  // (which triggers its dependents at once and writes only prefill rows):
  // the decode kernel may then start on SMs it leaves free.
  bool after_prefill;
  // The caller promised that no request has exactly one query row: the
  // decode kernel is not launched, and the prefill kernel flags a request
  // with one row as a bounds error instead of leaving its row unwritten.
  bool no_decode;
};

// Workspace carve-up shared by the launchers (sizes in bytes, 256-aligned).
struct DecodeWorkspace {
  float* part_o;    // [ctas * 2, num_q_heads, head_dim]
  float* part_ml;   // [ctas * 2, num_q_heads, 2]  (running max in log2 units, sum)
  int4* seq_rec;    // [num_seqs]
};

size_t decode_workspace_bytes(int ctas, int num_seqs, int num_q_heads, int head_dim);
DecodeWorkspace decode_workspace(void* base, int ctas, int num_seqs, int num_q_heads,
                                 int head_dim);
int decode_ctas(int sm_count);

// Each launcher returns cudaSuccess or the launch error.  Unsupported shapes
// are rejected by the API layer before these are called.
bool decode_supported(int head_dim, int group, int num_kv_heads);
cudaError_t launch_decode(const AttnArgs& a, const DecodeWorkspace& ws, int ctas,
                          cudaStream_t stream);
cudaError_t launch_decode_fp8(const AttnArgs& a, const DecodeWorkspace& ws, int ctas,
                              cudaStream_t stream);
cudaError_t launch_decode_fused(const AttnArgs& a, const DecodeWorkspace& ws, int ctas,
                                cudaStream_t stream);

bool prefill_supported(int head_dim, int group, int num_kv_heads);
// How the prefill kernel splits the keys of each query-tile pair, and the
// workspace bytes the pieces take (0 when nsplit == 1).
struct PrefillPlan {
  int nsplit;
  size_t bytes;
};
PrefillPlan prefill_plan(int num_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                         int max_q_len, int max_seq_len, int sm_count, size_t max_bytes);
// The most bytes any call with at most num_tokens tokens (and these bounds)
// would use for key pieces.
size_t prefill_workspace_bound(int num_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                               int max_q_len, int max_seq_len, int sm_count);
cudaError_t launch_prefill(const AttnArgs& a, const PrefillPlan& plan, void* ws, int sm_count,
                           cudaStream_t stream);

cudaError_t launch_reshape_and_cache(const uint16_t* k, const uint16_t* v, int32_t num_tokens,
                                     uint16_t* k_cache, uint16_t* v_cache, int64_t num_slots,
                                     int32_t row_elems, const int32_t* slot_mapping,
                                     unsigned* err, cudaStream_t stream);

cudaError_t launch_reshape_and_cache_fp8(const uint16_t* k, const uint16_t* v,
                                         int32_t num_tokens, uint8_t* k_cache, uint8_t* v_cache,
                                         int64_t num_slots, int32_t num_kv_heads,
                                         int32_t head_dim, const int32_t* slot_mapping,
                                         unsigned* err, cudaStream_t stream);
cudaError_t launch_copy_blocks(uint16_t* k_cache, uint16_t* v_cache, int32_t num_blocks,
                               int64_t block_elems, const int32_t* pairs, int32_t num_pairs,
                               unsigned* err, cudaStream_t stream);

// Block swap through a device staging buffer of 2 * n * block_elems values:
// out = true packs the blocks and copies them to host_k / host_v; out = false
// copies host_k / host_v in and unpacks them into the cache.
cudaError_t launch_swap(uint16_t* k_cache, uint16_t* v_cache, int32_t num_blocks,
                        int64_t block_elems, const int32_t* ids, int32_t n, uint16_t* staging,
                        uint16_t* host_k, uint16_t* host_v, bool out, unsigned* err,
                        cudaStream_t stream);

cudaError_t launch_wait_timeout_selftest(unsigned long long limit_ns, unsigned* err,
                                         cudaStream_t stream);

// Error reporting of the C ABI (sets the message pa_get_last_error returns)
// and the per-device state lookup, for the parts of the ABI outside pa_api.cu.
int api_fail(int status, const char* fmt, ...);
int api_warm_device();

}  // namespace pa
