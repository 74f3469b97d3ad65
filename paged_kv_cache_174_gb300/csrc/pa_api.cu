// pa_api.cu -- the C ABI of libpagedattn (declared in include/pagedattn.h):
// argument validation, error reporting, workspace carving and dispatch to
// the kernels.  No device memory is allocated here.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "pagedattn.h"
#include "pa_internal.h"

namespace {

// Device error word, one per device that loads the library.  Kernels OR
// pa::DEVERR_* bits into it; pa_check_device_errors reads and clears it.
__device__ unsigned g_pa_error_word = 0;

thread_local std::string t_last_error;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned* g_err_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};

int fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Per-device state: address of the error word and the SM count.
int device_state(unsigned** err, int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PA_ERR_UNSUPPORTED, "device id %d", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_err_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_pa_error_word);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(error word)");
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
    g_err_ptr[dev] = static_cast<unsigned*>(p);
    g_sm_count[dev] = n;
  }
  if (err) *err = g_err_ptr[dev];
  if (sms) *sms = g_sm_count[dev];
  return PA_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_cache_geometry(int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                         int32_t head_dim) {
  if (num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return fail(PA_ERR_INVALID_ARG,
                "cache geometry must be positive (num_blocks=%d block_size=%d "
                "num_kv_heads=%d head_dim=%d)",
                num_blocks, block_size, num_kv_heads, head_dim);
  if (((int64_t)num_kv_heads * head_dim * 2) % 16 != 0)
    return fail(PA_ERR_UNSUPPORTED, "a token row (num_kv_heads*head_dim*2 bytes) must be a "
                                    "multiple of 16 bytes");
  return PA_OK;
}

}  // namespace

namespace pa {

int api_fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return status;
}

int api_warm_device() { return device_state(nullptr, nullptr); }

}  // namespace pa

extern "C" {

int pa_version(void) { return 200; }  // 0.2.0: the 8-bit cache in pages of codes, then scales

const char* pa_get_last_error(void) { return t_last_error.c_str(); }

int pa_reshape_and_cache(const pa_bf16* k, const pa_bf16* v, int32_t num_tokens,
                         pa_bf16* k_cache, pa_bf16* v_cache, int32_t num_blocks,
                         int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                         const int32_t* slot_mapping, cudaStream_t stream) {
  if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_tokens %d < 0", num_tokens);
  int st = check_cache_geometry(num_blocks, block_size, num_kv_heads, head_dim);
  if (st) return st;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping)
    return fail(PA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 4))
    return fail(PA_ERR_INVALID_ARG, "bf16 arrays must be 16-byte aligned, slot_mapping 4-byte");
  unsigned* err = nullptr;
  st = device_state(&err, nullptr);
  if (st) return st;
  pa::NvtxRange range("pa_reshape_and_cache (slot scatter)");
  cudaError_t e = pa::launch_reshape_and_cache(
      k, v, num_tokens, k_cache, v_cache, (int64_t)num_blocks * block_size,
      num_kv_heads * head_dim, slot_mapping, err, stream);
  if (e != cudaSuccess) return cuda_fail(e, "reshape_and_cache launch");
  return PA_OK;
}

int pa_copy_blocks(pa_bf16* k_cache, pa_bf16* v_cache, int32_t num_blocks, int32_t block_size,
                   int32_t num_kv_heads, int32_t head_dim, const int32_t* src_dst_pairs,
                   int32_t num_pairs, cudaStream_t stream) {
  if (num_pairs < 0) return fail(PA_ERR_INVALID_ARG, "num_pairs %d < 0", num_pairs);
  int st = check_cache_geometry(num_blocks, block_size, num_kv_heads, head_dim);
  if (st) return st;
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !src_dst_pairs)
    return fail(PA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(src_dst_pairs, 4))
    return fail(PA_ERR_INVALID_ARG, "caches must be 16-byte aligned, pairs 4-byte");
  if (num_pairs > 0x7fffffff / 2) return fail(PA_ERR_INVALID_ARG, "too many pairs");
  unsigned* err = nullptr;
  st = device_state(&err, nullptr);
  if (st) return st;
  pa::NvtxRange range("pa_copy_blocks (copy-on-write)");
  cudaError_t e = pa::launch_copy_blocks(k_cache, v_cache, num_blocks,
                                         (int64_t)block_size * num_kv_heads * head_dim,
                                         src_dst_pairs, num_pairs, err, stream);
  if (e != cudaSuccess) return cuda_fail(e, "copy_blocks launch");
  return PA_OK;
}

size_t pa_fp8_page_bytes(int32_t num_kv_heads, int32_t head_dim) {
  if (num_kv_heads <= 0 || head_dim <= 0) return 0;
  return (size_t)pa::fp8_page_bytes(num_kv_heads, head_dim);
}

int pa_reshape_and_cache_fp8(const pa_bf16* k, const pa_bf16* v, int32_t num_tokens,
                             uint8_t* k_cache, uint8_t* v_cache, int32_t num_blocks,
                             int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                             const int32_t* slot_mapping, cudaStream_t stream) {
  if (num_tokens < 0) return fail(PA_ERR_INVALID_ARG, "num_tokens %d < 0", num_tokens);
  int st = check_cache_geometry(num_blocks, block_size, num_kv_heads, head_dim);
  if (st) return st;
  if (head_dim != 64 && head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "8-bit cache with head_dim %d (64 or 128)", head_dim);
  if (block_size % pa::kFp8PageTokens)
    return fail(PA_ERR_UNSUPPORTED, "8-bit cache with block_size %d (a multiple of 16)",
                block_size);
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping)
    return fail(PA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 4))
    return fail(PA_ERR_INVALID_ARG, "k, v and the caches must be 16-byte aligned");
  unsigned* err = nullptr;
  st = device_state(&err, nullptr);
  if (st) return st;
  pa::NvtxRange range("pa_reshape_and_cache_fp8 (quantising slot scatter)");
  cudaError_t e = pa::launch_reshape_and_cache_fp8(
      k, v, num_tokens, k_cache, v_cache, (int64_t)num_blocks * block_size, num_kv_heads,
      head_dim, slot_mapping, err, stream);
  if (e != cudaSuccess) return cuda_fail(e, "reshape_and_cache_fp8 launch");
  return PA_OK;
}

int pa_copy_blocks_fp8(uint8_t* k_cache, uint8_t* v_cache, int32_t num_blocks,
                       int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                       const int32_t* src_dst_pairs, int32_t num_pairs, cudaStream_t stream) {
  if (num_pairs < 0) return fail(PA_ERR_INVALID_ARG, "num_pairs %d < 0", num_pairs);
  int st = check_cache_geometry(num_blocks, block_size, num_kv_heads, head_dim);
  if (st) return st;
  if (block_size % pa::kFp8PageTokens)
    return fail(PA_ERR_UNSUPPORTED, "8-bit cache with block_size %d (a multiple of 16)",
                block_size);
  // whole 16-token pages, codes and scales together (a multiple of 16 bytes)
  const int64_t block_bytes =
      (int64_t)(block_size / pa::kFp8PageTokens) * pa::fp8_page_bytes(num_kv_heads, head_dim);
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !src_dst_pairs)
    return fail(PA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(src_dst_pairs, 4))
    return fail(PA_ERR_INVALID_ARG, "the caches must be 16-byte aligned, pairs 4-byte");
  if (num_pairs > 0x7fffffff / 2) return fail(PA_ERR_INVALID_ARG, "too many pairs");
  unsigned* err = nullptr;
  st = device_state(&err, nullptr);
  if (st) return st;
  pa::NvtxRange range("pa_copy_blocks_fp8 (copy-on-write)");
  // the copy kernel moves 16-byte vectors; sizes are given in 2-byte units
  cudaError_t e = pa::launch_copy_blocks(reinterpret_cast<uint16_t*>(k_cache),
                                         reinterpret_cast<uint16_t*>(v_cache), num_blocks,
                                         block_bytes / 2, src_dst_pairs, num_pairs, err, stream);
  if (e != cudaSuccess) return cuda_fail(e, "copy_blocks_fp8 launch");
  return PA_OK;
}

size_t pa_swap_staging_bytes(int32_t n, int32_t block_size, int32_t num_kv_heads,
                             int32_t head_dim) {
  if (n < 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
  return (size_t)2 * n * block_size * num_kv_heads * head_dim * sizeof(pa_bf16);
}

}  // extern "C"

namespace {

int swap_blocks(pa_bf16* k_cache, pa_bf16* v_cache, int32_t num_blocks, int32_t block_size,
                int32_t num_kv_heads, int32_t head_dim, const int32_t* block_ids, int32_t n,
                pa_bf16* staging, pa_bf16* host_k, pa_bf16* host_v, bool out,
                cudaStream_t stream) {
  if (n < 0) return fail(PA_ERR_INVALID_ARG, "n %d < 0", n);
  int st = check_cache_geometry(num_blocks, block_size, num_kv_heads, head_dim);
  if (st) return st;
  if (n == 0) return PA_OK;
  if (!k_cache || !v_cache || !block_ids || !staging || !host_k || !host_v)
    return fail(PA_ERR_INVALID_ARG, "null pointer argument");
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(staging, 16) ||
      !aligned(block_ids, 4))
    return fail(PA_ERR_INVALID_ARG, "caches and staging must be 16-byte aligned, ids 4-byte");
  unsigned* err = nullptr;
  st = device_state(&err, nullptr);
  if (st) return st;
  pa::NvtxRange range(out ? "pa_swap_out" : "pa_swap_in");
  cudaError_t e = pa::launch_swap(k_cache, v_cache, num_blocks,
                                  (int64_t)block_size * num_kv_heads * head_dim, block_ids, n,
                                  staging, host_k, host_v, out, err, stream);
  if (e != cudaSuccess) return cuda_fail(e, out ? "swap_out" : "swap_in");
  return PA_OK;
}

}  // namespace

extern "C" {

int pa_swap_out(const pa_bf16* k_cache, const pa_bf16* v_cache, int32_t num_blocks,
                int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                const int32_t* block_ids, int32_t n, pa_bf16* staging, pa_bf16* host_k,
                pa_bf16* host_v, cudaStream_t stream) {
  return swap_blocks(const_cast<pa_bf16*>(k_cache), const_cast<pa_bf16*>(v_cache), num_blocks,
                     block_size, num_kv_heads, head_dim, block_ids, n, staging, host_k, host_v,
                     true, stream);
}

int pa_swap_in(pa_bf16* k_cache, pa_bf16* v_cache, int32_t num_blocks, int32_t block_size,
               int32_t num_kv_heads, int32_t head_dim, const int32_t* block_ids, int32_t n,
               pa_bf16* staging, const pa_bf16* host_k, const pa_bf16* host_v,
               cudaStream_t stream) {
  return swap_blocks(k_cache, v_cache, num_blocks, block_size, num_kv_heads, head_dim,
                     block_ids, n, staging, const_cast<pa_bf16*>(host_k),
                     const_cast<pa_bf16*>(host_v), false, stream);
}

size_t pa_workspace_size(int32_t num_seqs, int32_t num_tokens, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, int32_t max_q_len,
                         int32_t max_seq_len) {
  if (num_seqs < 0 || num_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      head_dim <= 0 || max_q_len < 0 || max_seq_len < 0)
    return 0;
  int sms = 0;
  if (device_state(nullptr, &sms)) return 0;
  const int ctas = pa::decode_ctas(sms);
  size_t bytes = pa::decode_workspace_bytes(ctas, num_seqs, num_q_heads, head_dim);
  bytes += pa::prefill_workspace_bound(num_tokens, num_q_heads, num_kv_heads, head_dim,
                                       max_q_len, max_seq_len, sms);
  return bytes;
}

int pa_prefill_splits(int32_t num_tokens, int32_t num_q_heads, int32_t num_kv_heads,
                      int32_t head_dim, int32_t max_q_len, int32_t max_seq_len) {
  if (num_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      max_q_len < 0 || max_seq_len < 0 || num_q_heads % num_kv_heads != 0)
    return 0;
  int sms = 0;
  if (device_state(nullptr, &sms)) return 0;
  return pa::prefill_plan(num_tokens, num_q_heads, num_kv_heads, head_dim, max_q_len,
                          max_seq_len, sms, ~size_t(0))
      .nsplit;
}

}  // extern "C"

namespace {

// pa_paged_attention with a cap on the workspace the prefill key split may
// take (the allocation-free entry point has a fixed array).
// The cache an attention call reads: bf16 values, or pages of E4M3 codes
// and their fp32 row scales.
struct KvCache {
  const void* k;
  const void* v;
  bool fp8;
};

int paged_attention_impl(const pa_bf16* q, KvCache kv,
                         int32_t num_blocks, int32_t block_size, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, const int32_t* block_tables,
                         int32_t max_blocks, const int32_t* seq_lens,
                         const int32_t* query_start_loc, int32_t num_seqs, int32_t num_tokens,
                         int32_t min_q_len, int32_t max_q_len, int32_t max_seq_len, float scale,
                         pa_bf16* out, void* workspace, size_t workspace_bytes, size_t split_cap,
                         cudaStream_t stream, const pa_bf16* fuse_k_new = nullptr,
                         const pa_bf16* fuse_v_new = nullptr,
                         const int32_t* fuse_slot_mapping = nullptr,
                         bool fuse_any_q_len = false);

}  // namespace

extern "C" {

int pa_paged_attention(const pa_bf16* q, const pa_bf16* k_cache, const pa_bf16* v_cache,
                       int32_t num_blocks, int32_t block_size, int32_t num_q_heads,
                       int32_t num_kv_heads, int32_t head_dim, const int32_t* block_tables,
                       int32_t max_blocks, const int32_t* seq_lens,
                       const int32_t* query_start_loc, int32_t num_seqs, int32_t num_tokens,
                       int32_t max_q_len, int32_t max_seq_len, float scale, pa_bf16* out,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return paged_attention_impl(q, KvCache{k_cache, v_cache, false}, num_blocks,
                              block_size, num_q_heads, num_kv_heads, head_dim, block_tables,
                              max_blocks, seq_lens, query_start_loc, num_seqs, num_tokens, 0,
                              max_q_len, max_seq_len, scale, out, workspace, workspace_bytes,
                              ~size_t(0), stream);
}

int pa_paged_attention_qrange(const pa_bf16* q, const pa_bf16* k_cache, const pa_bf16* v_cache,
                              int32_t num_blocks, int32_t block_size, int32_t num_q_heads,
                              int32_t num_kv_heads, int32_t head_dim, const int32_t* block_tables,
                              int32_t max_blocks, const int32_t* seq_lens,
                              const int32_t* query_start_loc, int32_t num_seqs,
                              int32_t num_tokens, int32_t min_q_len, int32_t max_q_len,
                              int32_t max_seq_len, float scale, pa_bf16* out, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  return paged_attention_impl(q, KvCache{k_cache, v_cache, false}, num_blocks,
                              block_size, num_q_heads, num_kv_heads, head_dim, block_tables,
                              max_blocks, seq_lens, query_start_loc, num_seqs, num_tokens,
                              min_q_len, max_q_len, max_seq_len, scale, out, workspace,
                              workspace_bytes, ~size_t(0), stream);
}

int pa_decode_step(const pa_bf16* q, const pa_bf16* k_new, const pa_bf16* v_new,
                   pa_bf16* k_cache, pa_bf16* v_cache, int32_t num_blocks, int32_t block_size,
                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                   const int32_t* block_tables, int32_t max_blocks, const int32_t* seq_lens,
                   const int32_t* query_start_loc, int32_t num_seqs, int32_t num_tokens,
                   int32_t max_seq_len, const int32_t* slot_mapping, float scale, pa_bf16* out,
                   void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!slot_mapping && num_tokens > 0)
    return fail(PA_ERR_INVALID_ARG, "null pointer argument (slot_mapping)");
  return paged_attention_impl(q, KvCache{k_cache, v_cache, false}, num_blocks,
                              block_size, num_q_heads, num_kv_heads, head_dim, block_tables,
                              max_blocks, seq_lens, query_start_loc, num_seqs, num_tokens, 0, 1,
                              max_seq_len, scale, out, workspace, workspace_bytes, ~size_t(0),
                              stream, k_new, v_new, slot_mapping);
}

int pa_paged_attention_step(const pa_bf16* q, const pa_bf16* k_new, const pa_bf16* v_new,
                            pa_bf16* k_cache, pa_bf16* v_cache, int32_t num_blocks,
                            int32_t block_size, int32_t num_q_heads, int32_t num_kv_heads,
                            int32_t head_dim, const int32_t* block_tables, int32_t max_blocks,
                            const int32_t* seq_lens, const int32_t* query_start_loc,
                            int32_t num_seqs, int32_t num_tokens, int32_t max_q_len,
                            int32_t max_seq_len, const int32_t* slot_mapping, float scale,
                            pa_bf16* out, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
  if (!slot_mapping && num_tokens > 0)
    return fail(PA_ERR_INVALID_ARG, "null pointer argument (slot_mapping)");
  return paged_attention_impl(q, KvCache{k_cache, v_cache, false}, num_blocks,
                              block_size, num_q_heads, num_kv_heads, head_dim, block_tables,
                              max_blocks, seq_lens, query_start_loc, num_seqs, num_tokens, 0,
                              max_q_len, max_seq_len, scale, out, workspace, workspace_bytes,
                              ~size_t(0), stream, k_new, v_new, slot_mapping, true);
}

int pa_paged_attention_fp8(const pa_bf16* q, const uint8_t* k_cache, const uint8_t* v_cache,
                           int32_t num_blocks, int32_t block_size, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim, const int32_t* block_tables,
                           int32_t max_blocks, const int32_t* seq_lens,
                           const int32_t* query_start_loc, int32_t num_seqs, int32_t num_tokens,
                           int32_t max_q_len, int32_t max_seq_len, float scale, pa_bf16* out,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return paged_attention_impl(q, KvCache{k_cache, v_cache, true}, num_blocks,
                              block_size, num_q_heads, num_kv_heads, head_dim, block_tables,
                              max_blocks, seq_lens, query_start_loc, num_seqs, num_tokens, 0,
                              max_q_len, max_seq_len, scale, out, workspace, workspace_bytes,
                              ~size_t(0), stream);
}

}  // extern "C"

namespace {

int paged_attention_impl(const pa_bf16* q, KvCache kv,
                         int32_t num_blocks, int32_t block_size, int32_t num_q_heads,
                         int32_t num_kv_heads, int32_t head_dim, const int32_t* block_tables,
                         int32_t max_blocks, const int32_t* seq_lens,
                         const int32_t* query_start_loc, int32_t num_seqs, int32_t num_tokens,
                         int32_t min_q_len, int32_t max_q_len, int32_t max_seq_len, float scale,
                         pa_bf16* out, void* workspace, size_t workspace_bytes, size_t split_cap,
                         cudaStream_t stream, const pa_bf16* fuse_k_new,
                         const pa_bf16* fuse_v_new,
                         const int32_t* fuse_slot_mapping, bool fuse_any_q_len) {
  const bool fuse = fuse_slot_mapping != nullptr;  // pa_decode_step
  int st = check_cache_geometry(num_blocks, block_size, num_kv_heads, head_dim);
  if (st) return st;
  if (num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return fail(PA_ERR_INVALID_ARG, "num_q_heads %d must be a positive multiple of "
                "num_kv_heads %d", num_q_heads, num_kv_heads);
  if (num_seqs < 0 || num_tokens < 0 || max_blocks < 0 || max_q_len < 0 || max_seq_len < 0)
    return fail(PA_ERR_INVALID_ARG, "negative size argument");
  if (max_q_len > max_seq_len)
    return fail(PA_ERR_INVALID_ARG, "max_q_len %d > max_seq_len %d", max_q_len, max_seq_len);
  if (min_q_len > max_q_len)
    return fail(PA_ERR_INVALID_ARG, "min_q_len %d > max_q_len %d", min_q_len, max_q_len);
  if (!(scale == scale)) return fail(PA_ERR_INVALID_ARG, "scale is NaN");
  if (block_size != 16 && block_size != 32)
    return fail(PA_ERR_UNSUPPORTED, "block_size %d (16 and 32 are implemented)", block_size);
  if ((int64_t)num_blocks * block_size > INT32_MAX)
    return fail(PA_ERR_UNSUPPORTED, "num_blocks * block_size above 2^31 - 1 token slots");
  const int group = num_q_heads / num_kv_heads;
  if (!pa::decode_supported(head_dim, group, num_kv_heads))
    return fail(PA_ERR_UNSUPPORTED, "shape head_dim=%d group=%d num_kv_heads=%d", head_dim,
                group, num_kv_heads);
  if (num_seqs == 0 || num_tokens == 0 || max_seq_len == 0) return PA_OK;
  if (!q || !kv.k || !kv.v || !block_tables || !seq_lens || !query_start_loc || !out)
    return fail(PA_ERR_INVALID_ARG, "null pointer argument");
  if (fuse && (!fuse_k_new || !fuse_v_new || !aligned(fuse_k_new, 16) ||
               !aligned(fuse_v_new, 16) || !aligned(fuse_slot_mapping, 4)))
    return fail(PA_ERR_INVALID_ARG, "k_new / v_new must be 16-byte aligned, slot_mapping 4-byte");
  if (!aligned(q, 16) || !aligned(kv.k, 16) || !aligned(kv.v, 16) || !aligned(out, 16) ||
      !aligned(block_tables, 4) || !aligned(seq_lens, 4) || !aligned(query_start_loc, 4))
    return fail(PA_ERR_INVALID_ARG, "bf16 arrays must be 16-byte aligned, int32 arrays 4-byte");
  if ((int64_t)max_blocks * block_size < max_seq_len)
    return fail(PA_ERR_INVALID_ARG, "max_blocks %d * block_size cannot hold max_seq_len %d",
                max_blocks, max_seq_len);
  if (fuse && max_q_len > 1 && !fuse_any_q_len)
    return fail(PA_ERR_INVALID_ARG, "pa_decode_step takes decode rows only (max_q_len %d)",
                max_q_len);
  if (max_q_len >= 2 && !pa::prefill_supported(head_dim, group, num_kv_heads))
    return fail(PA_ERR_UNSUPPORTED, "prefill rows (q_len >= 2) for head_dim=%d group=%d",
                head_dim, group);

  unsigned* err = nullptr;
  int sms = 0;
  st = device_state(&err, &sms);
  if (st) return st;
  const int ctas = pa::decode_ctas(sms);
  const size_t need_decode = pa::decode_workspace_bytes(ctas, num_seqs, num_q_heads, head_dim);
  if (!workspace || !aligned(workspace, 256))
    return fail(PA_ERR_WORKSPACE, "workspace must be a non-null 256-byte aligned pointer");
  if (workspace_bytes < need_decode)
    return fail(PA_ERR_WORKSPACE, "workspace %zu bytes < required %zu", workspace_bytes,
                need_decode);
  // the prefill key split takes only what the workspace has left
  const size_t left = workspace_bytes - need_decode;
  const pa::PrefillPlan plan =
      pa::prefill_plan(num_tokens, num_q_heads, num_kv_heads, head_dim, max_q_len, max_seq_len,
                       sms, left < split_cap ? left : split_cap);

  pa::AttnArgs a;
  a.q = q;
  a.k_cache = kv.k;
  a.v_cache = kv.v;
  a.fp8 = kv.fp8;
  a.fuse_k_new = fuse_k_new;
  a.fuse_v_new = fuse_v_new;
  a.fuse_slot_mapping = fuse_slot_mapping;
  a.num_blocks = num_blocks;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_tables = block_tables;
  a.max_blocks = max_blocks;
  a.seq_lens = seq_lens;
  a.query_start_loc = query_start_loc;
  a.num_seqs = num_seqs;
  a.num_tokens = num_tokens;
  a.max_q_len = max_q_len;
  a.max_seq_len = max_seq_len;
  a.block_shift = block_size == 32 ? 1 : 0;
  a.scale = scale;
  a.out = out;
  a.err = err;
  a.after_prefill = false;
  a.no_decode = min_q_len >= 2;

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  if (max_q_len >= 2) {
    pa::NvtxRange range(plan.nsplit > 1 ? "prefill (tcgen05) + key-piece merge"
                                        : "prefill (tcgen05)");
    cudaError_t e = pa::launch_prefill(a, plan, ws + need_decode, sms, stream);
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    // with key pieces the merge kernel comes last and must not be overtaken
    a.after_prefill = plan.nsplit == 1;
  }
  if (a.no_decode) return PA_OK;  // no request has a single query row
  pa::DecodeWorkspace dws = pa::decode_workspace(ws, ctas, num_seqs, num_q_heads, head_dim);
  pa::NvtxRange range(fuse    ? "decode step (scatter + split-KV decode) + merge"
                      : kv.fp8 ? "8-bit split-KV decode + merge"
                               : "split-KV decode + merge");
  cudaError_t e = pa::launch_decode(a, dws, ctas, stream);
  if (e != cudaSuccess) return cuda_fail(e, "decode launch");
  return PA_OK;
}

}  // namespace

extern "C" {

int pa_selftest_wait_timeout(uint64_t limit_ns, cudaStream_t stream) {
  if (limit_ns == 0 || limit_ns > 1000000000ull)
    return fail(PA_ERR_INVALID_ARG, "limit_ns %llu outside (0, 1 s]",
                (unsigned long long)limit_ns);
  unsigned* err = nullptr;
  int st = device_state(&err, nullptr);
  if (st) return st;
  cudaError_t e = pa::launch_wait_timeout_selftest(limit_ns, err, stream);
  if (e != cudaSuccess) return cuda_fail(e, "wait timeout self-test launch");
  return PA_OK;
}

int pa_check_device_errors(cudaStream_t stream) {
  unsigned* err = nullptr;
  int st = device_state(&err, nullptr);
  if (st) return st;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  unsigned word = 0;
  e = cudaMemcpy(&word, err, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read device error word");
  const unsigned zero = 0;
  e = cudaMemcpy(err, &zero, sizeof zero, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "clear device error word");
  if (word & pa::DEVERR_TIMEOUT)
    return fail(PA_ERR_TIMEOUT, "a kernel gave up a bounded wait (device word 0x%x)", word);
  if (word & pa::DEVERR_BOUNDS)
    return fail(PA_ERR_DEVICE_BOUNDS,
                "a kernel found an index or length out of range (device word 0x%x)", word);
  return PA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free variant of pa_paged_attention.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the
// point where they run attention: code that executes while a stream is being
// captured into a CUDA graph, plugins whose host application owns every
// device allocation and only hands out pointers, or latency-critical serving
// loops that forbid allocation after start-up.  For them this entry point
// uses a fixed scratch array that lives in the library itself instead of a
// caller-provided workspace.  The array is a file-scope __device__ object, so
// every GPU that loads the library holds it until the process exits.
//
// Its device address is looked up once per device, on the first call made on
// that device (with the device current), and kept for the life of the
// process, like the error word's: after a cudaDeviceReset both are stale, so
// the library must not be used across one.  Make that first call before any
// stream capture begins; a call with no requests does the look-up and
// launches nothing.  All calls share the array and it keeps whatever the
// last call left there: nothing in it needs to start at zero, but calls whose
// executions overlap on the GPU (different streams, or different threads on
// one device) race on it and must be serialised by the caller.
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_pa_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[kMaxDevices] = {};

int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PA_ERR_UNSUPPORTED, "device id %d", dev);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_pa_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(no-alloc scratch)");
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return PA_OK;
}

}  // namespace

extern "C" {

size_t pa_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int pa_paged_attention_noalloc(const pa_bf16* q, const pa_bf16* k_cache,
                               const pa_bf16* v_cache, int32_t num_blocks, int32_t block_size,
                               int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                               const int32_t* block_tables, int32_t max_blocks,
                               const int32_t* seq_lens, const int32_t* query_start_loc,
                               int32_t num_seqs, int32_t num_tokens, int32_t max_q_len,
                               int32_t max_seq_len, float scale, pa_bf16* out,
                               cudaStream_t stream) {
  // the split-KV decode part must fit; the prefill key split takes what is left
  const size_t need = pa_workspace_size(num_seqs, num_tokens, num_q_heads, num_kv_heads,
                                        head_dim, max_q_len < 1 ? max_q_len : 1, max_seq_len);
  if (need == 0)
    return fail(PA_ERR_INVALID_ARG, "invalid sizes, or no CUDA device for the scratch size");
  if (need > kNoAllocScratchBytes)
    return fail(PA_ERR_WORKSPACE,
                "this call needs %zu bytes of scratch, more than the %zu-byte built-in array "
                "of the allocation-free entry point; use pa_paged_attention with a workspace",
                need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  int st = noalloc_scratch(&scratch);
  if (st) return st;
  return paged_attention_impl(q, KvCache{k_cache, v_cache, false}, num_blocks,
                              block_size, num_q_heads, num_kv_heads, head_dim, block_tables,
                              max_blocks, seq_lens, query_start_loc, num_seqs, num_tokens, 0,
                              max_q_len, max_seq_len, scale, out, scratch, kNoAllocScratchBytes,
                              kNoAllocScratchBytes - need, stream);
}

}  // extern "C"
