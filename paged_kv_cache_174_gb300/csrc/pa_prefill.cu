// pa_prefill.cu -- host side of the chunked-prefill attention (the kernels
// are in pa_prefill_kernel.cuh): which shapes run, the key-split plan and
// its workspace bound, and the launch of the plain and fused-step instances
// (the 8-bit cache's instance is compiled in pa_prefill_fp8.cu).
#include <algorithm>

#include "pa_prefill_kernel.cuh"

namespace pa {

bool prefill_supported(int head_dim, int group, int num_kv_heads) {
  return (head_dim == 64 || head_dim == 128) &&
         (group == 1 || group == 2 || group == 4 || group == 8) && num_kv_heads >= 1;
}

// Key splits: enough units to fill about 70% of the SMs when the query tiles
// alone would not (every token counted as a prefill row), at least four K/V
// tiles per piece of the longest request, at most kMaxSplit, and no more
// pieces than max_bytes of workspace hold.
PrefillPlan prefill_plan(int num_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                         int max_q_len, int max_seq_len, int sm_count, size_t max_bytes) {
  PrefillPlan plan;
  plan.nsplit = 1;
  plan.bytes = 0;
  if (max_q_len < 2 || num_kv_heads <= 0 || num_q_heads < num_kv_heads || head_dim <= 0)
    return plan;
  const int tm = kRows / (num_q_heads / num_kv_heads);
  const long long units = (long long)((num_tokens + tm - 1) / tm) * num_kv_heads;
  const int tiles = (max_seq_len + kKeysPerTile - 1) / kKeysPerTile;
  int ns = 1;
  while (ns < kMaxSplit && units * ns * 10 < (long long)sm_count * 7 && tiles >= 4 * (ns + 1))
    ++ns;
  while (ns > 1 && split_bytes(num_tokens, num_q_heads, head_dim, ns) > max_bytes) --ns;
  plan.nsplit = ns;
  plan.bytes = split_bytes(num_tokens, num_q_heads, head_dim, ns);
  return plan;
}

size_t prefill_workspace_bound(int num_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                               int max_q_len, int max_seq_len, int sm_count) {
  if (max_q_len < 2 || num_kv_heads <= 0 || num_q_heads < num_kv_heads || head_dim <= 0)
    return 0;
  // Fewer tokens can mean more pieces, so take the largest plan of any token
  // count up to num_tokens.  Past tm * sm_count tokens the query tiles alone
  // fill the SMs and nothing is split.
  const int tm = kRows / (num_q_heads / num_kv_heads);
  const long long last = std::min<long long>(num_tokens, (long long)tm * sm_count);
  size_t most = 0;
  for (long long t = 2; t <= last; ++t)
    most = std::max(most, prefill_plan((int)t, num_q_heads, num_kv_heads, head_dim, max_q_len,
                                       max_seq_len, sm_count, ~size_t(0))
                              .bytes);
  return most;
}

cudaError_t launch_prefill(const AttnArgs& a, const PrefillPlan& plan, void* ws, int sm_count,
                           cudaStream_t stream) {
  const int group = a.num_q_heads / a.num_kv_heads;
  if (a.fp8) return launch_prefill_fp8(a, plan, ws, sm_count, stream);
  // the fused step's instance loads new rows from k_new / v_new and stores
  // them; the plain one reads the cache only
  const bool fuse = a.fuse_slot_mapping != nullptr;
#define PA_PREFILL_CASE(D_, G_)                                                         \
  if (a.head_dim == D_ && group == G_)                                                  \
    return fuse ? launch_prefill_t<D_, G_, kKindFused>(a, plan, ws, sm_count, stream) \
                : launch_prefill_t<D_, G_, kKindPlain>(a, plan, ws, sm_count, stream);
  PA_PREFILL_CASE(128, 1)
  PA_PREFILL_CASE(128, 2)
  PA_PREFILL_CASE(128, 4)
  PA_PREFILL_CASE(128, 8)
  PA_PREFILL_CASE(64, 1)
  PA_PREFILL_CASE(64, 2)
  PA_PREFILL_CASE(64, 4)
  PA_PREFILL_CASE(64, 8)
#undef PA_PREFILL_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pa
