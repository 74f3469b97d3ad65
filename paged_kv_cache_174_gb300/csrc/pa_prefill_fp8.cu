// pa_prefill_fp8.cu -- the chunked-prefill kernel's instance for the 8-bit
// (E4M3 codes + row scales) cache: its own translation unit, so that the
// build compiles it beside the plain and fused-step instances.
#include "pa_prefill_kernel.cuh"

namespace pa {

cudaError_t launch_prefill_fp8(const AttnArgs& a, const PrefillPlan& plan, void* ws,
                               int sm_count, cudaStream_t stream) {
  const int group = a.num_q_heads / a.num_kv_heads;
#define PA_PREFILL_FP8_CASE(D_, G_)    \
  if (a.head_dim == D_ && group == G_) \
    return launch_prefill_t<D_, G_, kKindFp8>(a, plan, ws, sm_count, stream);
  PA_PREFILL_FP8_CASE(128, 1)
  PA_PREFILL_FP8_CASE(128, 2)
  PA_PREFILL_FP8_CASE(128, 4)
  PA_PREFILL_FP8_CASE(128, 8)
  PA_PREFILL_FP8_CASE(64, 1)
  PA_PREFILL_FP8_CASE(64, 2)
  PA_PREFILL_FP8_CASE(64, 4)
  PA_PREFILL_FP8_CASE(64, 8)
#undef PA_PREFILL_FP8_CASE
  return cudaErrorInvalidValue;
}

}  // namespace pa
