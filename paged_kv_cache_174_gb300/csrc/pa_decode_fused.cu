// pa_decode_fused.cu -- the instantiations of the split-KV decode kernel
// (pa_decode_kernel.cuh) that also do a decode-only step's slot scatter
// (pa_decode_step): each request's new row comes from k_new / v_new into its
// last page in shared memory and is stored from there.  A translation unit
// of its own so that the instantiations compile in parallel.
#include "pa_decode_kernel.cuh"

namespace pa {

cudaError_t launch_decode_fused(const AttnArgs& a, const DecodeWorkspace& ws, int ctas,
                                cudaStream_t stream) {
  return launch_decode_any<false, true>(a, ws, ctas, stream);
}

}  // namespace pa
