// pa_decode_fp8.cu -- the 8-bit-cache instantiations of the split-KV decode
// kernel (pa_decode_kernel.cuh): E4M3 codes with one fp32 scale per cached
// (token, kv head) row.  A translation unit of its own so that the two sets
// of instantiations compile in parallel.
#include "pa_decode_kernel.cuh"

namespace pa {

cudaError_t launch_decode_fp8(const AttnArgs& a, const DecodeWorkspace& ws, int ctas,
                              cudaStream_t stream) {
  return launch_decode_any<true, false>(a, ws, ctas, stream);
}

}  // namespace pa
