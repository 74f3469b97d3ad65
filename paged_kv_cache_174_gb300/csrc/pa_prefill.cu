// pa_prefill.cu -- chunked-prefill attention (requests with q_len >= 2) on
// the tcgen05 tensor cores.  Placeholder until the kernel lands.
#include "pa_internal.h"

namespace pa {

bool prefill_supported(int, int, int) { return false; }

size_t prefill_workspace_bytes(int, int, int, int, int) { return 0; }

cudaError_t launch_prefill(const AttnArgs&, void*, size_t, int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace pa
