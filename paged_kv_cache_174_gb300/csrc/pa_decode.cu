// pa_decode.cu -- the bf16-cache instantiations of the split-KV decode
// kernel (pa_decode_kernel.cuh), its workspace layout and the dispatch.
#include "pa_decode_kernel.cuh"

namespace pa {

int decode_ctas(int sm_count) { return sm_count; }

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

size_t decode_workspace_bytes(int ctas, int num_seqs, int num_q_heads, int head_dim) {
  return align256((size_t)ctas * 2 * num_q_heads * head_dim * sizeof(float)) +
         align256((size_t)ctas * 2 * num_q_heads * 2 * sizeof(float)) +
         align256((size_t)(num_seqs > 0 ? num_seqs : 1) * sizeof(int4));
}

DecodeWorkspace decode_workspace(void* base, int ctas, int num_seqs, int num_q_heads,
                                 int head_dim) {
  unsigned char* b = static_cast<unsigned char*>(base);
  DecodeWorkspace w;
  w.part_o = reinterpret_cast<float*>(b);
  b += align256((size_t)ctas * 2 * num_q_heads * head_dim * sizeof(float));
  w.part_ml = reinterpret_cast<float*>(b);
  b += align256((size_t)ctas * 2 * num_q_heads * 2 * sizeof(float));
  w.seq_rec = reinterpret_cast<int4*>(b);
  (void)num_seqs;
  return w;
}

bool decode_supported(int head_dim, int group, int num_kv_heads) {
  if (head_dim != 64 && head_dim != 128) return false;
  if (group != 1 && group != 2 && group != 4 && group != 8) return false;
  return num_kv_heads == 1 || num_kv_heads == 2 || num_kv_heads == 4 || num_kv_heads == 8;
}

cudaError_t launch_decode(const AttnArgs& a, const DecodeWorkspace& ws, int ctas,
                          cudaStream_t stream) {
  if (a.fp8) return launch_decode_fp8(a, ws, ctas, stream);
  if (a.fuse_slot_mapping) return launch_decode_fused(a, ws, ctas, stream);
  return launch_decode_any<false, false>(a, ws, ctas, stream);
}

}  // namespace pa
