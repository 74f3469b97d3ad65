// pa_cache.cu -- the two cache-maintenance kernels: the slot scatter that
// writes a step's new K/V rows into their physical slots, and the
// copy-on-write block copy.  Both are pure bit copies with 16-byte vectors;
// HBM-bound.
//
// Slot scatter: "PagedAttention 显存分页与连续批处理(Continuous Batching)实战",
//   comparison table (blocks allocated on demand as a block fills) and the
//   TypeScript Block Manager's appendToken (a new token lands in the last
//   block of the request's Block Table).
// Copy-on-write: same page, comparison table ("Copy-on-Write ... shared
//   blocks"); "连续批处理：推理吞吐的范式革命", section 4.2 (prefix sharing).
// Block swap: "连续批处理：推理吞吐的范式革命", section 3.3 (a preempted
//   request's KV cache goes to CPU memory and comes back without
//   recomputation); "vLLM中的PagedAttention机制与显存优化实践", section 2.1
//   (swap is block-grained and asynchronous on its own streams).  A kernel
//   packs the listed blocks into a staging buffer (or unpacks them), so the
//   host transfer is two large copies rather than one per block.
// 8-bit cache scatter: each (token, kv head) row is quantised to E4M3 codes
//   with one fp32 scale (row max / 448), written into the slot's 16-token
//   page (codes first, then the page's scales); the block copy of that cache
//   moves whole pages.
#include <cstdint>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kScatterWarps = 8;

// One warp per new token: copy its K row and V row (num_kv_heads * head_dim
// bf16 each, row_vec 16-byte vectors) to slot slot_mapping[t].
__global__ void __launch_bounds__(kScatterWarps * 32)
    reshape_and_cache_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                             int32_t num_tokens, uint4* __restrict__ k_cache,
                             uint4* __restrict__ v_cache, int64_t num_slots, int32_t row_vec,
                             const int32_t* __restrict__ slot_mapping, unsigned* err) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * kScatterWarps + warp;
  if (t >= num_tokens) return;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (lane == 0) flag_error(err, DEVERR_BOUNDS);
    return;
  }
  const uint4* ks = k + t * row_vec;
  const uint4* vs = v + t * row_vec;
  uint4* kd = k_cache + slot * row_vec;
  uint4* vd = v_cache + slot * row_vec;
  for (int i = lane; i < row_vec; i += 32) {
    const uint4 a = __ldg(ks + i);
    const uint4 b = __ldg(vs + i);
    kd[i] = a;
    vd[i] = b;
  }
}

// One warp per new token, quantising its K and V rows into the 8-bit cache:
// LPH = head_dim / 8 lanes per kv head, each with 8 elements; the row max
// comes from a shuffle reduction over those lanes, then scale = max / 448
// (1 for an all-zero row) and code = e4m3(x / scale), both divisions IEEE
// round-to-nearest, as the definition fixes.
template <int LPH>
__global__ void __launch_bounds__(kScatterWarps * 32)
    reshape_and_cache_fp8_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                 int32_t num_tokens, unsigned char* __restrict__ k_cache,
                                 unsigned char* __restrict__ v_cache, int64_t num_slots,
                                 int32_t num_kv_heads, const int32_t* __restrict__ slot_mapping,
                                 unsigned* err) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * kScatterWarps + warp;
  if (t >= num_tokens) return;
  const int64_t slot = slot_mapping[t];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (lane == 0) flag_error(err, DEVERR_BOUNDS);
    return;
  }
  constexpr int HPP = 32 / LPH;  // kv heads per pass of the warp
  constexpr int D = LPH * 8;
  const int sub = lane % LPH;
  const int row_vec = num_kv_heads * LPH;  // 8-element vectors per token row
  // the slot's page and row: codes at row * n_kv + h, scales after the codes
  const int64_t page_off = (slot / kFp8PageTokens) * fp8_page_bytes(num_kv_heads, D);
  const int r = (int)(slot % kFp8PageTokens);
  const int64_t scales_off = page_off + fp8_scales_offset(num_kv_heads, D);
  for (int h0 = 0; h0 < num_kv_heads; h0 += HPP) {
    const int h = h0 + lane / LPH;
    const bool on = h < num_kv_heads;
#pragma unroll
    for (int which = 0; which < 2; ++which) {
      const uint4* src = which ? v : k;
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (on) w = __ldg(src + t * row_vec + h * LPH + sub);
      const float2 x0 = bf16x2_to_float2(w.x), x1 = bf16x2_to_float2(w.y);
      const float2 x2 = bf16x2_to_float2(w.z), x3 = bf16x2_to_float2(w.w);
      float amax = fmaxf(fmaxf(fmaxf(fabsf(x0.x), fabsf(x0.y)), fmaxf(fabsf(x1.x), fabsf(x1.y))),
                         fmaxf(fmaxf(fabsf(x2.x), fabsf(x2.y)), fmaxf(fabsf(x3.x), fabsf(x3.y))));
#pragma unroll
      for (int m = LPH / 2; m >= 1; m >>= 1)
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
      const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
      uint2 codes;
      codes.x = (uint32_t)e4m3x2_from_floats(__fdiv_rn(x0.x, sc), __fdiv_rn(x0.y, sc)) |
                ((uint32_t)e4m3x2_from_floats(__fdiv_rn(x1.x, sc), __fdiv_rn(x1.y, sc)) << 16);
      codes.y = (uint32_t)e4m3x2_from_floats(__fdiv_rn(x2.x, sc), __fdiv_rn(x2.y, sc)) |
                ((uint32_t)e4m3x2_from_floats(__fdiv_rn(x3.x, sc), __fdiv_rn(x3.y, sc)) << 16);
      if (on) {
        unsigned char* cache = which ? v_cache : k_cache;
        *reinterpret_cast<uint2*>(cache + page_off + ((int64_t)r * row_vec + h * LPH + sub) * 8) =
            codes;
        if (sub == 0)
          *reinterpret_cast<float*>(cache + scales_off + ((int64_t)r * num_kv_heads + h) * 4) = sc;
      }
    }
  }
}

// Failure-detection self-test: the bounded wait every kernel uses, on a
// barrier that nothing ever completes, with a short limit.  The wait gives
// up, sets the timeout bit of the error word and the kernel returns, so the
// context stays usable.
__global__ void wait_timeout_selftest_kernel(unsigned long long limit_ns, unsigned* err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait(smem_addr(&bar), 0, err, &abort_flag, limit_ns);  // nothing arrives
}

constexpr int kCopyThreads = 256;

// One CTA per (src, dst) pair: copy the K block and the V block.
__global__ void __launch_bounds__(kCopyThreads)
    copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                       int32_t num_blocks, int64_t block_vec, const int32_t* __restrict__ pairs,
                       unsigned* err) {
  const int64_t src = pairs[2 * (int64_t)blockIdx.x];
  const int64_t dst = pairs[2 * (int64_t)blockIdx.x + 1];
  if (src == -1) return;  // padding of a fixed-size pair list
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0) flag_error(err, DEVERR_BOUNDS);
    return;
  }
  const uint4* ks = k_cache + src * block_vec;
  const uint4* vs = v_cache + src * block_vec;
  uint4* kd = k_cache + dst * block_vec;
  uint4* vd = v_cache + dst * block_vec;
  for (int64_t i = threadIdx.x; i < block_vec; i += kCopyThreads) {
    const uint4 a = ks[i];
    const uint4 b = vs[i];
    kd[i] = a;
    vd[i] = b;
  }
}

// One CTA per listed block: stage[i] <- cache[ids[i]] (to_stage) or
// cache[ids[i]] <- stage[i], for K and V.
__global__ void __launch_bounds__(kCopyThreads)
    swap_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                       uint4* __restrict__ k_stage, uint4* __restrict__ v_stage,
                       int32_t num_blocks, int64_t block_vec, const int32_t* __restrict__ ids,
                       bool to_stage, unsigned* err) {
  const int64_t b = ids[blockIdx.x];
  if (b < 0 || b >= num_blocks) {
    if (threadIdx.x == 0) flag_error(err, DEVERR_BOUNDS);
    return;
  }
  uint4* kc = k_cache + b * block_vec;
  uint4* vc = v_cache + b * block_vec;
  uint4* ks = k_stage + (int64_t)blockIdx.x * block_vec;
  uint4* vs = v_stage + (int64_t)blockIdx.x * block_vec;
  for (int64_t i = threadIdx.x; i < block_vec; i += kCopyThreads) {
    if (to_stage) {
      const uint4 a = kc[i];
      const uint4 c = vc[i];
      ks[i] = a;
      vs[i] = c;
    } else {
      const uint4 a = ks[i];
      const uint4 c = vs[i];
      kc[i] = a;
      vc[i] = c;
    }
  }
}

}  // namespace

cudaError_t launch_swap(uint16_t* k_cache, uint16_t* v_cache, int32_t num_blocks,
                        int64_t block_elems, const int32_t* ids, int32_t n, uint16_t* staging,
                        uint16_t* host_k, uint16_t* host_v, bool out, unsigned* err,
                        cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  const size_t bytes = (size_t)n * block_elems * sizeof(uint16_t);
  uint16_t* k_stage = staging;
  uint16_t* v_stage = staging + (size_t)n * block_elems;
  cudaError_t e;
  if (!out) {
    e = cudaMemcpyAsync(k_stage, host_k, bytes, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyAsync(v_stage, host_v, bytes, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return e;
  }
  swap_blocks_kernel<<<n, kCopyThreads, 0, stream>>>(
      reinterpret_cast<uint4*>(k_cache), reinterpret_cast<uint4*>(v_cache),
      reinterpret_cast<uint4*>(k_stage), reinterpret_cast<uint4*>(v_stage), num_blocks,
      block_elems / 8, ids, out, err);
  e = cudaGetLastError();
  if (e != cudaSuccess || !out) return e;
  e = cudaMemcpyAsync(host_k, k_stage, bytes, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  return cudaMemcpyAsync(host_v, v_stage, bytes, cudaMemcpyDeviceToHost, stream);
}

cudaError_t launch_reshape_and_cache(const uint16_t* k, const uint16_t* v, int32_t num_tokens,
                                     uint16_t* k_cache, uint16_t* v_cache, int64_t num_slots,
                                     int32_t row_elems, const int32_t* slot_mapping,
                                     unsigned* err, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int grid = (num_tokens + kScatterWarps - 1) / kScatterWarps;
  reshape_and_cache_kernel<<<grid, kScatterWarps * 32, 0, stream>>>(
      reinterpret_cast<const uint4*>(k), reinterpret_cast<const uint4*>(v), num_tokens,
      reinterpret_cast<uint4*>(k_cache), reinterpret_cast<uint4*>(v_cache), num_slots,
      row_elems / 8, slot_mapping, err);
  return cudaGetLastError();
}

cudaError_t launch_reshape_and_cache_fp8(const uint16_t* k, const uint16_t* v,
                                         int32_t num_tokens, uint8_t* k_cache, uint8_t* v_cache,
                                         int64_t num_slots, int32_t num_kv_heads,
                                         int32_t head_dim, const int32_t* slot_mapping,
                                         unsigned* err, cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int grid = (num_tokens + kScatterWarps - 1) / kScatterWarps;
  auto args = [&](auto kern) {
    kern<<<grid, kScatterWarps * 32, 0, stream>>>(
        reinterpret_cast<const uint4*>(k), reinterpret_cast<const uint4*>(v), num_tokens,
        k_cache, v_cache, num_slots, num_kv_heads, slot_mapping, err);
    return cudaGetLastError();
  };
  if (head_dim == 128) return args(reshape_and_cache_fp8_kernel<16>);
  if (head_dim == 64) return args(reshape_and_cache_fp8_kernel<8>);
  return cudaErrorInvalidValue;
}

cudaError_t launch_wait_timeout_selftest(unsigned long long limit_ns, unsigned* err,
                                         cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 64, 0, stream>>>(limit_ns, err);
  return cudaGetLastError();
}

cudaError_t launch_copy_blocks(uint16_t* k_cache, uint16_t* v_cache, int32_t num_blocks,
                               int64_t block_elems, const int32_t* pairs, int32_t num_pairs,
                               unsigned* err, cudaStream_t stream) {
  if (num_pairs == 0) return cudaSuccess;
  copy_blocks_kernel<<<num_pairs, kCopyThreads, 0, stream>>>(
      reinterpret_cast<uint4*>(k_cache), reinterpret_cast<uint4*>(v_cache), num_blocks,
      block_elems / 8, pairs, err);
  return cudaGetLastError();
}

}  // namespace pa
