// pa_decode_kernel.cuh -- split-KV decode attention over the paged KV cache,
// and the log-sum-exp merge of the splits.  Included by pa_decode.cu (bf16
// cache) and pa_decode_fp8.cu (8-bit cache), each of which instantiates the
// templates it launches.
//
// What it computes ("连续批处理：推理吞吐的范式革命", section 4.1): for every
// request with exactly one query token, walk its Block Table, score each
// cached key against q (scaled dot product), softmax over the keys, and sum
// the values with those weights; the page's "many small per-block matmuls
// then merge the softmax results" is the split/merge structure used here.
// The page's kernel is one thread block per (token, head) with a scalar loop;
// this kernel is organised around GB300's memory system instead:
//
//  * Work is the flat list of (request, page) pairs of all decode requests.
//    One persistent CTA per SM takes an equal contiguous slice of it, so the
//    load is balanced to within one page whatever the length mix.  A slice
//    may start or end inside a request; such pieces leave a partial result
//    (unnormalised o, running max m, sum l) that the merge kernel combines.
//  * A page of the cache ([16 tokens][num_kv_heads][head_dim]) is one
//    contiguous block of memory, so K and V pages are fetched whole with one
//    bulk asynchronous copy each into a ring of shared-memory stages, tracked
//    by mbarriers (the last warp to release a stage refills it): several
//    pages per SM are in flight at once, which is what keeps HBM busy.
//  * 8-bit cache (F8): the page holds E4M3 codes and, after all 16 rows, one
//    fp32 scale per (token, kv head) row, so one copy per K or V page brings
//    both (two small scale copies per page beside the codes cost 4 us more
//    on the 8-bit decode batch).
//    A key row's score is (q . codes) * scale; a value row is codes * scale.
//  * Each consumer warp owns one kv head (and a slice of the page's tokens)
//    and all q heads of its GQA group, so every K/V byte is read from HBM
//    once.  Lanes hold a 16-byte slice of head_dim; q.k is reduced with
//    warp shuffles that also spread the group's heads across lanes.
//  * Online softmax per page in base 2 (q is pre-scaled by scale * log2 e),
//    fp32 accumulation with packed fp32x2 FMAs.
#pragma once
#include <type_traits>

#include <cstdint>
#include <cfloat>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kBlock = 16;  // tokens per physical block
constexpr float kNegInf = -INFINITY;

struct DecodeParams {
  const uint16_t* q;
  const void* k_cache;     // bf16 values, or (F8) pages of E4M3 codes and row scales
  const void* v_cache;
  // Fused scatter (bf16 cache, decode-only steps): the new token of a decode
  // request comes from k_new / v_new into its page in shared memory and is
  // stored from there to its slot slot_mapping[t], which must be the slot of
  // position seq_len - 1; null when the scatter ran separately.
  const uint16_t* k_new;
  const uint16_t* v_new;
  const int32_t* slot_mapping;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* qsl;
  uint16_t* out;
  float* part_o;
  float* part_ml;
  int4* seq_rec;
  unsigned* err;
  int32_t num_blocks, max_blocks, num_seqs, num_tokens, n_q, n_kv, max_seq_len;
  int32_t block_shift;  // log2(block_size / 16)
  float scale_log2;
  int32_t nstages;
  int32_t ctas;
  uint32_t stage_bytes;  // K page + V page
  uint32_t page_bytes;   // one K (or V) page of 16 tokens: 16 * n_kv * head_dim * elem,
                         // F8: the codes, then their 16 * n_kv fp32 scales
  uint32_t row_bytes;    // one token row of one cache: n_kv * head_dim * elem
};

// Pages this kernel processes for request s (0 if it is not a decode request
// or is invalid; invalid ones flag the error word once, from CTA 0).
__device__ __forceinline__ int decode_pages(const DecodeParams& p, int s, bool report) {
  const int a = __ldg(p.qsl + s), b = __ldg(p.qsl + s + 1);
  if (b - a != 1) return 0;
  const int L = __ldg(p.seq_lens + s);
  if (L < 1 || L > p.max_seq_len || L > (p.max_blocks << p.block_shift) * kBlock || a < 0 ||
      a >= p.num_tokens) {
    if (report) flag_error(p.err, DEVERR_BOUNDS);
    return 0;
  }
  return (L + kBlock - 1) / kBlock;
}

__device__ __forceinline__ int64_t slice_begin(int64_t c, int64_t F, int64_t C) {
  return c * F / C;
}

// Shared-memory state after the stage ring (dynamic shared memory).
template <int G>
struct PBuf {          // hand-off from the QK warp to the PV warp of one kv head
  float p[kBlock][G];  // exp2(score - m) of the page's tokens
  float alpha[G];      // rescale of the running output for this page
  float m[G];          // running max after this page (segment end only)
  float l[G];          // running sum after this page (segment end only)
};

template <int G, int NKV>
struct DecodeSmem {
  uint64_t full[8];           // stage holds its page (bulk-copy transaction count)
  uint64_t p_full[NKV][2];    // QK warp -> PV warp: page's p is ready
  uint64_t p_empty[NKV][2];   // PV warp -> QK warp: buffer may be rewritten
  int released[8];            // warps done with the page in the stage
  int last_issued[8];         // last page whose copies went into the stage (-1: none)
  int fused_slot[8];          // slot the stage's last row goes to (fused scatter), else -1
  PBuf<G> pb[NKV][2];
  int plan[2];
  int abort_flag;
};

// 8-bit cache: running state of the odd-page warp of one kv head at the end
// of a segment, read by the even-page warp (after the stage ring and DecodeSmem).
template <int G, int D>
struct Comb {
  float o[G][D];  // unnormalised output of the odd pages
  float m[2][G];  // running max per page parity
  float l[2][G];  // running sum per page parity
};

template <int G, int NKV>
__host__ __device__ constexpr size_t comb_offset() {
  return (sizeof(DecodeSmem<G, NKV>) + 15) / 16 * 16;
}

// Walks the flat page list of the decode requests: (request s, page j).
struct PageCursor {
  int s, j, np;
  __device__ __forceinline__ void next(const DecodeParams& p) {
    if (++j == np) {
      j = 0;
      do {
        ++s;
      } while (s < p.num_seqs && (np = decode_pages(p, s, false)) == 0);
    }
  }
};

// L2 policy for data read once per call (evicted before other lines), and a
// bulk copy that carries it.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst_smem, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst_smem),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

// Issue the bulk copies of page (c.s, c.j) into a stage.  *fused_slot gets the
// slot the stage's last row must be stored to (fused scatter), or -1.
template <bool FUSE, bool F8>
__device__ __forceinline__ void fetch_page(const DecodeParams& p, const PageCursor& c,
                                           uint32_t stage_smem, uint32_t full_bar,
                                           int* fused_slot) {
  const int L = __ldg(p.seq_lens + c.s);
  const int ntok = min(kBlock, L - c.j * kBlock);
  const int phys =
      __ldg(p.block_tables + (int64_t)c.s * p.max_blocks + (c.j >> p.block_shift));
  *fused_slot = -1;
  if (phys < 0 || phys >= p.num_blocks) {
    flag_error(p.err, DEVERR_BOUNDS);
    mbar_arrive_expect_tx(full_bar, 0);  // completes the phase with no data
    return;
  }
  // the page's rows (F8: the whole page, whose scales follow all 16 rows;
  // rows past ntok are never used)
  const uint32_t bytes = F8 ? p.page_bytes : (uint32_t)ntok * p.row_bytes;
  mbar_arrive_expect_tx(full_bar, 2 * bytes);
  // 16-token page index in the pool: a block of 32 tokens is two pages
  const size_t page = ((size_t)phys << p.block_shift) + (c.j & ((1 << p.block_shift) - 1));
  const size_t off = page * p.page_bytes;
  // the pages are read once per call: evict-first keeps them from pushing
  // the call's reused data (tables, q, partial results) out of L2 (decode
  // batch on GB300: 91.3 against 93.6 us per call)
  const uint64_t pol = l2_evict_first_policy();
  if (FUSE && c.j == c.np - 1) {
    // the request's new token (position L - 1, last row of this page) comes
    // from k_new / v_new instead of the cache, which does not hold it yet
    const int a = __ldg(p.qsl + c.s);
    const int64_t slot = __ldg(p.slot_mapping + a);
    const int64_t want = (int64_t)page * kBlock + (ntok - 1);
    if (slot == want) {
      const uint32_t head = (uint32_t)(ntok - 1) * p.row_bytes;  // rows before the new one
      if (head) {
        bulk_g2s_hint(stage_smem, reinterpret_cast<const unsigned char*>(p.k_cache) + off, head,
                      full_bar, pol);
        bulk_g2s_hint(stage_smem + p.page_bytes,
                      reinterpret_cast<const unsigned char*>(p.v_cache) + off, head, full_bar,
                      pol);
      }
      bulk_g2s(stage_smem + head, p.k_new + (int64_t)a * (p.row_bytes / 2), p.row_bytes,
               full_bar);
      bulk_g2s(stage_smem + p.page_bytes + head, p.v_new + (int64_t)a * (p.row_bytes / 2),
               p.row_bytes, full_bar);
      *fused_slot = (int)slot;
      return;
    }
    // a negative slot is a token not to be written: the cache's row is read,
    // as with a separate scatter; any other slot breaks the precondition
    if (slot >= 0) flag_error(p.err, DEVERR_BOUNDS);
  }
  bulk_g2s_hint(stage_smem, reinterpret_cast<const unsigned char*>(p.k_cache) + off, bytes,
                full_bar, pol);
  bulk_g2s_hint(stage_smem + p.page_bytes, reinterpret_cast<const unsigned char*>(p.v_cache) + off,
                bytes, full_bar, pol);
}

template <int N>
__device__ __forceinline__ void lds_floats(uint32_t addr, float (&v)[N]) {
  if constexpr (N % 4 == 0) {
#pragma unroll
    for (int i = 0; i < N; i += 4) {
      const float4 x = lds128f(addr + 4 * i);
      v[i] = x.x, v[i + 1] = x.y, v[i + 2] = x.z, v[i + 3] = x.w;
    }
  } else if constexpr (N == 2) {
    float2 x;
    asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(x.x), "=f"(x.y) : "r"(addr));
    v[0] = x.x, v[1] = x.y;
  } else {
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v[0]) : "r"(addr));
  }
}

// Sum over the LPT lanes of one token, handing out the G values: after the
// call, lane holds the total of value index (lane % LPT) / (LPT / G).
template <int G, int LPT>
__device__ __forceinline__ float reduce_scatter(float (&part)[G], int lane) {
  int cnt = G;
#pragma unroll
  for (int m = LPT / 2; m >= 1; m >>= 1) {
    if (cnt > 1) {
      const int half = cnt / 2;
      const bool upper = (lane & m) != 0;
#pragma unroll
      for (int x = 0; x < G / 2; ++x) {
        if (x < half) {
          const float send = upper ? part[x] : part[x + half];
          const float keep = upper ? part[x + half] : part[x];
          part[x] = keep + __shfl_xor_sync(0xffffffffu, send, m);
        }
      }
      cnt = half;
    } else {
      part[0] += __shfl_xor_sync(0xffffffffu, part[0], m);
    }
  }
  return part[0];
}

// Scores of one page for one QK warp.  kb points at this lane's 16-byte piece
// of its first token's key row in the stage; FULL pages need no per-token
// predicate.  sc[it] is the base-2 score of token it * TPI + tok_lane for the
// head this lane holds after the reduce-scatter (-inf past the page's end).
// (bf16 cache; the 8-bit cache runs on the tensor cores, qk_scores_mma.)
template <int D, int G, int E_QK, int LPT, uint32_t ROW, bool FULL>
__device__ __forceinline__ void qk_scores(const unsigned char* kb, int ntok,
                                          int tok_lane, const float2 (&qf)[G][E_QK / 2],
                                          float (&sc)[kBlock / (32 / LPT)], int lane) {
  constexpr int TPI = 32 / LPT;
  constexpr int NIT = kBlock / TPI;
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    const bool valid = FULL || (it * TPI + tok_lane < ntok);
    float2 a2[G];
#pragma unroll
    for (int h = 0; h < G; ++h) a2[h] = make_float2(0.f, 0.f);
    if (valid) {
#pragma unroll
      for (int piece = 0; piece < E_QK / 8; ++piece) {
        float2 k2[4];
        const uint4 kw = *reinterpret_cast<const uint4*>(kb + it * TPI * ROW + piece * D);
        k2[0] = bf16x2_to_float2(kw.x), k2[1] = bf16x2_to_float2(kw.y);
        k2[2] = bf16x2_to_float2(kw.z), k2[3] = bf16x2_to_float2(kw.w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
#pragma unroll
          for (int h = 0; h < G; ++h) a2[h] = __ffma2_rn(qf[h][piece * 4 + e], k2[e], a2[h]);
        }
      }
    }
    float part[G];
#pragma unroll
    for (int h = 0; h < G; ++h) part[h] = a2[h].x + a2[h].y;
    const float s = reduce_scatter<G, LPT>(part, lane);
    sc[it] = valid ? s : kNegInf;
  }
}

// 8-bit cache: q . k of one page on the tensor cores (mma.sync m16n8k16,
// f16 operands, f32 accumulation).  The MMA rows are the G q heads of the kv
// group (rows G..15 zero), the columns the page's 16 tokens (two n-tiles of
// 8), the reduction head_dim.  The reduction order is free, so lane (g, t) =
// (lane / 4, lane % 4) takes head_dim elements [t * D/4, (t + 1) * D/4) for
// every k-step: k-step s holds elements t * D/4 + 4s .. + 3, which is one
// 32-bit word of codes per token -- two f16x2 B registers -- and the same
// elements of q in its A registers.  E4M3 values are exact in f16.
__device__ __forceinline__ void mma_f16_16816(float (&c)[4], uint32_t a0, uint32_t a2,
                                              uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t chunk_word(const uint4& x, int q) {
  return q == 0 ? x.x : q == 1 ? x.y : q == 2 ? x.z : x.w;
}
__device__ __forceinline__ uint32_t chunk_word(const uint2& x, int q) {
  return q == 0 ? x.x : x.y;
}
// Barrier over the `threads` threads (whole warps) that name barrier `id`.
__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ void mma_f16_16816_full(float (&c)[4], uint32_t a0, uint32_t a1,
                                                   uint32_t a2, uint32_t a3, uint32_t b0,
                                                   uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Scores of one page on the tensor cores (bf16 cache), as qk_scores_mma
// below but with the cached bf16 values as B directly (two 32-bit words per
// k-step) and q unscaled in A; the fp32 score takes scale * log2(e).
template <int D, uint32_t ROW>
__device__ __forceinline__ void qk_scores_mma_bf16(const unsigned char* kb, int ntok,
                                                   const uint32_t (&qa)[D / 16][2],
                                                   float scale_log2, float (&sc)[4], int lane) {
  const int g = lane >> 2, t = lane & 3;
  float c[2][4];
#pragma unroll
  for (int T = 0; T < 2; ++T) {
#pragma unroll
    for (int e = 0; e < 4; ++e) c[T][e] = 0.f;
    // this lane's D/4 values of token 8T + g (2 bytes each)
    const unsigned char* src = kb + (8 * T + g) * ROW + t * (D / 2);
    uint32_t w[D / 8];
#pragma unroll
    for (int v = 0; v < D / 32; ++v) {
      const uint4 x = *reinterpret_cast<const uint4*>(src + 16 * v);
      w[4 * v] = x.x, w[4 * v + 1] = x.y, w[4 * v + 2] = x.z, w[4 * v + 3] = x.w;
    }
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks)
      mma_bf16_16816(c[T], qa[ks][0], 0u, qa[ks][1], 0u, w[2 * ks], w[2 * ks + 1]);
  }
#pragma unroll
  for (int T = 0; T < 2; ++T)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int tok = 8 * T + 2 * t + j;
      sc[2 * T + j] = tok < ntok ? c[T][j] * scale_log2 : kNegInf;
    }
}

// Scores of one page on the tensor cores (8-bit cache): sc[2T + j] is the
// base-2 score of head lane / 4 for token 8T + 2 (lane % 4) + j (-inf past
// the page's end).  kb: the page's codes of this kv head (token 0); ksc: the
// page's key scales of this kv head (token 0; stride n_kv).  The product is
// S^T = K Q^T per 8-token tile with m16n8k16: rows the heads (q in A, rows
// G.. zero), columns the tokens, the reduction head_dim; lane (r, t) takes
// its k-steps from head_dim chunk [t D/4, (t + 1) D/4) so that one 32-bit
// word of codes is one k-step.
template <int D, int NKV, uint32_t ROW>
__device__ __forceinline__ void qk_scores_mma(const unsigned char* kb, const float* ksc,
                                              int ntok, const uint32_t (&qa)[D / 16][2],
                                              float (&sc)[4], int lane) {
  const int g = lane >> 2, t = lane & 3;
  float c[2][4];
#pragma unroll
  for (int T = 0; T < 2; ++T) {
#pragma unroll
    for (int e = 0; e < 4; ++e) c[T][e] = 0.f;
    // this lane's D/4 codes of token 8T + g
    const unsigned char* src = kb + (8 * T + g) * ROW + t * (D / 4);
    uint32_t w[D / 16];
#pragma unroll
    for (int v = 0; v < D / 64; ++v) {
      const uint4 x = *reinterpret_cast<const uint4*>(src + 16 * v);
      w[4 * v] = x.x, w[4 * v + 1] = x.y, w[4 * v + 2] = x.z, w[4 * v + 3] = x.w;
    }
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks)
    {
      uint32_t b0, b1;
      f16x2x2_from_e4m3x4(w[ks], b0, b1);
      mma_f16_16816(c[T], qa[ks][0], qa[ks][1], b0, b1);
    }
  }
#pragma unroll
  for (int T = 0; T < 2; ++T)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int tok = 8 * T + 2 * t + j;
      sc[2 * T + j] = tok < ntok ? c[T][j] * ksc[tok * NKV] : kNegInf;
    }
}

// p * V of one page for one PV warp: vb points at this lane's 16-byte piece of
// its first token's value row, pp at p[tok_lane][0] of the page's hand-off
// (bf16 cache).
template <int D, int G, int LPT, uint32_t ROW, bool FULL>
__device__ __forceinline__ void pv_accumulate(const unsigned char* vb, const float* pp, int ntok,
                                              int tok_lane,
                                              float2 (&acc)[G][4]) {
  constexpr int TPI = 32 / LPT;
  constexpr int NIT = kBlock / TPI;
#pragma unroll
  for (int it = 0; it < NIT; ++it) {
    if (FULL || it * TPI + tok_lane < ntok) {
      float2 v2[4];
      const uint4 vw = *reinterpret_cast<const uint4*>(vb + it * TPI * ROW);
      v2[0] = bf16x2_to_float2(vw.x), v2[1] = bf16x2_to_float2(vw.y);
      v2[2] = bf16x2_to_float2(vw.z), v2[3] = bf16x2_to_float2(vw.w);
      float pr[G];
      if constexpr (G % 4 == 0) {
#pragma unroll
        for (int h = 0; h < G; h += 4) {
          const float4 x = *reinterpret_cast<const float4*>(pp + it * TPI * G + h);
          pr[h] = x.x, pr[h + 1] = x.y, pr[h + 2] = x.z, pr[h + 3] = x.w;
        }
      } else {
#pragma unroll
        for (int h = 0; h < G; ++h) pr[h] = pp[it * TPI * G + h];
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
#pragma unroll
        for (int h = 0; h < G; ++h)
          acc[h][e] = __ffma2_rn(v2[e], make_float2(pr[h], pr[h]), acc[h][e]);
      }
    }
  }
}

// Threads of a decode CTA: MW (tensor-core warps) with a bf16 cache runs one
// warp per kv head, every other form two.
template <int NKV, bool F8, bool MW>
__host__ __device__ constexpr int decode_threads() {
  return (MW && !F8 ? 1 : 2) * NKV * 32;
}

// D: head_dim; G: q heads per kv head; NKV: kv heads.  F8: 8-bit cache;
// FUSE: decode-only step with the scatter done here (bf16); MW: the page's
// arithmetic on the tensor cores by one warp (always with F8).
//  * MW: a warp computes q . k, the softmax and p * V of a page for all G
//    heads of its kv head, p staying in registers.  With a bf16 cache warp g
//    serves kv head g and takes every page; with the 8-bit cache warps g and
//    NKV + g take the even and the odd pages.
//  * otherwise: warps 0..NKV-1 compute scores and the softmax (QK warps),
//    warps NKV..2*NKV-1 accumulate p * V (PV warps) on the FMA pipe; warp g
//    and warp NKV + g serve kv head g and hand over p through a
//    double-buffered slot in shared memory.
template <int D, int G, int NKV, bool F8, bool FUSE, bool MW>
__global__ void __launch_bounds__(decode_threads<NKV, F8, MW>(), 1)
    decode_kernel(const DecodeParams p) {
  constexpr bool MMA = F8 || MW;
  constexpr int R = F8 ? 2 : 1;  // tensor-core warps per kv head
  constexpr int NW = decode_threads<NKV, F8, MW>() / 32;
  // QK lanes: E_QK head_dim elements each (two 16-byte pieces when 16)
  constexpr int E_QK = (G <= 4 && D == 128) ? 16 : 8;
  constexpr int LPT_QK = D / E_QK;
  constexpr int TPI_QK = 32 / LPT_QK;
  constexpr int NIT_QK = kBlock / TPI_QK;
  constexpr int REP_QK = LPT_QK / G;
  // PV lanes: 8 elements (16 bytes) each
  constexpr int LPT_PV = D / 8;
  constexpr uint32_t ES = F8 ? 1 : 2;      // bytes per cached element
  constexpr uint32_t ROW = NKV * D * ES;  // bytes of one token row in a page
  static_assert(LPT_QK >= G && LPT_QK % G == 0, "group too large for the lane split");

  extern __shared__ __align__(128) unsigned char smem_raw[];
  using Smem = DecodeSmem<G, NKV>;
  unsigned char* stages = smem_raw;
  Smem& S = *reinterpret_cast<Smem*>(smem_raw + (size_t)p.nstages * p.stage_bytes);
  Comb<G, D>* comb = reinterpret_cast<Comb<G, D>*>(
      smem_raw + (size_t)p.nstages * p.stage_bytes + comb_offset<G, NKV>());
  __shared__ long long red[NW];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = p.ctas;
  const int c = blockIdx.x;
  const int NST = p.nstages;
  // the merge kernel waits for this whole grid anyway; let it be scheduled
  asm volatile("griddepcontrol.launch_dependents;");

  // ---------------------------------------------------------------- plan
  // pass 1: total decode pages F (all threads)
  long long mine = 0;
  for (int s = threadIdx.x; s < p.num_seqs; s += blockDim.x)
    mine += decode_pages(p, s, c == 0);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
  if (lane == 0) red[warp] = mine;
  __syncthreads();
  long long F = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) F += red[w];
  const int64_t f0 = slice_begin(c, F, C), f1 = slice_begin(c + 1, F, C);
  const int n_pages = (int)(f1 - f0);
  if (n_pages <= 0) return;  // uniform: the whole CTA leaves
  if (MMA && R == 2 && (NST & 1)) {  // see the stage count in the launcher
    if (threadIdx.x == 0) flag_error(p.err, DEVERR_BOUNDS);
    return;  // uniform
  }

  // pass 2: locate the request holding flat page f0 (warp 0), start the ring
  if (warp == 0) {
    long long run = 0;
    int found_s = -1, found_j = 0;
    for (int base = 0; base < p.num_seqs && found_s < 0; base += 32) {
      const int s = base + lane;
      const int np = s < p.num_seqs ? decode_pages(p, s, false) : 0;
      long long incl = np;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const long long excl = run + incl - np;
      const bool hit = np > 0 && f0 >= excl && f0 < excl + np;
      const unsigned ball = __ballot_sync(0xffffffffu, hit);
      if (ball) {
        const int src = __ffs(ball) - 1;
        found_s = base + src;
        found_j = (int)(f0 - __shfl_sync(0xffffffffu, excl, src));
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      S.plan[0] = found_s;
      S.plan[1] = found_j;
      S.abort_flag = 0;
      for (int i = 0; i < NST; ++i) {
        mbar_init(smem_addr(&S.full[i]), 1);
        S.released[i] = 0;
        S.last_issued[i] = -1;
        S.fused_slot[i] = -1;
      }
      for (int g = 0; g < NKV; ++g)
        for (int b = 0; b < 2; ++b) {
          mbar_init(smem_addr(&S.p_full[g][b]), 1);
          mbar_init(smem_addr(&S.p_empty[g][b]), 1);
        }
      fence_mbar_init();
    }
    __syncwarp();
    // the slice's first NST pages, one lane each: each copy waits for two
    // dependent table loads, which then overlap instead of queueing
    if (found_s >= 0 && lane < NST && lane < n_pages) {
      PageCursor fc{found_s, found_j, decode_pages(p, found_s, false)};
      for (int i = 0; i < lane; ++i) fc.next(p);
      fetch_page<FUSE, F8>(p, fc, smem_addr(stages + (size_t)lane * p.stage_bytes),
                           smem_addr(&S.full[lane]), &S.fused_slot[lane]);
      S.last_issued[lane] = lane;
    }
  }
  __syncthreads();
  const int s_begin = S.plan[0];
  const int j_begin = S.plan[1];
  if (s_begin < 0) return;  // cannot happen when n_pages > 0
  volatile int* abort_flag = &S.abort_flag;

  const bool is_qk = warp < NKV;
  const int g = is_qk ? warp : warp - NKV;  // kv head served by this warp
  PageCursor cur{s_begin, j_begin, decode_pages(p, s_begin, false)};
  PageCursor fc = cur;  // page to fetch when this warp is the last to release a stage
  for (int i = 0; i < NST; ++i) fc.next(p);

  int L = __ldg(p.seq_lens + cur.s);
  int seg_j0 = j_begin;

  if constexpr (MMA) {
    // ================================================== tensor-core warps
    // The score fragment of the q * k product (head r = lane / 4, tokens 2t,
    // 2t + 1, 2t + 8, 2t + 9 with t = lane % 4) is exactly the B fragment of
    // the p * V product, so p stays in registers.  With the 8-bit cache the
    // odd-page warp of a kv head hands its running state to the even-page
    // warp through shared memory at the end of each segment (a request's
    // pages in this CTA), which merges and writes.
    //
    // p * V is O^T [D x heads] += V^T [D x 16 tokens] * P^T [16 tokens x heads]
    // (mma.sync m16n8k16, f32 accumulate; f16 for codes, bf16 for a bf16
    // cache): MMA rows are head_dim, columns heads (G..7 unused), the
    // reduction the page's tokens.  Rows are assigned so that lane r reads one
    // contiguous run of D/8 elements per token: in tile pair q the first tile
    // holds d = r D/8 + 4q + {0, 1} in rows (r, r + 8), the second d + {2, 3};
    // accumulator o[2q + u][c] is element r D/8 + 4q + 2u + (c >> 1) of head
    // 2t + (c & 1).
    const int rho = (R == 1 || is_qk) ? 0 : 1;  // page parity served (8-bit cache)
    const int r = lane >> 2, t = lane & 3;
    constexpr uint32_t ESZ = F8 ? 1 : 2;
    constexpr int VW = D / 8 * ESZ / 4;  // 4-byte words per lane and token of p * V
    constexpr float OUT_SCALE = F8 ? 1.f / 512.f : 1.f;
    uint32_t qa[D / 16][2];  // A registers of q for head r (see qk_scores_mma)
    float o[D / 16][4];
    float m_run = kNegInf, l_lane = 0.f;
    bool stored = false;  // this lane issued fused-scatter stores
    auto load_q = [&](int seq) {
      const int tok = __ldg(p.qsl + seq);
      const uint16_t* qrow = p.q + ((int64_t)tok * p.n_q + g * G + (r < G ? r : 0)) * D;
#pragma unroll
      for (int v = 0; v < D / 32; ++v) {  // D/4 elements, 8 per load
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (r < G) w = __ldg(reinterpret_cast<const uint4*>(qrow + t * (D / 4) + 8 * v));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; e += 2) {  // 4 elements = one k-step
          if constexpr (F8) {
            const float2 f0 = bf16x2_to_float2(ws[e]), f1 = bf16x2_to_float2(ws[e + 1]);
            qa[2 * v + e / 2][0] = f16x2_from_floats(f0.x * p.scale_log2, f0.y * p.scale_log2);
            qa[2 * v + e / 2][1] = f16x2_from_floats(f1.x * p.scale_log2, f1.y * p.scale_log2);
          } else {
            qa[2 * v + e / 2][0] = ws[e];
            qa[2 * v + e / 2][1] = ws[e + 1];
          }
        }
      }
    };
    load_q(cur.s);
#pragma unroll
    for (int m = 0; m < D / 16; ++m)
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) o[m][cc] = 0.f;
    Comb<G, D>& cb = comb[g];  // 8-bit cache only
    int st = 0, st_phase = 0;
    const unsigned char* stage = stages;
    for (int i = 0; i < n_pages; ++i) {
      const bool seq_done = (cur.j + 1 == cur.np);
      const bool seg_end = seq_done || (i + 1 == n_pages);
      if (R == 1 || (i & 1) == rho) {
        // Page i (phase-parity wait: the stage must be at page i or past
        // it, never at page i - NST).  A stage's pages are i, i + NST, ...;
        // with R == 1 this warp reads every one of them, with R == 2 they
        // all have this warp's parity because NST is even (refused above
        // otherwise), so this warp waited for page i - NST itself.  Page
        // i + NST is copied only after every reader, this warp among them,
        // released page i.
        mbar_wait(smem_addr(&S.full[st]), st_phase, p.err, abort_flag);
        const int ntok = min(kBlock, L - cur.j * kBlock);
        const int fslot = FUSE ? S.fused_slot[st] : -1;
        if (FUSE && fslot >= 0 && lane == 0) {
          // fused scatter: this kv head's slices of the new key and value rows
          bulk_s2g(reinterpret_cast<unsigned char*>(const_cast<void*>(p.k_cache)) +
                       (size_t)fslot * ROW + g * D * ES,
                   smem_addr(stage + (ntok - 1) * ROW + g * D * ES), D * ES);
          bulk_s2g(reinterpret_cast<unsigned char*>(const_cast<void*>(p.v_cache)) +
                       (size_t)fslot * ROW + g * D * ES,
                   smem_addr(stage + p.page_bytes + (ntok - 1) * ROW + g * D * ES), D * ES);
          bulk_commit();
          stored = true;
        }
        // Scores from the key codes; value codes of tokens 2t, 2t + 1, 2t + 8,
        // 2t + 9 at lane r's D/8 head_dim offsets, and their scales, for p * V
        // (rows past the page's end hold stale codes whose p is 0, but a stale
        // NaN code would still poison the sum: read token 0 instead).  The
        // stage is released after p * V: releasing it earlier, with the codes
        // held in registers, measured slower (the loads' latency is then
        // exposed instead of overlapping the arithmetic).
        float sc4[4];
        if constexpr (F8)
          qk_scores_mma<D, NKV, ROW>(
              stage + g * D, reinterpret_cast<const float*>(stage + kBlock * ROW + g * 4),
              ntok, qa, sc4, lane);
        else
          qk_scores_mma_bf16<D, ROW>(stage + g * D * ES, ntok, qa, p.scale_log2, sc4, lane);
        // online softmax (base 2) of head r: its 16 scores sit in lanes 4r .. 4r + 3
        float mx = fmaxf(fmaxf(sc4[0], sc4[1]), fmaxf(sc4[2], sc4[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run, mx);
        const float m_use = (m_new == kNegInf) ? 0.f : m_new;
        const float alpha = fast_exp2(m_run - m_use);
        uint32_t x[4][VW];
        float vs[4];
        {
          const unsigned char* vb = stage + p.page_bytes + (g * D + r * (D / 8)) * ES;
          const float* vsc =
              reinterpret_cast<const float*>(stage + p.page_bytes + kBlock * ROW + g * 4);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int tok = 2 * t + (k & 1) + 8 * (k >> 1);
            const unsigned char* src = vb + (tok < ntok ? tok : 0) * ROW;
            if constexpr (VW % 4 == 0) {
#pragma unroll
              for (int v = 0; v < VW / 4; ++v) {
                const uint4 w = *reinterpret_cast<const uint4*>(src + 16 * v);
                x[k][4 * v] = w.x, x[k][4 * v + 1] = w.y, x[k][4 * v + 2] = w.z,
                x[k][4 * v + 3] = w.w;
              }
            } else {
              const uint2 w = *reinterpret_cast<const uint2*>(src);
              x[k][0] = w.x, x[k][1] = w.y;
            }
            vs[k] = F8 ? vsc[tok * NKV] : 1.f;
          }
        }
        float pv[4];
        float lsum = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int tok = 2 * t + (k & 1) + 8 * (k >> 1);
          float pr = fast_exp2(sc4[k] - m_use);  // 0 past the page's end
          // bf16 cache: p enters p * V in bf16, so the sum takes the same
          // rounded value (numerator and denominator stay consistent)
          if constexpr (!F8) pr = __uint_as_float(pack_bf16x2(pr, 0.f) << 16);
          lsum += pr;
          // B = P^T; for codes times the token's value scale and 2^9, which
          // keeps the product in f16's normal range for row maxima from about
          // 1e-3 to 5e4 (the 2^9 comes out exactly when the result is written)
          pv[k] = tok < ntok ? (F8 ? pr * (vs[k] * 512.f) : pr) : 0.f;
        }
        l_lane = l_lane * alpha + lsum;
        m_run = m_new;
        // the accumulator columns are heads 2t, 2t + 1: their rescale factors
        // live in lanes 8t and 8t + 4
        // (skipped when no head's running max moved, the common case)
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * t);
          const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * t + 4);
#pragma unroll
          for (int m = 0; m < D / 16; ++m) {
            o[m][0] *= a0, o[m][1] *= a1, o[m][2] *= a0, o[m][3] *= a1;
          }
        }
        if constexpr (!F8) {
          // A = V^T from the bf16 values in x: words 2q, 2q + 1 of a token
          // are its elements d, d + 1 and d + 2, d + 3 of tile pair q
          const uint32_t b0 = pack_bf16x2(pv[0], pv[1]);
          const uint32_t b1 = pack_bf16x2(pv[2], pv[3]);
#pragma unroll
          for (int q = 0; q < D / 32; ++q) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const uint32_t wa = x[0][2 * q + u], wb = x[1][2 * q + u];
              const uint32_t wc = x[2][2 * q + u], wd = x[3][2 * q + u];
              uint32_t a0, a1, a2, a3;
              asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(a0) : "r"(wa), "r"(wb));
              asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(a1) : "r"(wa), "r"(wb));
              asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(a2) : "r"(wc), "r"(wd));
              asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(a3) : "r"(wc), "r"(wd));
              mma_bf16_16816(o[2 * q + u], a0, a1, a2, a3, b0, b1);
            }
          }
        } else {
        const uint32_t b0 = f16x2_from_floats(pv[0], pv[1]);
        const uint32_t b1 = f16x2_from_floats(pv[2], pv[3]);
        // A = V^T from the value codes in x
#pragma unroll
        for (int q = 0; q < D / 32; ++q) {
          const uint32_t w0 = x[0][q], w1 = x[1][q];
          const uint32_t w2 = x[2][q], w3 = x[3][q];
          // (token 2t, token 2t + 1) code pairs of d + 0 | d + 1, and d + 2 | d + 3
          uint32_t lo01, hi01, lo23, hi23;
          asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(lo01) : "r"(w0), "r"(w1));
          asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(hi01) : "r"(w0), "r"(w1));
          asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(lo23) : "r"(w2), "r"(w3));
          asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(hi23) : "r"(w2), "r"(w3));
          uint32_t a[2][4];
          f16x2x2_from_e4m3x4(lo01, a[0][0], a[0][1]);
          f16x2x2_from_e4m3x4(lo23, a[0][2], a[0][3]);
          f16x2x2_from_e4m3x4(hi01, a[1][0], a[1][1]);
          f16x2x2_from_e4m3x4(hi23, a[1][2], a[1][3]);
          mma_f16_16816_full(o[2 * q], a[0][0], a[0][1], a[0][2], a[0][3], b0, b1);
          mma_f16_16816_full(o[2 * q + 1], a[1][0], a[1][1], a[1][2], a[1][3], b0, b1);
        }
        }
        __syncwarp();
        if (lane == 0) {
          if (FUSE && fslot >= 0) bulk_wait_read();  // the stores have read the stage
          // release the stage; the last of the NKV warps of this parity refills it
          if (atomicAdd(&S.released[st], 1) == NKV - 1) {
            S.released[st] = 0;
            if (i + NST < n_pages && !*abort_flag) {
              fetch_page<FUSE, F8>(p, fc, smem_addr(stage), smem_addr(&S.full[st]),
                               &S.fused_slot[st]);
              S.last_issued[st] = i + NST;
            }
          }
        }
      }
      if (lane == 0) fc.next(p);
      stage += p.stage_bytes;
      if (++st == NST) st = 0, st_phase ^= 1, stage = stages;
      if (seg_end) {
        // running sum of head r over its four lanes
        float lt = l_lane;
        lt += __shfl_xor_sync(0xffffffffu, lt, 1);
        lt += __shfl_xor_sync(0xffffffffu, lt, 2);
        // running max and sum of the accumulator columns' heads 2t, 2t + 1
        // (lanes 8t and 8t + 4 hold them)
        float mh[2], lh[2];
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          mh[cc] = __shfl_sync(0xffffffffu, m_run, 8 * t + 4 * cc);
          lh[cc] = __shfl_sync(0xffffffffu, lt, 8 * t + 4 * cc);
        }
        if (R == 2 && t == 0 && r < G) {
          cb.m[rho][r] = m_run;
          cb.l[rho][r] = lt;
        }
        if (R == 2 && rho == 1) {
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int h = 2 * t + cc;
            if (h >= G) continue;
#pragma unroll
            for (int m = 0; m < D / 16; ++m) {
              const int d = r * (D / 8) + 4 * (m >> 1) + 2 * (m & 1);
              *reinterpret_cast<float2*>(&cb.o[h][d]) = make_float2(o[m][cc], o[m][2 + cc]);
            }
          }
        }
        if (R == 2) named_barrier_sync(1 + g, 64);  // the pair's state is in shared memory
        if (rho == 0) {
          const int tok = __ldg(p.qsl + cur.s);
          const bool whole = (seg_j0 == 0) && seq_done;
          const int slot = 2 * c + (cur.s == s_begin ? 0 : 1);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int h = 2 * t + cc;
            if (h >= G) continue;
            const int qh = g * G + h;
            // 8-bit cache: merge the even-page (this warp) and odd-page states
            // of head h; a warp with no page in the segment has m = -inf,
            // l = 0, o = 0
            float mm = mh[cc], s0 = 1.f, s1 = 0.f, l_all = lh[cc];
            if constexpr (R == 2) {
              const float m0 = cb.m[0][h], m1 = cb.m[1][h];
              mm = fmaxf(m0, m1);
              s0 = fast_exp2(m0 - mm), s1 = fast_exp2(m1 - mm);
              l_all = cb.l[0][h] * s0 + cb.l[1][h] * s1;
            }
            const float inv = 1.f / l_all;
#pragma unroll
            for (int m = 0; m < D / 16; ++m) {
              const int d = r * (D / 8) + 4 * (m >> 1) + 2 * (m & 1);
              float2 w = make_float2(0.f, 0.f);
              if constexpr (R == 2) w = *reinterpret_cast<const float2*>(&cb.o[h][d]);
              // elements d, d + 1 (for codes the 2^9 of B taken out, exact)
              const float v0 = (o[m][cc] * s0 + w.x * s1) * OUT_SCALE;
              const float v1 = (o[m][2 + cc] * s0 + w.y * s1) * OUT_SCALE;
              if (whole) {
                *reinterpret_cast<uint32_t*>(p.out + ((int64_t)tok * p.n_q + qh) * D + d) =
                    pack_bf16x2(v0 * inv, v1 * inv);
              } else {
                *reinterpret_cast<float2*>(p.part_o + ((int64_t)slot * p.n_q + qh) * D + d) =
                    make_float2(v0, v1);
              }
            }
            if (!whole && r == 0) {
              p.part_ml[((int64_t)slot * p.n_q + qh) * 2 + 0] = mm;
              p.part_ml[((int64_t)slot * p.n_q + qh) * 2 + 1] = l_all;
            }
          }
          if (g == 0 && lane == 0 && seg_j0 == 0) {
            // this CTA owns the request's first page: record where its pieces are
            int c_last = c;
            if (!seq_done) {
              const int64_t f_last = f0 + i + (cur.np - 1 - cur.j);
              const int64_t cl = ((f_last + 1) * C + F - 1) / F - 1;
              c_last = (int)(cl < C - 1 ? cl : C - 1);
            }
            p.seq_rec[cur.s] = make_int4(c, c_last, slot, (int)F);
          }
        }
        if (R == 2) named_barrier_sync(1 + g, 64);  // the state buffer may be rewritten
#pragma unroll
        for (int m = 0; m < D / 16; ++m)
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) o[m][cc] = 0.f;
        m_run = kNegInf;
        l_lane = 0.f;
      }
      const int prev_s = cur.s;
      cur.next(p);
      if (seg_end && cur.s != prev_s && i + 1 < n_pages) {
        L = __ldg(p.seq_lens + cur.s);
        seg_j0 = 0;
        load_q(cur.s);
      }
    }
    if (FUSE && stored) bulk_wait_all();  // the stores are complete before the CTA exits
  } else {
  if (is_qk) {
    // ================================================================ QK warp
    const int tok_lane = lane / LPT_QK;
    const int dl = lane % LPT_QK;
    const int my_h = dl / REP_QK;
    const int rep = dl % REP_QK;
    float2 qf[G][E_QK / 2];  // bf16 cache: this lane's slice of q, fp32
    float m_run = kNegInf, l_lane = 0.f;
    bool stored = false;  // this lane issued fused-scatter stores
    auto load_q = [&](int seq) {
      const int tok = __ldg(p.qsl + seq);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const uint16_t* qrow = p.q + ((int64_t)tok * p.n_q + g * G + h) * D;
#pragma unroll
        for (int piece = 0; piece < E_QK / 8; ++piece) {
          const uint4 w =
              __ldg(reinterpret_cast<const uint4*>(qrow + piece * (D / 2) + dl * 8));
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = bf16x2_to_float2(ws[e]);
            qf[h][piece * 4 + e] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
          }
        }
      }
      m_run = kNegInf;
      l_lane = 0.f;
    };
    load_q(cur.s);
    // this lane's piece of its first token's key row, relative to a stage
    const uint32_t k_off = (uint32_t)(g * D * ES + dl * 8 * ES) + (uint32_t)tok_lane * ROW;
    int st = 0, st_phase = 0;
    const unsigned char* stage = stages;
    for (int i = 0; i < n_pages; ++i) {
      const int b = i & 1;
      // p buffer b freed by the PV warp after page i - 2: this warp waited
      // for the release of page i - 4 on it, and the release of page i needs
      // the p this warp writes next
      if (i >= 2) mbar_wait(smem_addr(&S.p_empty[g][b]), ((i >> 1) - 1) & 1, p.err, abort_flag);
      // page i: every warp reads every page, so this warp waited for page
      // i - NST of the stage; page i + NST is copied after all release page i
      mbar_wait(smem_addr(&S.full[st]), st_phase, p.err, abort_flag);
      const int ntok = min(kBlock, L - cur.j * kBlock);
      const int fslot = FUSE ? S.fused_slot[st] : -1;
      if (FUSE && fslot >= 0 && lane == 0) {
        // fused scatter: this kv head's slice of the new key row to its slot
        bulk_s2g(reinterpret_cast<unsigned char*>(const_cast<void*>(p.k_cache)) +
                     (size_t)fslot * ROW + g * D * ES,
                 smem_addr(stage + (ntok - 1) * ROW + g * D * ES), D * ES);
        bulk_commit();
        stored = true;
      }
      const bool seq_done = (cur.j + 1 == cur.np);
      const bool seg_end = seq_done || (i + 1 == n_pages);
      PBuf<G>& pb = S.pb[g][b];
      float sc[NIT_QK];
      if (ntok == kBlock)
        qk_scores<D, G, E_QK, LPT_QK, ROW, true>(stage + k_off, ntok, tok_lane, qf, sc, lane);
      else
        qk_scores<D, G, E_QK, LPT_QK, ROW, false>(stage + k_off, ntok, tok_lane, qf, sc, lane);
      // online softmax (base 2) for head my_h over the page's 16 tokens
      float mx = sc[0];
#pragma unroll
      for (int it = 1; it < NIT_QK; ++it) mx = fmaxf(mx, sc[it]);
#pragma unroll
      for (int m = LPT_QK; m < 32; m <<= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
      const float m_new = fmaxf(m_run, mx);
      const float m_use = (m_new == kNegInf) ? 0.f : m_new;
      const float alpha = fast_exp2(m_run - m_use);
      float* pw = &pb.p[tok_lane][my_h];
      float lsum = 0.f;
#pragma unroll
      for (int it = 0; it < NIT_QK; ++it) {
        const float pr = fast_exp2(sc[it] - m_use);
        lsum += pr;
        if (rep == 0) pw[it * TPI_QK * G] = pr;
      }
      l_lane = l_lane * alpha + lsum;
      m_run = m_new;
      if (tok_lane == 0 && rep == 0) pb.alpha[my_h] = alpha;
      if (seg_end) {
        float lt = l_lane;
#pragma unroll
        for (int m = LPT_QK; m < 32; m <<= 1) lt += __shfl_xor_sync(0xffffffffu, lt, m);
        if (tok_lane == 0 && rep == 0) {
          pb.m[my_h] = m_run;
          pb.l[my_h] = lt;
        }
      }
      __syncwarp();
      if (lane == 0) {
        if (FUSE && fslot >= 0) bulk_wait_read();  // the store has read the stage
        mbar_arrive(smem_addr(&S.p_full[g][b]));
        // release the stage; the last warp out refills it NST pages ahead
        if (atomicAdd(&S.released[st], 1) == NW - 1) {
          S.released[st] = 0;
          if (i + NST < n_pages && !*abort_flag) {
            fetch_page<FUSE, F8>(p, fc, smem_addr(stage), smem_addr(&S.full[st]),
                             &S.fused_slot[st]);
            S.last_issued[st] = i + NST;
          }
        }
        fc.next(p);
      }
      stage += p.stage_bytes;
      if (++st == NST) st = 0, st_phase ^= 1, stage = stages;
      const int prev_s = cur.s;
      cur.next(p);
      if (seg_end && cur.s != prev_s && i + 1 < n_pages) {
        L = __ldg(p.seq_lens + cur.s);
        load_q(cur.s);
      }
    }
    if (FUSE && stored) bulk_wait_all();  // the stores are complete before the CTA exits
  } else {
    // ================================================================ PV warp
    const int tok_lane = lane / LPT_PV;
    const int dl = lane % LPT_PV;
    float2 acc[G][4];
    bool stored = false;  // this lane issued fused-scatter stores
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[h][e] = make_float2(0.f, 0.f);
    // this lane's piece of its first token's value row, relative to a stage
    const uint32_t v_off =
        p.page_bytes + (uint32_t)(g * D * ES + dl * 8 * ES) + (uint32_t)tok_lane * ROW;
    int st = 0, st_phase = 0;
    const unsigned char* stage = stages;
    for (int i = 0; i < n_pages; ++i) {
      const int b = i & 1;
      // page i: as for the QK warps (every warp reads every page)
      mbar_wait(smem_addr(&S.full[st]), st_phase, p.err, abort_flag);
      const int ntok = min(kBlock, L - cur.j * kBlock);
      const int fslot = FUSE ? S.fused_slot[st] : -1;
      if (FUSE && fslot >= 0 && lane == 0) {
        // fused scatter: this kv head's slice of the new value row to its slot
        bulk_s2g(reinterpret_cast<unsigned char*>(const_cast<void*>(p.v_cache)) +
                     (size_t)fslot * ROW + g * D * ES,
                 smem_addr(stage + p.page_bytes + (ntok - 1) * ROW + g * D * ES), D * ES);
        bulk_commit();
        stored = true;
      }
      // p of page i: this warp waited for page i - 2's on buffer b, and the
      // QK warp writes page i + 2's only after this warp frees b (p_empty)
      mbar_wait(smem_addr(&S.p_full[g][b]), (i >> 1) & 1, p.err, abort_flag);
      const PBuf<G>& pb = S.pb[g][b];
      const uint32_t pb_addr = smem_addr(&pb);
      float al[G];
      lds_floats<G>(pb_addr + offsetof(PBuf<G>, alpha), al);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float2 a2 = make_float2(al[h], al[h]);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[h][e] = __fmul2_rn(acc[h][e], a2);
      }
      const float* pp = &pb.p[tok_lane][0];
      if (ntok == kBlock)
        pv_accumulate<D, G, LPT_PV, ROW, true>(stage + v_off, pp, ntok, tok_lane, acc);
      else
        pv_accumulate<D, G, LPT_PV, ROW, false>(stage + v_off, pp, ntok, tok_lane, acc);
      const bool seq_done = (cur.j + 1 == cur.np);
      const bool seg_end = seq_done || (i + 1 == n_pages);
      float m_fin[G], l_fin[G];
      if (seg_end) {
        lds_floats<G>(pb_addr + offsetof(PBuf<G>, m), m_fin);
        lds_floats<G>(pb_addr + offsetof(PBuf<G>, l), l_fin);
      }
      __syncwarp();
      if (lane == 0) {
        if (FUSE && fslot >= 0) bulk_wait_read();  // the store has read the stage
        mbar_arrive(smem_addr(&S.p_empty[g][b]));
        if (atomicAdd(&S.released[st], 1) == NW - 1) {
          S.released[st] = 0;
          if (i + NST < n_pages && !*abort_flag) {
            fetch_page<FUSE, F8>(p, fc, smem_addr(stage), smem_addr(&S.full[st]),
                             &S.fused_slot[st]);
            S.last_issued[st] = i + NST;
          }
        }
        fc.next(p);
      }
      stage += p.stage_bytes;
      if (++st == NST) st = 0, st_phase ^= 1, stage = stages;
      if (seg_end) {
        // sum over the token lanes of the warp
#pragma unroll
        for (int m = LPT_PV; m < 32; m <<= 1)
#pragma unroll
          for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              acc[h][e].x += __shfl_xor_sync(0xffffffffu, acc[h][e].x, m);
              acc[h][e].y += __shfl_xor_sync(0xffffffffu, acc[h][e].y, m);
            }
        if (tok_lane == 0) {
          const int tok = __ldg(p.qsl + cur.s);
          const bool whole = (seg_j0 == 0) && seq_done;
          const int slot = 2 * c + (cur.s == s_begin ? 0 : 1);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const int qh = g * G + h;
            if (whole) {
              const float inv = 1.f / l_fin[h];
              uint4 w;
              w.x = pack_bf16x2(acc[h][0].x * inv, acc[h][0].y * inv);
              w.y = pack_bf16x2(acc[h][1].x * inv, acc[h][1].y * inv);
              w.z = pack_bf16x2(acc[h][2].x * inv, acc[h][2].y * inv);
              w.w = pack_bf16x2(acc[h][3].x * inv, acc[h][3].y * inv);
              *reinterpret_cast<uint4*>(p.out + ((int64_t)tok * p.n_q + qh) * D + dl * 8) = w;
            } else {
              float4* dst = reinterpret_cast<float4*>(
                  p.part_o + ((int64_t)slot * p.n_q + qh) * D + dl * 8);
              dst[0] = make_float4(acc[h][0].x, acc[h][0].y, acc[h][1].x, acc[h][1].y);
              dst[1] = make_float4(acc[h][2].x, acc[h][2].y, acc[h][3].x, acc[h][3].y);
              if (dl == 0) {
                p.part_ml[((int64_t)slot * p.n_q + qh) * 2 + 0] = m_fin[h];
                p.part_ml[((int64_t)slot * p.n_q + qh) * 2 + 1] = l_fin[h];
              }
            }
          }
          if (g == 0 && lane == 0 && seg_j0 == 0) {
            // this CTA owns the request's first page: record where its pieces are
            int c_last = c;
            if (!seq_done) {
              const int64_t f_last = f0 + i + (cur.np - 1 - cur.j);
              const int64_t cl = ((f_last + 1) * C + F - 1) / F - 1;
              c_last = (int)(cl < C - 1 ? cl : C - 1);
            }
            p.seq_rec[cur.s] = make_int4(c, c_last, slot, (int)F);
          }
        }
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[h][e] = make_float2(0.f, 0.f);
      }
      const int prev_s = cur.s;
      cur.next(p);
      if (seg_end && cur.s != prev_s && i + 1 < n_pages) {
        L = __ldg(p.seq_lens + cur.s);
        seg_j0 = 0;
      }
    }
    if (FUSE && stored) bulk_wait_all();  // the stores are complete before the CTA exits
  }
  }
  // never hand back shared memory with a copy still landing in it: the
  // last page copied into each stage (the one before it was read, and so
  // complete, before this copy was issued; nothing is copied after it)
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int st = 0; st < NST; ++st) {
      const int i = S.last_issued[st];
      if (i < 0) continue;
      const uint32_t full = smem_addr(&S.full[st]);
      const unsigned long long t0 = global_ns();
      while (!mbar_try_wait(full, (i / NST) & 1)) {
        if (global_ns() - t0 > kWaitLimitNs) {
          flag_error(p.err, DEVERR_TIMEOUT);
          break;
        }
      }
    }
  }
}

// Combine the pieces of every decode request that spans several CTAs, eight
// pieces' loads in flight at a time.  Two shapes, chosen on the host from the
// number of requests per CTA of the decode grid:
//  * SPLIT = false (many requests, a few pieces each): a warp per (request,
//    q head), kMergeWarps heads per CTA;
//  * SPLIT = true (few long requests, up to a piece per decode CTA each): a
//    CTA per (request, q head) whose warps take every kMergeWarps-th piece,
//    then warp 0 combines the warps' partial results.
// Lanes own 4 consecutive elements of head_dim.  Launched as a programmatic
// dependent of the decode kernel: it may start while the decode grid drains
// and waits for it before reading partials.
constexpr int kMergeWarps = 4;
// Up to this many sequences the merge finds a request's pieces from the
// call's inputs before waiting for the decode grid (each warp reads them all,
// eight per lane); past it, it reads the record the decode kernel wrote.
constexpr int kMergeScanMax = 256;

template <int D, bool SPLIT>
__global__ void __launch_bounds__(kMergeWarps * 32) decode_merge_kernel(const DecodeParams p) {
  __shared__ float w_m[kMergeWarps], w_l[kMergeWarps];
  __shared__ float4 w_o[kMergeWarps][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.x;
  const int h = SPLIT ? (int)blockIdx.y : (int)blockIdx.y * kMergeWarps + warp;
  if (!SPLIT && h >= p.n_q) return;
  // the request's shape and output row come from the call's inputs, which
  // are complete before the decode grid starts: read them before waiting for
  // it (with SPLIT every early return below is the same for the whole CTA)
  const int np_s = decode_pages(p, s, false);
  if (np_s == 0) return;  // not a (valid) decode request
  const int a_row = __ldg(p.qsl + s);
  const int C = p.ctas;
  int c_first, c_last, first_slot;
  int64_t F;
  if (p.num_seqs <= kMergeScanMax) {
    // where the request's pieces are follows from the same inputs: its pages
    // are flat pages fa .. fa + np_s - 1 of the F pages the decode grid cuts
    // into slices, so they are known before the wait, and a request whole in
    // one slice leaves without waiting at all
    long long tot = 0, before = 0;
#pragma unroll
    for (int i = 0; i < kMergeScanMax / 32; ++i) {  // all loads in flight at once
      const int s2 = lane + 32 * i;
      const int n = s2 < p.num_seqs ? decode_pages(p, s2, false) : 0;
      tot += n;
      if (s2 < s) before += n;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      tot += __shfl_xor_sync(0xffffffffu, tot, o);
      before += __shfl_xor_sync(0xffffffffu, before, o);
    }
    F = tot;
    const int64_t fa = before, fb = before + np_s - 1;
    // the CTA whose slice holds flat page f: the last c with slice_begin(c) <= f
    auto owner = [&](int64_t f) {
      const int64_t c = ((f + 1) * C + F - 1) / F - 1;
      return (int)(c < C - 1 ? c : C - 1);
    };
    c_first = owner(fa);
    c_last = owner(fb);
    // the first CTA wrote its piece to its first slot when its slice starts
    // with this request, else to its second (as the decode kernel chooses)
    first_slot = 2 * c_first + (slice_begin(c_first, F, C) == fa ? 0 : 1);
    if (c_first == c_last) return;  // written directly by the decode kernel
    asm volatile("griddepcontrol.wait;" ::: "memory");
  } else {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int4 rec = p.seq_rec[s];
    c_first = rec.x, c_last = rec.y, first_slot = rec.z;
    F = rec.w;
    if (c_first == c_last) return;  // written directly by the decode kernel
  }
  if (c_first < 0 || c_last >= C || c_first > c_last || first_slot < 0 || first_slot >= 2 * C ||
      F <= 0) {
    if (threadIdx.x == 0) flag_error(p.err, DEVERR_BOUNDS);
    return;
  }
  // with at least as many pages as CTAs no slice is empty (skip the divisions)
  const bool may_be_empty = F < C;
  const bool active = lane * 4 < D;
  float M = kNegInf, Lsum = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int STEP = SPLIT ? kMergeWarps : 1;  // piece stride of this warp
  for (int cc0 = c_first + (SPLIT ? warp : 0); cc0 <= c_last; cc0 += 8 * STEP) {
    float2 ml[8];
    float4 o[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int cc = cc0 + k * STEP;
      const bool v = cc <= c_last &&
                     (!may_be_empty || slice_begin(cc, F, C) != slice_begin(cc + 1, F, C));
      const int slot = (cc == c_first) ? first_slot : 2 * cc;
      ml[k] = make_float2(kNegInf, 0.f);
      o[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (v) {
        ml[k] = __ldg(reinterpret_cast<const float2*>(p.part_ml) + (int64_t)slot * p.n_q + h);
        if (active)
          o[k] = __ldg(reinterpret_cast<const float4*>(
              p.part_o + ((int64_t)slot * p.n_q + h) * D + lane * 4));
      }
    }
    float bm = M;
#pragma unroll
    for (int k = 0; k < 8; ++k) bm = fmaxf(bm, ml[k].x);
    const float mu = (bm == kNegInf) ? 0.f : bm;
    const float f = fast_exp2(M - mu);
    Lsum *= f;
    O.x *= f, O.y *= f, O.z *= f, O.w *= f;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float w = fast_exp2(ml[k].x - mu);
      Lsum += ml[k].y * w;
      O.x += o[k].x * w, O.y += o[k].y * w, O.z += o[k].z * w, O.w += o[k].w * w;
    }
    M = bm;
  }
  if constexpr (!SPLIT) {
    if (active) {
      const float inv = 1.f / Lsum;
      uint2 wv;
      wv.x = pack_bf16x2(O.x * inv, O.y * inv);
      wv.y = pack_bf16x2(O.z * inv, O.w * inv);
      *reinterpret_cast<uint2*>(p.out + ((int64_t)a_row * p.n_q + h) * D + lane * 4) = wv;
    }
    return;
  }
  if (lane == 0) w_m[warp] = M, w_l[warp] = Lsum;
  w_o[warp][lane] = O;
  __syncthreads();
  if (warp != 0) return;
  float bm = kNegInf;
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) bm = fmaxf(bm, w_m[w]);
  const float mu = (bm == kNegInf) ? 0.f : bm;
  float Lt = 0.f;
  float4 Ot = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int w = 0; w < kMergeWarps; ++w) {
    const float f = fast_exp2(w_m[w] - mu);
    const float4 ow = w_o[w][lane];
    Lt += w_l[w] * f;
    Ot.x += ow.x * f, Ot.y += ow.y * f, Ot.z += ow.z * f, Ot.w += ow.w * f;
  }
  if (active) {
    const float inv = 1.f / Lt;
    uint2 wv;
    wv.x = pack_bf16x2(Ot.x * inv, Ot.y * inv);
    wv.y = pack_bf16x2(Ot.z * inv, Ot.w * inv);
    *reinterpret_cast<uint2*>(p.out + ((int64_t)a_row * p.n_q + h) * D + lane * 4) = wv;
  }
}

constexpr size_t kSmemBudget = 220 * 1024;
constexpr size_t kSmemBudgetF8 = 226 * 1024;  // below the 227 KB opt-in limit per block

template <int D, int G, int NKV, bool F8, bool FUSE, bool MW>
cudaError_t launch_decode_t(const AttnArgs& a, const DecodeWorkspace& ws, int ctas,
                            cudaStream_t stream) {
  DecodeParams p;
  p.q = a.q;
  p.k_cache = a.k_cache;
  p.v_cache = a.v_cache;
  p.k_new = a.fuse_k_new;
  p.v_new = a.fuse_v_new;
  p.slot_mapping = a.fuse_slot_mapping;
  p.block_tables = a.block_tables;
  p.seq_lens = a.seq_lens;
  p.qsl = a.query_start_loc;
  p.out = a.out;
  p.part_o = ws.part_o;
  p.part_ml = ws.part_ml;
  p.seq_rec = ws.seq_rec;
  p.err = a.err;
  p.num_blocks = a.num_blocks;
  p.max_blocks = a.max_blocks;
  p.num_seqs = a.num_seqs;
  p.num_tokens = a.num_tokens;
  p.n_q = a.num_q_heads;
  p.n_kv = a.num_kv_heads;
  p.max_seq_len = a.max_seq_len;
  p.block_shift = a.block_shift;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.ctas = ctas;
  p.row_bytes = (uint32_t)NKV * D * (F8 ? 1 : 2);
  p.page_bytes = F8 ? (uint32_t)fp8_page_bytes(NKV, D) : kBlock * p.row_bytes;
  p.stage_bytes = 2 * p.page_bytes;
  // the 8-bit kernel also holds the per-kv-head merge buffers, and takes
  // the shared memory up to the opt-in limit to keep six stages
  const size_t fixed =
      F8 ? comb_offset<G, NKV>() + NKV * sizeof(Comb<G, D>) : sizeof(DecodeSmem<G, NKV>);
  const size_t budget = F8 ? kSmemBudgetF8 : kSmemBudget;
  int nst = (int)((budget - fixed) / p.stage_bytes);
  nst = nst > 8 ? 8 : nst;
  // The 8-bit kernel's two warps per kv head take alternate pages and wait
  // only on their own pages' stages.  With an odd stage count a stage would
  // hold pages of both parities in turn, so a warp could wait on a barrier
  // two phases ahead, where the phase-parity wait cannot tell the phase it
  // wants from the one before it; an even count keeps each stage to one
  // parity (the kernel refuses an odd count).
  if (F8) nst &= ~1;
  if (nst < 2) return cudaErrorInvalidConfiguration;
  p.nstages = nst;
  const size_t smem = (size_t)nst * p.stage_bytes + fixed;
  auto kern = decode_kernel<D, G, NKV, F8, FUSE, MW>;
  constexpr int threads = decode_threads<NKV, F8, MW>();
  static int configured_device = -1;  // one attribute set per process and device
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(F8 ? kSmemBudgetF8 : kSmemBudget + 4096));
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  cudaError_t e;
  if (a.after_prefill) {
    // overlaps the prefill grid (no data dependence: different output rows,
    // and the cache writes of the step finished before the prefill started)
    cudaLaunchConfig_t pcfg = {};
    pcfg.gridDim = dim3(ctas);
    pcfg.blockDim = dim3(threads);
    pcfg.dynamicSmemBytes = smem;
    pcfg.stream = stream;
    cudaLaunchAttribute pattr[1];
    pattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    pattr[0].val.programmaticStreamSerializationAllowed = 1;
    pcfg.attrs = pattr;
    pcfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&pcfg, kern, p);
  } else {
    kern<<<ctas, threads, smem, stream>>>(p);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  // a request spans about ctas / num_seqs + 1 CTAs: with eight or more, split
  // each request's pieces over a CTA's warps
  const bool split = ctas >= 8 * a.num_seqs;
  cfg.gridDim = split ? dim3(a.num_seqs, a.num_q_heads, 1)
                      : dim3(a.num_seqs, (a.num_q_heads + kMergeWarps - 1) / kMergeWarps, 1);
  cfg.blockDim = dim3(kMergeWarps * 32, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return split ? cudaLaunchKernelEx(&cfg, decode_merge_kernel<D, true>, p)
               : cudaLaunchKernelEx(&cfg, decode_merge_kernel<D, false>, p);
}

// Tensor-core warps for the 8-bit cache always; for a bf16 cache when the
// group is 8 (the FMA form's accumulators do not fit its registers there).
template <bool F8, int G>
constexpr bool decode_uses_mma() {
  return F8 || G == 8;
}

template <int D, int G, bool F8, bool FUSE>
cudaError_t launch_decode_dg(const AttnArgs& a, const DecodeWorkspace& ws, int ctas,
                             cudaStream_t stream) {
  constexpr bool MW = decode_uses_mma<F8, G>();
  switch (a.num_kv_heads) {
    case 1: return launch_decode_t<D, G, 1, F8, FUSE, MW>(a, ws, ctas, stream);
    case 2: return launch_decode_t<D, G, 2, F8, FUSE, MW>(a, ws, ctas, stream);
    case 4: return launch_decode_t<D, G, 4, F8, FUSE, MW>(a, ws, ctas, stream);
    case 8: return launch_decode_t<D, G, 8, F8, FUSE, MW>(a, ws, ctas, stream);
  }
  return cudaErrorInvalidValue;
}

template <bool F8, bool FUSE>
cudaError_t launch_decode_any(const AttnArgs& a, const DecodeWorkspace& ws, int ctas,
                              cudaStream_t stream) {
  const int group = a.num_q_heads / a.num_kv_heads;
  if (a.head_dim == 128) {
    if (group == 1) return launch_decode_dg<128, 1, F8, FUSE>(a, ws, ctas, stream);
    if (group == 2) return launch_decode_dg<128, 2, F8, FUSE>(a, ws, ctas, stream);
    if (group == 4) return launch_decode_dg<128, 4, F8, FUSE>(a, ws, ctas, stream);
    if (group == 8) return launch_decode_dg<128, 8, F8, FUSE>(a, ws, ctas, stream);
  } else if (a.head_dim == 64) {
    if (group == 1) return launch_decode_dg<64, 1, F8, FUSE>(a, ws, ctas, stream);
    if (group == 2) return launch_decode_dg<64, 2, F8, FUSE>(a, ws, ctas, stream);
    if (group == 4) return launch_decode_dg<64, 4, F8, FUSE>(a, ws, ctas, stream);
    if (group == 8) return launch_decode_dg<64, 8, F8, FUSE>(a, ws, ctas, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace pa
