// pa_decode.cu -- split-KV decode attention over the paged KV cache, and the
// log-sum-exp merge of the splits.
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
//  * A page of the cache ([16 tokens][num_kv_heads][head_dim] bf16) is one
//    contiguous block of memory, so K and V pages are fetched whole with one
//    bulk asynchronous copy each into a ring of shared-memory stages, issued
//    by a producer warp and tracked by mbarriers: several pages per SM are in
//    flight at once, which is what keeps HBM busy.
//  * Each consumer warp owns one kv head (and a slice of the page's tokens)
//    and all q heads of its GQA group, so every K/V byte is read from HBM
//    once.  Lanes hold a 16-byte slice of head_dim; q.k is reduced with
//    warp shuffles that also spread the group's heads across lanes.
//  * Online softmax per page in base 2 (q is pre-scaled by scale * log2 e),
//    fp32 accumulation with packed fp32x2 FMAs.
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
  const uint16_t* k_cache;
  const uint16_t* v_cache;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* qsl;
  uint16_t* out;
  float* part_o;
  float* part_ml;
  int4* seq_rec;
  unsigned* err;
  int32_t num_blocks, max_blocks, num_seqs, num_tokens, n_q, n_kv, max_seq_len;
  float scale_log2;
  int32_t nstages;
  int32_t ctas;
  uint32_t stage_bytes;  // K page + V page
  uint32_t page_bytes;   // one K (or V) page: 16 * n_kv * head_dim * 2
  uint32_t row_bytes;    // one token row of one cache: n_kv * head_dim * 2
};

// Pages this kernel processes for request s (0 if it is not a decode request
// or is invalid; invalid ones flag the error word once, from CTA 0).
__device__ __forceinline__ int decode_pages(const DecodeParams& p, int s, bool report) {
  const int a = __ldg(p.qsl + s), b = __ldg(p.qsl + s + 1);
  if (b - a != 1) return 0;
  const int L = __ldg(p.seq_lens + s);
  if (L < 1 || L > p.max_seq_len || L > p.max_blocks * kBlock || a < 0 || a >= p.num_tokens) {
    if (report) flag_error(p.err, DEVERR_BOUNDS);
    return 0;
  }
  return (L + kBlock - 1) / kBlock;
}

__device__ __forceinline__ int64_t slice_begin(int64_t c, int64_t F, int64_t C) {
  return c * F / C;
}

// Shared-memory layout after the stage ring (dynamic shared memory).
template <int D, int G, int NW>
struct DecodeSmem {
  uint64_t full[8];      // stage holds its page (bulk-copy transaction count)
  int released[8];       // warps done with the page in the stage
  int last_issued[8];    // last page whose copies went into the stage (-1: none)
  float p_s[NW][kBlock][G];
  float alpha_s[NW][G];
  float seg_ml[NW][G][2];
  int plan[2];
  int abort_flag;
};

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

// Issue the bulk copies of page (c.s, c.j) into stage st.
__device__ __forceinline__ void fetch_page(const DecodeParams& p, const PageCursor& c,
                                           uint32_t stage_smem, uint32_t full_bar) {
  const int L = __ldg(p.seq_lens + c.s);
  const int ntok = min(kBlock, L - c.j * kBlock);
  const int phys = __ldg(p.block_tables + (int64_t)c.s * p.max_blocks + c.j);
  if (phys < 0 || phys >= p.num_blocks) {
    flag_error(p.err, DEVERR_BOUNDS);
    mbar_arrive_expect_tx(full_bar, 0);  // completes the phase with no data
    return;
  }
  const uint32_t bytes = (uint32_t)ntok * p.row_bytes;
  mbar_arrive_expect_tx(full_bar, 2 * bytes);
  const size_t off = (size_t)phys * p.page_bytes;
  bulk_g2s(stage_smem, reinterpret_cast<const unsigned char*>(p.k_cache) + off, bytes, full_bar);
  bulk_g2s(stage_smem + p.page_bytes, reinterpret_cast<const unsigned char*>(p.v_cache) + off,
           bytes, full_bar);
}

// D: head_dim; G: q heads per kv head; NW: warps; NSUB: warps per kv head
// (each takes 16 / NSUB tokens of every page), so num_kv_heads = NW / NSUB.
template <int D, int G, int NW, int NSUB>
__global__ void __launch_bounds__(NW * 32, 1) decode_kernel(const DecodeParams p) {
  constexpr int LPT = D / 8;          // lanes per token: each holds 8 elements = 16 bytes
  constexpr int TPI = 32 / LPT;       // tokens per warp iteration
  constexpr int TPS = kBlock / NSUB;  // tokens of a page per warp
  constexpr int NIT = (TPS + TPI - 1) / TPI;
  constexpr int REP = LPT / G;        // lanes that end up holding the same score
  static_assert(LPT >= G && LPT % G == 0, "group too large for the lane split");
  static_assert(NW % NSUB == 0, "warps must split evenly over kv heads");

  extern __shared__ __align__(128) unsigned char smem_raw[];
  using Smem = DecodeSmem<D, G, NW>;
  unsigned char* stages = smem_raw;
  Smem& S = *reinterpret_cast<Smem*>(smem_raw + (size_t)p.nstages * p.stage_bytes);
  // cross-warp buffer for the o of subsets 1.. of each kv head
  float* seg_o = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(&S) + sizeof(Smem));
  __shared__ long long red[NW];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = p.ctas;
  const int c = blockIdx.x;
  const int NST = p.nstages;

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
      }
      fence_mbar_init();
      if (found_s >= 0) {
        PageCursor fc{found_s, found_j, decode_pages(p, found_s, false)};
        for (int i = 0; i < NST && i < n_pages; ++i) {
          fetch_page(p, fc, smem_addr(stages + (size_t)i * p.stage_bytes),
                     smem_addr(&S.full[i]));
          S.last_issued[i] = i;
          fc.next(p);
        }
      }
    }
  }
  __syncthreads();
  const int s_begin = S.plan[0];
  const int j_begin = S.plan[1];
  if (s_begin < 0) return;  // cannot happen when n_pages > 0
  volatile int* abort_flag = &S.abort_flag;

  // ---------------------------------------------------------------- main loop
  const int n_kv = NW / NSUB;
  const int g = warp % n_kv;   // kv head
  const int sub = warp / n_kv; // token subset of the page
  const int tok_lane = lane / LPT;
  const int dl = lane % LPT;
  const int my_h = dl / REP;   // head whose score this lane holds after the reduce-scatter
  const int rep = dl % REP;

  float2 qf[G][4];
  float2 acc[G][4];
  float m_run = kNegInf, l_run = 0.f;

  PageCursor cur{s_begin, j_begin, decode_pages(p, s_begin, false)};
  PageCursor fc = cur;  // page to fetch when this warp is the last to release a stage
  for (int i = 0; i < NST; ++i) fc.next(p);
  int seg_j0 = j_begin;

  auto load_q = [&](int seq) {
    const int tok = __ldg(p.qsl + seq);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(
          p.q + ((int64_t)tok * p.n_q + g * G + h) * D + dl * 8));
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = bf16x2_to_float2(ws[e]);
        qf[h][e] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
        acc[h][e] = make_float2(0.f, 0.f);
      }
    }
    m_run = kNegInf;
    l_run = 0.f;
  };

  load_q(cur.s);
  const uint32_t stage0 = smem_addr(stages);
  const uint32_t gh_off = (uint32_t)(g * D * 2 + dl * 16);

  for (int i = 0; i < n_pages; ++i) {
    const int st = i % NST;
    // A failed wait leaves the page's contents meaningless (the error word
    // says so) but the page is still processed: control flow must stay the
    // same in every warp because of the CTA barriers at segment ends.
    mbar_wait(smem_addr(&S.full[st]), (i / NST) & 1, p.err, abort_flag);
    const int L = __ldg(p.seq_lens + cur.s);
    const int ntok = min(kBlock, L - cur.j * kBlock);
    const uint32_t kst = stage0 + (uint32_t)st * p.stage_bytes;
    const uint32_t vst = kst + p.page_bytes;

    // ---- scores of this warp's tokens, one (token, head) per lane
    float sc[NIT];
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
      const int tl = it * TPI + tok_lane;  // token index within the subset
      const int t = sub * TPS + tl;
      const bool valid = tl < TPS && t < ntok;
      uint4 kw = make_uint4(0, 0, 0, 0);
      if (valid) kw = lds128(kst + (uint32_t)t * p.row_bytes + gh_off);
      const uint32_t ks[4] = {kw.x, kw.y, kw.z, kw.w};
      float part[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float2 a = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 4; ++e) a = __ffma2_rn(qf[h][e], bf16x2_to_float2(ks[e]), a);
        part[h] = a.x + a.y;
      }
      // reduce-scatter over the LPT lanes of the token: each halving step
      // hands half of the remaining heads to the partner lane
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
      sc[it] = valid ? part[0] : kNegInf;
    }
    // ---- online softmax update (base 2) for head my_h
    float mx = kNegInf;
#pragma unroll
    for (int it = 0; it < NIT; ++it) mx = fmaxf(mx, sc[it]);
#pragma unroll
    for (int m = LPT; m < 32; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
    const float m_new = fmaxf(m_run, mx);
    const float m_use = (m_new == kNegInf) ? 0.f : m_new;
    const float alpha = fast_exp2(m_run - m_use);
    float lsum = 0.f;
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
      const float pr = fast_exp2(sc[it] - m_use);
      lsum += pr;
      const int tl = it * TPI + tok_lane;
      if (rep == 0 && tl < TPS) S.p_s[warp][tl][my_h] = pr;
    }
    l_run = l_run * alpha + lsum;
    m_run = m_new;
    if (tok_lane == 0 && rep == 0) S.alpha_s[warp][my_h] = alpha;
    __syncwarp();

    // ---- rescale, then accumulate p * v
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float a = S.alpha_s[warp][h];
      const float2 a2 = make_float2(a, a);
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[h][e] = __fmul2_rn(acc[h][e], a2);
    }
#pragma unroll
    for (int it = 0; it < NIT; ++it) {
      const int tl = it * TPI + tok_lane;
      const int t = sub * TPS + tl;
      if (tl < TPS && t < ntok) {
        const uint4 vw = lds128(vst + (uint32_t)t * p.row_bytes + gh_off);
        const uint32_t vs[4] = {vw.x, vw.y, vw.z, vw.w};
        float pr[G];
#pragma unroll
        for (int h = 0; h < G; ++h) pr[h] = S.p_s[warp][tl][h];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 v2 = bf16x2_to_float2(vs[e]);
#pragma unroll
          for (int h = 0; h < G; ++h)
            acc[h][e] = __ffma2_rn(v2, make_float2(pr[h], pr[h]), acc[h][e]);
        }
      }
    }
    __syncwarp();
    // ---- release the stage; the last warp out refills it NST pages ahead
    if (lane == 0) {
      const int before = atomicAdd(&S.released[st], 1);
      if (before == NW - 1) {
        S.released[st] = 0;
        // after a failed wait nothing more is issued: the stage's previous
        // copy may still be landing
        if (i + NST < n_pages && !*abort_flag) {
          fetch_page(p, fc, kst, smem_addr(&S.full[st]));
          S.last_issued[st] = i + NST;
        }
      }
      fc.next(p);
    }

    // ---- end of a segment: the request is finished, or this CTA's slice ends
    const bool seq_done = (cur.j + 1 == cur.np);
    const bool slice_done = (i + 1 == n_pages);
    if (seq_done || slice_done) {
      // sum over the token lanes of the warp
#pragma unroll
      for (int m = LPT; m < 32; m <<= 1) {
        l_run += __shfl_xor_sync(0xffffffffu, l_run, m);
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[h][e].x += __shfl_xor_sync(0xffffffffu, acc[h][e].x, m);
            acc[h][e].y += __shfl_xor_sync(0xffffffffu, acc[h][e].y, m);
          }
      }
      float m_fin[G], l_fin[G];
      if constexpr (NSUB > 1) {
        // combine the warps of each kv head through shared memory
        if (tok_lane == 0 && rep == 0) {
          S.seg_ml[warp][my_h][0] = m_run;
          S.seg_ml[warp][my_h][1] = l_run;
        }
        if (sub > 0 && tok_lane == 0) {
          float* dst = seg_o + ((size_t)(warp - n_kv) * G) * D + dl * 8;
#pragma unroll
          for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              dst[h * D + 2 * e] = acc[h][e].x;
              dst[h * D + 2 * e + 1] = acc[h][e].y;
            }
        }
        __syncthreads();
        if (sub == 0) {
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float mm = kNegInf;
#pragma unroll
            for (int u = 0; u < NSUB; ++u) mm = fmaxf(mm, S.seg_ml[u * n_kv + g][h][0]);
            const float mu = (mm == kNegInf) ? 0.f : mm;
            float ll = 0.f;
#pragma unroll
            for (int u = 0; u < NSUB; ++u)
              ll += S.seg_ml[u * n_kv + g][h][1] * fast_exp2(S.seg_ml[u * n_kv + g][h][0] - mu);
            const float w0s = fast_exp2(S.seg_ml[g][h][0] - mu);
            const float2 w0 = make_float2(w0s, w0s);
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[h][e] = __fmul2_rn(acc[h][e], w0);
#pragma unroll
            for (int u = 1; u < NSUB; ++u) {
              const float* src = seg_o + ((size_t)((u - 1) * n_kv + g) * G + h) * D + dl * 8;
              const float w = fast_exp2(S.seg_ml[u * n_kv + g][h][0] - mu);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                acc[h][e].x += src[2 * e] * w;
                acc[h][e].y += src[2 * e + 1] * w;
              }
            }
            m_fin[h] = mm;
            l_fin[h] = ll;
          }
        }
        __syncthreads();
      } else {
        // one warp per kv head: gather each head's (m, l) from its lanes
#pragma unroll
        for (int h = 0; h < G; ++h) {
          m_fin[h] = __shfl_sync(0xffffffffu, m_run, h * REP);
          l_fin[h] = __shfl_sync(0xffffffffu, l_run, h * REP);
        }
      }
      if (sub == 0 && tok_lane == 0) {
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
        if (warp == 0 && lane == 0 && seg_j0 == 0) {
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
      if (seq_done && !slice_done) {
        cur.next(p);
        seg_j0 = 0;
        load_q(cur.s);
        continue;
      }
    }
    cur.next(p);
  }

  // never hand back shared memory with a copy still landing in it
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

// Combine the pieces of every decode request that spans several CTAs.
template <int D>
__global__ void __launch_bounds__(256) decode_merge_kernel(const DecodeParams p) {
  const int s = blockIdx.x;
  const int a = __ldg(p.qsl + s);
  if (decode_pages(p, s, false) == 0) return;  // not a (valid) decode request
  const int4 rec = p.seq_rec[s];
  const int C = p.ctas;
  const int c_first = rec.x, c_last = rec.y, first_slot = rec.z;
  const int64_t F = rec.w;
  if (c_first == c_last) return;
  if (c_first < 0 || c_last >= C || c_first > c_last || first_slot < 0 || first_slot >= 2 * C ||
      F <= 0) {
    if (threadIdx.x == 0) flag_error(p.err, DEVERR_BOUNDS);
    return;
  }
  for (int idx = threadIdx.x; idx < p.n_q * D; idx += blockDim.x) {
    const int h = idx / D, e = idx % D;
    float M = kNegInf;
    for (int cc = c_first; cc <= c_last; ++cc) {
      if (slice_begin(cc, F, C) == slice_begin(cc + 1, F, C)) continue;
      const int slot = (cc == c_first) ? first_slot : 2 * cc;
      M = fmaxf(M, p.part_ml[((int64_t)slot * p.n_q + h) * 2]);
    }
    const float mu = (M == kNegInf) ? 0.f : M;
    float Lsum = 0.f, O = 0.f;
    for (int cc = c_first; cc <= c_last; ++cc) {
      if (slice_begin(cc, F, C) == slice_begin(cc + 1, F, C)) continue;
      const int slot = (cc == c_first) ? first_slot : 2 * cc;
      const float w = fast_exp2(p.part_ml[((int64_t)slot * p.n_q + h) * 2] - mu);
      Lsum += p.part_ml[((int64_t)slot * p.n_q + h) * 2 + 1] * w;
      O += p.part_o[((int64_t)slot * p.n_q + h) * D + e] * w;
    }
    p.out[((int64_t)a * p.n_q + h) * D + e] = float_to_bf16_rn(O / Lsum);
  }
}

template <int D, int G, int NW>
size_t decode_smem_bytes(int nstages, uint32_t stage_bytes, int n_kv) {
  const int nsub = NW / n_kv;
  return (size_t)nstages * stage_bytes + sizeof(DecodeSmem<D, G, NW>) +
         (size_t)(nsub - 1) * n_kv * G * D * sizeof(float);
}

constexpr int warps_for_group(int g) { return g <= 4 ? 16 : 8; }

constexpr size_t kSmemBudget = 220 * 1024;

template <int D, int G, int NW, int NSUB>
cudaError_t launch_decode_t(const AttnArgs& a, const DecodeWorkspace& ws, int ctas,
                            cudaStream_t stream) {
  DecodeParams p;
  p.q = a.q;
  p.k_cache = a.k_cache;
  p.v_cache = a.v_cache;
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
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.ctas = ctas;
  p.row_bytes = (uint32_t)a.num_kv_heads * D * 2;
  p.page_bytes = kBlock * p.row_bytes;
  p.stage_bytes = 2 * p.page_bytes;
  const size_t fixed = decode_smem_bytes<D, G, NW>(0, p.stage_bytes, a.num_kv_heads);
  int nst = (int)((kSmemBudget - fixed) / p.stage_bytes);
  nst = nst > 8 ? 8 : nst;
  if (nst < 2) return cudaErrorInvalidConfiguration;
  p.nstages = nst;
  const size_t smem = decode_smem_bytes<D, G, NW>(nst, p.stage_bytes, a.num_kv_heads);
  auto kern = decode_kernel<D, G, NW, NSUB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<ctas, NW * 32, smem, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  decode_merge_kernel<D><<<a.num_seqs, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

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
  if (num_kv_heads != 1 && num_kv_heads != 2 && num_kv_heads != 4 && num_kv_heads != 8)
    return false;
  return num_kv_heads * head_dim <= 1024;
}

template <int D, int G>
static cudaError_t launch_decode_dg(const AttnArgs& a, const DecodeWorkspace& ws, int ctas,
                                    cudaStream_t stream) {
  constexpr int NW = warps_for_group(G);
  switch (NW / a.num_kv_heads) {
    case 1: return launch_decode_t<D, G, NW, 1>(a, ws, ctas, stream);
    case 2: return launch_decode_t<D, G, NW, 2>(a, ws, ctas, stream);
    case 4: return launch_decode_t<D, G, NW, 4>(a, ws, ctas, stream);
    case 8: return launch_decode_t<D, G, NW, 8>(a, ws, ctas, stream);
    case 16:
      if constexpr (NW == 16) return launch_decode_t<D, G, NW, 16>(a, ws, ctas, stream);
      break;
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode(const AttnArgs& a, const DecodeWorkspace& ws, int ctas,
                          cudaStream_t stream) {
  const int group = a.num_q_heads / a.num_kv_heads;
  if (a.head_dim == 128) {
    if (group == 1) return launch_decode_dg<128, 1>(a, ws, ctas, stream);
    if (group == 2) return launch_decode_dg<128, 2>(a, ws, ctas, stream);
    if (group == 4) return launch_decode_dg<128, 4>(a, ws, ctas, stream);
    if (group == 8) return launch_decode_dg<128, 8>(a, ws, ctas, stream);
  } else if (a.head_dim == 64) {
    if (group == 1) return launch_decode_dg<64, 1>(a, ws, ctas, stream);
    if (group == 2) return launch_decode_dg<64, 2>(a, ws, ctas, stream);
    if (group == 4) return launch_decode_dg<64, 4>(a, ws, ctas, stream);
    if (group == 8) return launch_decode_dg<64, 8>(a, ws, ctas, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pa
