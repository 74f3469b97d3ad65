// pa_prefill.cu -- chunked-prefill attention over the paged KV cache on the
// tcgen05 tensor cores (requests with q_len >= 2).
//
// What it computes ("PagedAttention 显存分页与连续批处理(Continuous Batching)
// 实战", Chunked Prefill section: a long prompt is cut into fixed slices, each
// computed together with the running decodes; prefill is compute-bound and
// suits tensor-core GEMM; "连续批处理：推理吞吐的范式革命", section 4.1 for the
// attention itself): query row i of a request with q_len rows sits at position
// p = seq_len - q_len + i and attends to keys 0..p of its Block Table.
//
// Layout of the work (GB300 design, not the pages' scalar kernel):
//  * An item is (request, tile of 128/G query tokens, kv head g).  Its 128 MMA
//    rows are the tile's tokens x the G q heads that share kv head g, so every
//    K/V tile is loaded once for the whole GQA group.
//  * Warp 0 streams Q and K tiles, warp 6 V tiles, of 128 keys (8 pages of 16
//    tokens, one TMA box per page and 64-element half of head_dim, 128-byte
//    swizzle) into rings of shared-memory stages; separate K and V producers
//    let the next K tiles load while the V of earlier tiles is still in use.
//  * Warp 1 (one thread) issues tcgen05.mma: S = Q K^T into one of two TMEM
//    buffers, then O += P V into a TMEM accumulator.
//  * Warps 2-5 own one MMA row each: they read S from TMEM, apply the causal
//    mask and scale, keep the running max / sum (base 2), write P (bf16) back
//    over the S buffer in TMEM, where the P V MMA reads it as its A operand,
//    and rescale O in TMEM only when the max grows by more than 2^8 (exact: the
//    same reference max scales the numerator and the denominator).  At the end
//    they normalise O and store bf16 rows.
//  * Persistent CTAs (at most one per SM) walk the item list.
#include <cstdint>
#include <mutex>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int kBlock = 16;        // tokens per physical block
constexpr int kKeysPerTile = 128; // keys per K/V tile (8 blocks)
constexpr int kRows = 128;        // MMA rows (tokens x group heads)
constexpr int kStagesK = 3;       // K tile stages
constexpr int kStagesV = 3;       // V tile stages
constexpr float kNegInf = -INFINITY;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kThreads = 224;  // K/Q producer, MMA, 4 softmax, V producer

struct PrefillParams {
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* qsl;
  uint16_t* out;
  unsigned* err;
  int32_t num_blocks, max_blocks, num_seqs, num_tokens, n_q, n_kv, max_seq_len;
  float scale_log2;
};

// Query tiles of request s (0 unless it has q_len >= 2 and is valid).
template <int TM>
__device__ __forceinline__ int prefill_tiles(const PrefillParams& p, int s, bool report) {
  const int a = __ldg(p.qsl + s), b = __ldg(p.qsl + s + 1);
  const int ql = b - a;
  if (ql < 2) return 0;
  const int L = __ldg(p.seq_lens + s);
  if (L < ql || L > p.max_seq_len || L > p.max_blocks * kBlock || a < 0 || b > p.num_tokens) {
    if (report) flag_error(p.err, DEVERR_BOUNDS);
    return 0;
  }
  return (ql + TM - 1) / TM;
}

// Geometry of one item.
struct Item {
  int s, mt, g;
  int q0;         // first query token of the tile
  int ntok;       // valid query tokens in the tile
  int p_first;    // position of the first query token
  int kv_end;     // keys needed: 0 .. kv_end - 1
  int nkt;        // K/V tiles
};

// Walks the item list (request-major, then query tile, then kv head).
template <int TM>
struct ItemCursor {
  int s = 0, tile_base = 0, tiles = 0;
  __device__ __forceinline__ bool locate(const PrefillParams& p, long long item, Item& it) {
    const long long tile = item / p.n_kv;
    const int g = (int)(item % p.n_kv);
    while (s < p.num_seqs && tile >= (long long)tile_base + tiles) {
      tile_base += tiles;
      ++s;
      tiles = s < p.num_seqs ? prefill_tiles<TM>(p, s, false) : 0;
    }
    if (s >= p.num_seqs) return false;
    const int a = __ldg(p.qsl + s), b = __ldg(p.qsl + s + 1);
    const int L = __ldg(p.seq_lens + s);
    it.s = s;
    it.mt = (int)(tile - tile_base);
    it.g = g;
    it.q0 = a + it.mt * TM;
    it.ntok = min(TM, (b - a) - it.mt * TM);
    it.p_first = L - (b - a) + it.mt * TM;
    it.kv_end = it.p_first + it.ntok;
    it.nkt = (it.kv_end + kKeysPerTile - 1) / kKeysPerTile;
    return true;
  }
  __device__ __forceinline__ void init(const PrefillParams& p) {
    s = 0;
    tile_base = 0;
    tiles = p.num_seqs > 0 ? prefill_tiles<TM>(p, 0, false) : 0;
  }
};

struct PrefillBarriers {
  uint64_t q_full, q_empty;
  uint64_t k_full[kStagesK], k_empty[kStagesK];
  uint64_t v_full[kStagesV], v_empty[kStagesV];
  uint64_t s_full[2];
  uint64_t p_full[2], pv_done[2];
  uint64_t o_full, o_empty;
  uint64_t mma_done;
  uint32_t tmem_slot;
  int abort_flag;
  long long total_items;
};

// Byte offset of 16-byte chunk c (0..7) of row r inside a [rows][64 x bf16]
// block stored with the 128-byte swizzle (8-row, 1024-byte atoms).
__device__ __forceinline__ uint32_t sw128_chunk(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

template <int D, int G>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap) {
  constexpr int TM = kRows / G;       // query tokens per tile
  constexpr int NH = D / 64;          // 64-element halves of head_dim
  constexpr uint32_t HALF = kRows * 128;  // bytes of one [128 rows][64] block
  constexpr uint32_t Q_BYTES = NH * HALF;
  constexpr uint32_t KV_BYTES = NH * HALF;  // 128 keys
  constexpr uint32_t TMEM_COLS = 512;
  constexpr uint32_t S_COL0 = 0, O_COL = 256;
  constexpr uint32_t IDESC_S = tc::idesc_bf16_f32(kRows, kKeysPerTile, 0, 0);
  constexpr uint32_t IDESC_O = tc::idesc_bf16_f32(kRows, D, 0, 1);

  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* q_s = base;
  unsigned char* k_s = q_s + Q_BYTES;
  unsigned char* v_s = k_s + kStagesK * KV_BYTES;
  PrefillBarriers& B = *reinterpret_cast<PrefillBarriers*>(v_s + kStagesV * KV_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // decode rows of the same step may use the SMs this grid leaves free
  asm volatile("griddepcontrol.launch_dependents;");

  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&B.q_full), 1);
    mbar_init(smem_addr(&B.q_empty), 1);
    for (int i = 0; i < kStagesK; ++i) {
      mbar_init(smem_addr(&B.k_full[i]), 1);
      mbar_init(smem_addr(&B.k_empty[i]), 1);
    }
    for (int i = 0; i < kStagesV; ++i) {
      mbar_init(smem_addr(&B.v_full[i]), 1);
      mbar_init(smem_addr(&B.v_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&B.s_full[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(&B.p_full[i]), 4);
      mbar_init(smem_addr(&B.pv_done[i]), 1);
    }
    mbar_init(smem_addr(&B.o_full), 1);
    mbar_init(smem_addr(&B.o_empty), 4);
    mbar_init(smem_addr(&B.mma_done), 1);
    B.abort_flag = 0;
    fence_mbar_init();
    long long total = 0;
    for (int s = 0; s < p.num_seqs; ++s) total += prefill_tiles<TM>(p, s, blockIdx.x == 0);
    B.total_items = total * p.n_kv;
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_addr(&B.tmem_slot), TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = B.tmem_slot;
  const long long total_items = B.total_items;
  volatile int* abort_flag = &B.abort_flag;

  if (warp == 0 || warp == 6) {
    // ============================================================ producers
    if (lane == 0) {
      const bool is_k = (warp == 0);  // warp 0: Q and K, warp 6: V
      const CUtensorMap* map = is_k ? &kmap : &vmap;
      unsigned char* ring = is_k ? k_s : v_s;
      uint64_t* full = is_k ? B.k_full : B.v_full;
      uint64_t* empty = is_k ? B.k_empty : B.v_empty;
      const int nst = is_k ? kStagesK : kStagesV;
      ItemCursor<TM> cur;
      cur.init(p);
      int n_item = 0, c = 0;
      for (long long item = blockIdx.x; item < total_items; item += gridDim.x, ++n_item) {
        Item it;
        if (!cur.locate(p, item, it)) break;
        if (is_k) {
          if (n_item > 0) mbar_wait(smem_addr(&B.q_empty), (n_item - 1) & 1, p.err, abort_flag);
          mbar_arrive_expect_tx(smem_addr(&B.q_full), Q_BYTES);
#pragma unroll
          for (int h = 0; h < NH; ++h)
            tc::tma_load_3d(smem_addr(q_s + h * HALF), &qmap, h * 64, it.g * G, it.q0,
                            smem_addr(&B.q_full));
        }
        const int pages = (it.kv_end + kBlock - 1) / kBlock;
        const int32_t* table = p.block_tables + (int64_t)it.s * p.max_blocks;
        for (int kt = 0; kt < it.nkt; ++kt, ++c) {
          const int p0 = kt * (kKeysPerTile / kBlock);
          const int npg = min(kKeysPerTile / kBlock, pages - p0);
          int phys[kKeysPerTile / kBlock];
          int nvalid = 0;
          for (int i = 0; i < npg; ++i) {
            phys[i] = __ldg(table + p0 + i);
            if (phys[i] < 0 || phys[i] >= p.num_blocks) {
              flag_error(p.err, DEVERR_BOUNDS);
              phys[i] = -1;
            } else {
              ++nvalid;
            }
          }
          const int st = c % nst;
          if (c >= nst)
            mbar_wait(smem_addr(&empty[st]), ((c / nst) - 1) & 1, p.err, abort_flag);
          mbar_arrive_expect_tx(smem_addr(&full[st]),
                                (uint32_t)nvalid * NH * (kBlock * 128));
          for (int i = 0; i < npg; ++i) {
            if (phys[i] < 0) continue;
#pragma unroll
            for (int h = 0; h < NH; ++h)
              tc::tma_load_3d(smem_addr(ring + st * KV_BYTES + h * HALF + i * (kBlock * 128)),
                              map, h * 64, it.g, phys[i] * kBlock, smem_addr(&full[st]));
          }
        }
      }
      // never hand back shared memory with a TMA copy still landing in it
      for (int i = max(0, c - nst); i < c; ++i)
        mbar_wait(smem_addr(&full[i % nst]), (i / nst) & 1, p.err, abort_flag);
      if (is_k && n_item > 0)
        mbar_wait(smem_addr(&B.q_full), (n_item - 1) & 1, p.err, abort_flag);
    }
  } else if (warp == 1) {
    // ============================================================ MMA issuer
    if (lane == 0) {
      ItemCursor<TM> cur;
      cur.init(p);
      int n_item = 0;
      long long T = 0;  // K/V tiles so far (all items)
      const uint32_t q_addr = smem_addr(q_s);
      bool issued = false;
      for (long long item = blockIdx.x; item < total_items; item += gridDim.x, ++n_item) {
        Item it;
        if (!cur.locate(p, item, it)) break;
        mbar_wait(smem_addr(&B.q_full), n_item & 1, p.err, abort_flag);
        auto issue_pv = [&](long long t, bool first) {
          const int b = (int)(t & 1);
          mbar_wait(smem_addr(&B.p_full[b]), (int)((t >> 1) & 1), p.err, abort_flag);
          mbar_wait(smem_addr(&B.v_full[t % kStagesV]), (int)((t / kStagesV) & 1), p.err,
                    abort_flag);
          if (first && n_item > 0)
            mbar_wait(smem_addr(&B.o_empty), (n_item - 1) & 1, p.err, abort_flag);
          tc::fence_after_sync();
          // P (bf16, 64 packed columns) sits in the S buffer it came from
          const uint32_t pt = tmem + S_COL0 + b * kKeysPerTile;
          const uint32_t va = smem_addr(v_s + (t % kStagesV) * KV_BYTES);
#pragma unroll
          for (int kk = 0; kk < kKeysPerTile / 16; ++kk) {
            const uint64_t bd = tc::sw128_desc(va + kk * 2048, HALF, 1024);
            tc::mma_bf16_tmem_a(tmem + O_COL, pt + kk * 8, bd, IDESC_O,
                                (first && kk == 0) ? 0u : 1u);
          }
          tc::commit(smem_addr(&B.v_empty[t % kStagesV]));
          tc::commit(smem_addr(&B.pv_done[b]));
        };
        for (int kt = 0; kt < it.nkt; ++kt, ++T) {
          const int sb = (int)(T & 1);
          mbar_wait(smem_addr(&B.k_full[T % kStagesK]), (int)((T / kStagesK) & 1), p.err,
                    abort_flag);
          // buffer sb holds P of tile T - 2 until its PV has run
          if (T >= 2)
            mbar_wait(smem_addr(&B.pv_done[sb]), (int)(((T - 2) >> 1) & 1), p.err, abort_flag);
          tc::fence_after_sync();
          const uint32_t ka = smem_addr(k_s + (T % kStagesK) * KV_BYTES);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t ad =
                tc::sw128_desc(q_addr + (kk >> 2) * HALF + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = tc::sw128_desc(ka + (kk >> 2) * HALF + (kk & 3) * 32, 16, 1024);
            tc::mma_bf16(tmem + S_COL0 + sb * kKeysPerTile, ad, bd, IDESC_S, kk > 0 ? 1u : 0u);
          }
          tc::commit(smem_addr(&B.s_full[sb]));
          tc::commit(smem_addr(&B.k_empty[T % kStagesK]));
          if (kt == it.nkt - 1) tc::commit(smem_addr(&B.q_empty));
          if (kt > 0) issue_pv(T - 1, kt == 1);
          issued = true;
        }
        issue_pv(T - 1, it.nkt == 1);
        tc::commit(smem_addr(&B.o_full));
      }
      if (issued) {
        tc::commit(smem_addr(&B.mma_done));
        mbar_wait(smem_addr(&B.mma_done), 0, p.err, abort_flag);
      }
    }
  } else {
    // ============================================================ softmax
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const int tl = r / G, hl = r % G;
    ItemCursor<TM> cur;
    cur.init(p);
    int n_item = 0;
    long long T = 0;
    for (long long item = blockIdx.x; item < total_items; item += gridDim.x, ++n_item) {
      Item it;
      if (!cur.locate(p, item, it)) break;
      const bool row_valid = tl < it.ntok;
      const int p_row = row_valid ? it.p_first + tl : it.kv_end - 1;
      float m_ref = kNegInf, l = 0.f;
      for (int kt = 0; kt < it.nkt; ++kt, ++T) {
        const int sb = (int)(T & 1);
        mbar_wait(smem_addr(&B.s_full[sb]), (int)((T >> 1) & 1), p.err, abort_flag);
        tc::fence_after_sync();
        uint32_t sr[kKeysPerTile];
#pragma unroll
        for (int c = 0; c < kKeysPerTile / 32; ++c)
          tc::tmem_ld32(tmem + lane_addr + S_COL0 + sb * kKeysPerTile + c * 32,
                        *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
        tc::tmem_wait_ld();

        // causal mask, tile max (8 independent chains).  With a positive
        // scale the max of the raw scores gives the max of the scaled ones,
        // and the scale folds into the exponent's FMA below.
        const int k0 = kt * kKeysPerTile;
        const int lim = p_row - k0;  // keys c <= lim are visible
        const float sl2 = p.scale_log2;
        const bool pos_scale = sl2 > 0.f;
        const float mul = pos_scale ? 1.f : sl2;  // applied now; sl2 is applied in the exp
        const float emul = pos_scale ? sl2 : 1.f;
        float m8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) m8[j] = kNegInf;
        if (__all_sync(0xffffffffu, lim >= kKeysPerTile - 1)) {
          if (!pos_scale) {
#pragma unroll
            for (int c = 0; c < kKeysPerTile; ++c)
              sr[c] = __float_as_uint(__uint_as_float(sr[c]) * mul);
          }
#pragma unroll
          for (int c = 0; c < kKeysPerTile; ++c) m8[c & 7] = fmaxf(m8[c & 7], __uint_as_float(sr[c]));
        } else {
#pragma unroll
          for (int c = 0; c < kKeysPerTile; ++c) {
            const float s = (c <= lim) ? __uint_as_float(sr[c]) * mul : kNegInf;
            sr[c] = __float_as_uint(s);
            m8[c & 7] = fmaxf(m8[c & 7], s);
          }
        }
        float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                         fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        mx = (mx == kNegInf) ? kNegInf : mx * emul;  // now in scaled base-2 units
        float alpha = 1.f;
        if (m_ref == kNegInf) {
          m_ref = mx;  // first tile: O not yet written
        } else if (mx > m_ref + kRescaleThreshold) {
          alpha = fast_exp2(m_ref - mx);
          l *= alpha;
          m_ref = mx;
        }
        // p = 2^(emul * s - m_ref), packed in bf16 pairs in place (sr[j] holds
        // keys 2j, 2j+1), then stored over the S buffer's first 64 columns
        const float nm = -m_ref;
        float l8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) l8[j] = 0.f;
#pragma unroll
        for (int j = 0; j < kKeysPerTile / 2; ++j) {
          const float p0 = fast_exp2(fmaf(__uint_as_float(sr[2 * j]), emul, nm));
          const float p1 = fast_exp2(fmaf(__uint_as_float(sr[2 * j + 1]), emul, nm));
          l8[(2 * j) & 7] += p0;
          l8[(2 * j + 1) & 7] += p1;
          sr[j] = pack_bf16x2(p0, p1);
        }
        tc::tmem_st32(tmem + lane_addr + S_COL0 + sb * kKeysPerTile,
                      *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tc::tmem_st32(tmem + lane_addr + S_COL0 + sb * kKeysPerTile + 32,
                      *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        l += ((l8[0] + l8[1]) + (l8[2] + l8[3])) + ((l8[4] + l8[5]) + (l8[6] + l8[7]));
        // rescale the running output when the reference max moved (rare)
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          mbar_wait(smem_addr(&B.pv_done[(T - 1) & 1]), (int)(((T - 1) >> 1) & 1), p.err,
                    abort_flag);
          tc::fence_after_sync();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tc::tmem_ld32(tmem + lane_addr + O_COL + c * 32, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tc::tmem_st32(tmem + lane_addr + O_COL + c * 32, o);
          }
          tc::tmem_wait_st();
        }
        // keys past the last needed one: V rows there may hold stale or
        // poisoned data; zero them so that P = 0 times V stays 0
        const int kv_local = it.kv_end - k0;
        if (kv_local < kKeysPerTile) {
          mbar_wait(smem_addr(&B.v_full[T % kStagesV]), (int)((T / kStagesV) & 1), p.err,
                    abort_flag);
          if (r >= kv_local) {
            unsigned char* vrow = v_s + (T % kStagesV) * KV_BYTES;
#pragma unroll
            for (int h = 0; h < NH; ++h)
#pragma unroll
              for (int c8 = 0; c8 < 8; ++c8)
                *reinterpret_cast<uint4*>(vrow + h * HALF + sw128_chunk(r, c8)) =
                    make_uint4(0, 0, 0, 0);
          }
        }
        tc::tmem_wait_st();
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&B.p_full[sb]));
      }
      // epilogue: O / l -> bf16 rows
      mbar_wait(smem_addr(&B.o_full), n_item & 1, p.err, abort_flag);
      tc::fence_after_sync();
      const float inv = 1.f / l;
      uint16_t* orow = p.out + ((int64_t)(it.q0 + tl) * p.n_q + it.g * G + hl) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tc::tmem_ld32(tmem + lane_addr + O_COL + c * 32, o);
        tc::tmem_wait_ld();
        if (row_valid) {
#pragma unroll
          for (int j = 0; j < 32; j += 8) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(o[j + 4]) * inv, __uint_as_float(o[j + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(o[j + 6]) * inv, __uint_as_float(o[j + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + c * 32 + j) = w;
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&B.o_empty));
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// 3-D bf16 map {inner, mid, outer} with a {64, box_mid, box_outer} box and
// the 128-byte swizzle.
cudaError_t make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t mid,
                     uint64_t outer, uint32_t box_mid, uint32_t box_outer) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {inner, mid, outer};
  const cuuint64_t strides[2] = {inner * 2, inner * mid * 2};
  const cuuint32_t box[3] = {64, box_mid, box_outer};
  const cuuint32_t es[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                         strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, int G>
size_t prefill_smem_bytes() {
  constexpr size_t half = kRows * 128;
  return 1024 + (size_t)(D / 64) * half * (1 + kStagesK + kStagesV) +
         sizeof(PrefillBarriers);
}

template <int D, int G>
cudaError_t launch_prefill_t(const AttnArgs& a, int sm_count, cudaStream_t stream) {
  constexpr int TM = kRows / G;
  PrefillParams p;
  p.block_tables = a.block_tables;
  p.seq_lens = a.seq_lens;
  p.qsl = a.query_start_loc;
  p.out = a.out;
  p.err = a.err;
  p.num_blocks = a.num_blocks;
  p.max_blocks = a.max_blocks;
  p.num_seqs = a.num_seqs;
  p.num_tokens = a.num_tokens;
  p.n_q = a.num_q_heads;
  p.n_kv = a.num_kv_heads;
  p.max_seq_len = a.max_seq_len;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  CUtensorMap qm, km, vm;
  cudaError_t e = make_map(&qm, a.q, D, a.num_q_heads, a.num_tokens, G, TM);
  if (e != cudaSuccess) return e;
  e = make_map(&km, a.k_cache, D, a.num_kv_heads, (uint64_t)a.num_blocks * kBlock, 1, kBlock);
  if (e != cudaSuccess) return e;
  e = make_map(&vm, a.v_cache, D, a.num_kv_heads, (uint64_t)a.num_blocks * kBlock, 1, kBlock);
  if (e != cudaSuccess) return e;
  // upper bound of the number of items; the kernel reads the exact count
  const long long tiles_bound = (long long)a.num_tokens / TM + a.num_seqs;
  long long items_bound = tiles_bound * a.num_kv_heads;
  const int grid = (int)(items_bound < sm_count ? items_bound : sm_count);
  if (grid <= 0) return cudaSuccess;
  const size_t smem = prefill_smem_bytes<D, G>();
  auto kern = prefill_kernel<D, G>;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  kern<<<grid, kThreads, smem, stream>>>(p, qm, km, vm);
  return cudaGetLastError();
}

}  // namespace

bool prefill_supported(int head_dim, int group, int num_kv_heads) {
  return (head_dim == 64 || head_dim == 128) &&
         (group == 1 || group == 2 || group == 4 || group == 8) && num_kv_heads >= 1;
}

size_t prefill_workspace_bytes(int, int, int, int, int) { return 0; }

cudaError_t launch_prefill(const AttnArgs& a, void*, size_t, int sm_count, cudaStream_t stream) {
  const int group = a.num_q_heads / a.num_kv_heads;
#define PA_PREFILL_CASE(D_, G_) \
  if (a.head_dim == D_ && group == G_) return launch_prefill_t<D_, G_>(a, sm_count, stream);
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
