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
//  * Warp 0 streams Q and K tiles, warp 10 V tiles, of 128 keys (8 pages of 16
//    tokens, one TMA box per page and 64-element half of head_dim, 128-byte
//    swizzle) into rings of shared-memory stages; separate K and V producers
//    let the next K tiles load while the V of earlier tiles is still in use.
//  * Warp 1 (one thread) issues tcgen05.mma: S = Q K^T into one of three
//    TMEM buffers, then O += P V into a TMEM accumulator.  S of the next tile
//    is queued before the P V of the current one, so the tensor pipe works on
//    one tile while the softmax warps work on the other.
//  * Warps 2-9 run the softmax, two warps per MMA row: the warp pair that
//    shares a TMEM lane quarter splits the 128 keys of a tile in halves and
//    swaps partial row maxima through shared memory.  They apply the causal
//    mask and scale, keep the running max / sum (base 2), write P (bf16) back
//    over their half of the S buffer in TMEM, where the P V MMA reads it as its
//    A operand, and rescale O in TMEM only when the max grows by more than 2^8
//    (exact: the same reference max scales the numerator and the denominator).
//    At the end they normalise O and store bf16 rows.
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
constexpr int kStagesK = 2;       // K tile stages
constexpr int kStagesV = 3;       // V tile stages (held from the S to the P V product)
constexpr int kSBufs = 3;         // S / P buffers in TMEM
constexpr int kSoftmaxWarps = 8;  // two per TMEM lane quarter
constexpr float kNegInf = -INFINITY;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kWarpV = 2 + kSoftmaxWarps;    // V producer
constexpr int kThreads = 32 * (kWarpV + 1);  // Q/K producer, MMA, softmax, V producer

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
  uint64_t s_full[kSBufs], p_full[kSBufs], pv_done[kSBufs];
  uint64_t o_full, o_empty;
  uint64_t mma_done;
  uint32_t tmem_slot;
  int abort_flag;
  long long total_items;
  float xmax[2][2][kRows];  // partial row maxima: [tile parity][key half][row]
  float xsum[2][kRows];     // partial row sums at the end of an item: [key half][row]
};

// Byte offset of 16-byte chunk c (0..7) of row r inside a [rows][64 x bf16]
// block stored with the 128-byte swizzle (8-row, 1024-byte atoms).
__device__ __forceinline__ uint32_t sw128_chunk(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// Position in a ring of pipeline stages: the stage and the parity of its
// current use, which flips each time the ring wraps around.
struct Ring {
  uint32_t stage = 0, phase = 0;
  __device__ __forceinline__ void next(uint32_t n) {
    if (++stage == n) {
      stage = 0;
      phase ^= 1u;
    }
  }
};

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
  constexpr uint32_t S_COL0 = 0, O_COL = kSBufs * kKeysPerTile;
  static_assert(O_COL + D <= TMEM_COLS, "TMEM columns");
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
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(smem_addr(&B.s_full[i]), 1);
      mbar_init(smem_addr(&B.p_full[i]), kSoftmaxWarps);
      mbar_init(smem_addr(&B.pv_done[i]), 1);
    }
    mbar_init(smem_addr(&B.o_full), 1);
    mbar_init(smem_addr(&B.o_empty), kSoftmaxWarps);
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

  if (warp == 0 || warp == kWarpV) {
    // ============================================================ producers
    if (lane == 0) {
      const bool is_k = (warp == 0);  // warp 0: Q and K, the last warp: V
      const CUtensorMap* map = is_k ? &kmap : &vmap;
      unsigned char* ring = is_k ? k_s : v_s;
      uint64_t* full = is_k ? B.k_full : B.v_full;
      uint64_t* empty = is_k ? B.k_empty : B.v_empty;
      const uint32_t nst = is_k ? kStagesK : kStagesV;
      ItemCursor<TM> cur;
      cur.init(p);
      int n_item = 0, c = 0;
      Ring pos;
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
          const uint32_t st = pos.stage;
          if (c >= (int)nst) mbar_wait(smem_addr(&empty[st]), pos.phase ^ 1u, p.err, abort_flag);
          mbar_arrive_expect_tx(smem_addr(&full[st]),
                                (uint32_t)nvalid * NH * (kBlock * 128));
          for (int i = 0; i < npg; ++i) {
            if (phys[i] < 0) continue;
#pragma unroll
            for (int h = 0; h < NH; ++h)
              tc::tma_load_3d(smem_addr(ring + st * KV_BYTES + h * HALF + i * (kBlock * 128)),
                              map, h * 64, it.g, phys[i] * kBlock, smem_addr(&full[st]));
          }
          pos.next(nst);
        }
      }
      // never hand back shared memory with a TMA copy still landing in it
      for (int i = max(0, c - (int)nst); i < c; ++i)
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
      uint32_t ntiles = 0;  // K/V tiles so far (all items)
      Ring kr, vr, sbr, prev;  // K stages, V stages, S buffers, S buffer of the last tile
      const uint32_t q_addr = smem_addr(q_s);
      bool issued = false;
      for (long long item = blockIdx.x; item < total_items; item += gridDim.x, ++n_item) {
        Item it;
        if (!cur.locate(p, item, it)) break;
        mbar_wait(smem_addr(&B.q_full), n_item & 1, p.err, abort_flag);
        auto issue_pv = [&](const Ring& pb, bool first) {
          mbar_wait(smem_addr(&B.p_full[pb.stage]), pb.phase, p.err, abort_flag);
          mbar_wait(smem_addr(&B.v_full[vr.stage]), vr.phase, p.err, abort_flag);
          if (first && n_item > 0)
            mbar_wait(smem_addr(&B.o_empty), (n_item - 1) & 1, p.err, abort_flag);
          tc::fence_after_sync();
          // P (bf16 pairs) of keys 64h .. 64h + 63 sits in columns 64h .. 64h + 31
          // of the S buffer it came from
          const uint32_t pt = tmem + S_COL0 + pb.stage * kKeysPerTile;
          const uint32_t va = smem_addr(v_s + vr.stage * KV_BYTES);
#pragma unroll
          for (int kk = 0; kk < kKeysPerTile / 16; ++kk) {
            const uint64_t bd = tc::sw128_desc(va + kk * 2048, HALF, 1024);
            tc::mma_bf16_tmem_a(tmem + O_COL, pt + (kk >> 2) * 64 + (kk & 3) * 8, bd, IDESC_O,
                                (first && kk == 0) ? 0u : 1u);
          }
          tc::commit(smem_addr(&B.v_empty[vr.stage]));
          tc::commit(smem_addr(&B.pv_done[pb.stage]));
          vr.next(kStagesV);
        };
        for (int kt = 0; kt < it.nkt; ++kt, ++ntiles) {
          mbar_wait(smem_addr(&B.k_full[kr.stage]), kr.phase, p.err, abort_flag);
          // the S buffer holds P of the tile kSBufs back until its PV has run
          if (ntiles >= kSBufs)
            mbar_wait(smem_addr(&B.pv_done[sbr.stage]), sbr.phase ^ 1u, p.err, abort_flag);
          tc::fence_after_sync();
          const uint32_t ka = smem_addr(k_s + kr.stage * KV_BYTES);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t ad =
                tc::sw128_desc(q_addr + (kk >> 2) * HALF + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = tc::sw128_desc(ka + (kk >> 2) * HALF + (kk & 3) * 32, 16, 1024);
            tc::mma_bf16(tmem + S_COL0 + sbr.stage * kKeysPerTile, ad, bd, IDESC_S,
                         kk > 0 ? 1u : 0u);
          }
          tc::commit(smem_addr(&B.s_full[sbr.stage]));
          tc::commit(smem_addr(&B.k_empty[kr.stage]));
          kr.next(kStagesK);
          if (kt == it.nkt - 1) tc::commit(smem_addr(&B.q_empty));
          if (kt > 0) issue_pv(prev, kt == 1);
          prev = sbr;
          sbr.next(kSBufs);
          issued = true;
        }
        issue_pv(prev, it.nkt == 1);
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
    const int kh = (warp - 2) >> 2;  // key half of each tile: 64*kh .. 64*kh + 63
    const int r = quarter * 32 + lane;
    const int pair_bar = 1 + quarter;  // named barrier of the two warps on these rows
    const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
    const int tl = r / G, hl = r % G;
    const float sl2 = p.scale_log2;
    // With a positive scale the max of the raw scores gives the max of the
    // scaled ones and the scale folds into the exponent's FMA; otherwise the
    // scores are scaled first.
    const bool pos_scale = sl2 > 0.f;
    const float mul = pos_scale ? 1.f : sl2;
    const float emul = pos_scale ? sl2 : 1.f;
    ItemCursor<TM> cur;
    cur.init(p);
    int n_item = 0;
    Ring sbr, prev, vr;  // S buffer of this tile and of the last one, V stage
    uint32_t xpar = 0;   // exchange slot parity
    for (long long item = blockIdx.x; item < total_items; item += gridDim.x, ++n_item) {
      Item it;
      if (!cur.locate(p, item, it)) break;
      const bool row_valid = tl < it.ntok;
      const int p_row = row_valid ? it.p_first + tl : it.kv_end - 1;
      float m_ref = kNegInf, l = 0.f;
      for (int kt = 0; kt < it.nkt; ++kt) {
        const uint32_t s_cols = tmem + lane_addr + S_COL0 + sbr.stage * kKeysPerTile + kh * 64;
        mbar_wait(smem_addr(&B.s_full[sbr.stage]), sbr.phase, p.err, abort_flag);
        tc::fence_after_sync();
        uint32_t sr[64];
        tc::tmem_ld32(s_cols, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tc::tmem_ld32(s_cols + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tc::tmem_wait_ld();

        // causal mask and the max of this half (three-input max, 4 chains)
        const int k0 = kt * kKeysPerTile + kh * 64;
        const int lim = p_row - k0;  // keys c <= lim of this half are visible
        float m4[4] = {kNegInf, kNegInf, kNegInf, kNegInf};
        if (__all_sync(0xffffffffu, lim >= 63)) {
          if (!pos_scale) {
#pragma unroll
            for (int c = 0; c < 64; ++c) sr[c] = __float_as_uint(__uint_as_float(sr[c]) * mul);
          }
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c)
            sr[c] = __float_as_uint((c <= lim) ? __uint_as_float(sr[c]) * mul : kNegInf);
        }
#pragma unroll
        for (int c = 0; c < 64; c += 8) {
          m4[(c >> 3) & 3] = fmax3(m4[(c >> 3) & 3], __uint_as_float(sr[c]),
                                   __uint_as_float(sr[c + 1]));
          m4[(c >> 3) & 3] = fmax3(m4[(c >> 3) & 3], __uint_as_float(sr[c + 2]),
                                   __uint_as_float(sr[c + 3]));
          m4[(c >> 3) & 3] = fmax3(m4[(c >> 3) & 3], __uint_as_float(sr[c + 4]),
                                   __uint_as_float(sr[c + 5]));
          m4[(c >> 3) & 3] = fmax3(m4[(c >> 3) & 3], __uint_as_float(sr[c + 6]),
                                   __uint_as_float(sr[c + 7]));
        }
        const float mh = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        // swap the half maxima with the other warp on these rows (slots alternate
        // with the tile parity, so a slot is rewritten only after a later barrier)
        B.xmax[xpar][kh][r] = mh;
        named_barrier(pair_bar, 64);
        float mx = fmaxf(mh, B.xmax[xpar][kh ^ 1][r]);
        mx = (mx == kNegInf) ? kNegInf : mx * emul;  // now in scaled base-2 units
        // both warps of the pair see the same maxima and take the same branch
        float alpha = 1.f;
        if (m_ref == kNegInf) {
          m_ref = mx;  // first tile: O not yet written
        } else if (mx > m_ref + kRescaleThreshold) {
          alpha = fast_exp2(m_ref - mx);
          l *= alpha;
          m_ref = mx;
        }
        // p = 2^(emul * s - m_ref), packed in bf16 pairs in place (sr[j] holds
        // keys 2j, 2j+1 of this half), stored over the first 32 columns of the half
        const float2 e2 = make_float2(emul, emul);
        const float2 nm2 = make_float2(-m_ref, -m_ref);
        float2 l4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) l4[j] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float2 x = __ffma2_rn(
              make_float2(__uint_as_float(sr[2 * j]), __uint_as_float(sr[2 * j + 1])), e2, nm2);
          const float2 pj = make_float2(fast_exp2(x.x), fast_exp2(x.y));
          l4[j & 3] = __fadd2_rn(l4[j & 3], pj);
          sr[j] = pack_bf16x2(pj.x, pj.y);
        }
        tc::tmem_st32(s_cols, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        l += ((l4[0].x + l4[0].y) + (l4[1].x + l4[1].y)) + ((l4[2].x + l4[2].y) + (l4[3].x + l4[3].y));
        // rescale this half of the running output when the reference max moved (rare)
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          mbar_wait(smem_addr(&B.pv_done[prev.stage]), prev.phase, p.err, abort_flag);
          tc::fence_after_sync();
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            const uint32_t oc = tmem + lane_addr + O_COL + kh * (D / 2) + c * 32;
            uint32_t o[32];
            tc::tmem_ld32(oc, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tc::tmem_st32(oc, o);
          }
        }
        // keys past the last needed one: V rows there may hold stale or
        // poisoned data; zero them so that P = 0 times V stays 0 (each warp of
        // the pair clears half of the row's 16-byte chunks)
        const int kv_local = it.kv_end - kt * kKeysPerTile;
        if (kv_local < kKeysPerTile) {
          mbar_wait(smem_addr(&B.v_full[vr.stage]), vr.phase, p.err, abort_flag);
          if (r >= kv_local) {
            unsigned char* vrow = v_s + vr.stage * KV_BYTES;
#pragma unroll
            for (int h = 0; h < NH; ++h)
#pragma unroll
              for (int c8 = 4 * kh; c8 < 4 * kh + 4; ++c8)
                *reinterpret_cast<uint4*>(vrow + h * HALF + sw128_chunk(r, c8)) =
                    make_uint4(0, 0, 0, 0);
          }
        }
        tc::tmem_wait_st();
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&B.p_full[sbr.stage]));
        prev = sbr;
        sbr.next(kSBufs);
        vr.next(kStagesV);
        xpar ^= 1u;
      }
      // epilogue: O / l -> bf16 rows; each warp of the pair writes half of d
      B.xsum[kh][r] = l;
      named_barrier(pair_bar, 64);
      const float inv = 1.f / (l + B.xsum[kh ^ 1][r]);
      mbar_wait(smem_addr(&B.o_full), n_item & 1, p.err, abort_flag);
      tc::fence_after_sync();
      uint16_t* orow = p.out + ((int64_t)(it.q0 + tl) * p.n_q + it.g * G + hl) * D + kh * (D / 2);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t o[32];
        tc::tmem_ld32(tmem + lane_addr + O_COL + kh * (D / 2) + c * 32, o);
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
