// pa_prefill_kernel.cuh -- chunked-prefill attention over the paged KV cache
// on the tcgen05 tensor cores (requests with q_len >= 2): the kernel, its
// key-piece merge and their launcher, included by pa_prefill.cu (plain and
// fused-step instances) and pa_prefill_fp8.cu (the 8-bit cache's instance).
//
// What it computes ("PagedAttention 显存分页与连续批处理(Continuous Batching)
// 实战", Chunked Prefill section: a long prompt is cut into fixed slices, each
// computed together with the running decodes; prefill is compute-bound and
// suits tensor-core GEMM; "连续批处理：推理吞吐的范式革命", section 4.1 for the
// attention itself): query row i of a request with q_len rows sits at position
// p = seq_len - q_len + i and attends to keys 0..p of its Block Table.
//
// Layout of the work (GB300 design, not the pages' scalar kernel):
//  * A query tile is 128/G tokens x the G q heads that share kv head g: the
//    128 rows of one MMA, so every K/V tile is loaded once for the whole GQA
//    group.  A unit is (request, query tile, kv head, key split).
//  * K/V tiles hold 128 keys (8 pages).  K lands as 16 TMA boxes (one per page
//    and 64-column half, 128-byte swizzle: the layout the S = Q K^T MMA reads
//    as 128 rows); V as 8 boxes of one page and both halves each (the P V MMA
//    consumes one page per instruction).  A single thread issues TMA boxes
//    slowly, so six producer warps share them, 96 rows of 128 bytes each
//    per tile.
//  * One thread of warp 1 issues S = Q K^T into one of three TMEM buffers and
//    one thread of warp 15 issues O += P V into a TMEM accumulator.  The
//    tensor pipe queues only a few MMAs, so a single issuing thread that
//    waits and commits between products leaves it idle; with two, one
//    thread's waits overlap the other's MMAs, and S runs ahead of P V.  Descriptors are built once and advanced
//    by constants: a 64-cycle MMA leaves the issuing thread little time.
//  * Warps 2-9 run the softmax, two warps per MMA row: the warp pair that
//    shares a TMEM lane quarter splits the 128 keys of a tile in halves and
//    swaps partial row maxima through shared memory.  They apply the causal
//    mask and scale, keep the running max / sum (base 2), write P (bf16) back
//    over their half of the S buffer, where the P V MMA reads it as its A
//    operand, and rescale O in TMEM only when the max grows by more than 2^8
//    (exact: the same reference max scales numerator and denominator).
//  * When the query tiles alone would leave SMs idle, the keys of each tile
//    are split over several units; each writes (O / l, m, l) per row and a
//    merge kernel combines the pieces with log-sum-exp weights.
//  * Persistent CTAs (at most one per SM) walk the unit list.
//  * Fused step (pa_paged_attention_step): the step's new key and value rows
//    are not in the cache yet.  The producers take pages of new positions
//    straight from k_new / v_new (their own tensor maps: a request's new
//    tokens are consecutive rows there), and the one page that holds both
//    cached and new positions is loaded from the cache and has its new rows
//    copied over in shared memory before it is handed to the products.  The
//    unit of each query tile's last key piece stores that tile's new rows
//    (its kv head) to their slots; no other unit reads them from the cache,
//    so the stores need no ordering within the kernel.
//  * 8-bit cache (pa_paged_attention_fp8): the producers read a page's E4M3
//    codes and row scales with plain loads and write f16(code * f16(scale))
//    into the stage, in the layout the TMA gives the bf16 instance (both types
//    are 16 bits wide).  The query tile is rewritten in place as
//    f16(q * scale * log2 e) once it lands, so the products run with f16
//    operands (one tcgen05 kind::f16 product takes A and B of one type) and
//    P is packed as f16; the softmax then works in base-2 units directly.
#pragma once

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr int kBlock = 16;         // tokens per physical block
constexpr int kKeysPerTile = 128;  // keys per K/V tile (8 blocks)
constexpr int kPagesPerTile = kKeysPerTile / kBlock;
constexpr int kRows = 128;         // MMA rows of a query tile
constexpr int kStagesK = 3;        // K tile stages (bf16 cache)
constexpr int kStagesV = 2;        // V tile stages (bf16 cache)
constexpr int kStagesMax = 3;      // the most stages of one kind in any instance
constexpr int kSBufs = 3;          // S / P buffers in TMEM
constexpr int kSoftmaxWarps = 8;   // two per TMEM lane quarter
constexpr int kKWarps = 3;         // warp 0 (which also loads Q) and warps 10-11
constexpr int kVWarps = 3;         // warps 12-14
constexpr int kWarpK1 = 10, kWarpV0 = 12;
constexpr int kWarpPV = 15;        // issues the P V products
constexpr int kThreads = 512;
constexpr float kNegInf = -INFINITY;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr int kMaxSplit = 4;
constexpr int kMaxListed = 1024;   // prefill requests the shared-memory unit list holds

// Instances of the kernel: the plain one reads the bf16 cache; the fused
// step's also takes the step's new rows from k_new / v_new and stores them;
// the 8-bit one reads E4M3 codes and row scales.
enum : int { kKindPlain = 0, kKindFused = 1, kKindFp8 = 2 };

struct PrefillParams {
  // fused step (the kernel's FUSE instance): new rows [num_tokens, n_kv, D]
  // and their slots, and the caches they are stored to
  const uint16_t* k_new;
  const uint16_t* v_new;
  const int32_t* slot_mapping;
  uint16_t* k_cache;
  uint16_t* v_cache;
  // 8-bit cache: 16-token pages of codes [16, n_kv, D], then their scales
  // [16, n_kv] (fp32); the query tile is scaled by q_mul (scale * log2 e)
  // into f16
  const uint8_t* k_codes;
  const uint8_t* v_codes;
  float q_mul;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* qsl;
  uint16_t* out;
  float* part_o;   // [num_tokens * n_q * nsplit, D] (nsplit > 1)
  float* part_ml;  // [num_tokens * n_q * nsplit, 2]
  unsigned* err;
  int32_t num_blocks, max_blocks, num_seqs, num_tokens, n_q, n_kv, max_seq_len, nsplit;
  int32_t block_shift;  // log2(block_size / 16)
  int32_t no_decode;    // a request with one query row is an error (no decode kernel runs)
  float scale_log2;
};

// Whether request s runs here (q_len >= 2) and its lengths are valid.
__device__ __forceinline__ bool prefill_request(const PrefillParams& p, int s, int& a, int& ql,
                                                int& L, bool report) {
  a = __ldg(p.qsl + s);
  const int b = __ldg(p.qsl + s + 1);
  ql = b - a;
  if (ql < 2) {
    if (ql == 1 && p.no_decode && report) flag_error(p.err, DEVERR_BOUNDS);
    return false;
  }
  L = __ldg(p.seq_lens + s);
  if (L < ql || L > p.max_seq_len || L > (p.max_blocks << p.block_shift) * kBlock || a < 0 ||
      b > p.num_tokens) {
    if (report) flag_error(p.err, DEVERR_BOUNDS);
    return false;
  }
  return true;
}

// Query tiles of request s.
template <int TM>
__device__ __forceinline__ int prefill_tiles(const PrefillParams& p, int s, bool report) {
  int a, ql, L;
  if (!prefill_request(p, s, a, ql, L, report)) return 0;
  return (ql + TM - 1) / TM;
}

// Geometry of one unit.
struct Unit {
  int s, g, ks;
  int a;        // first query token of the request
  int c0;       // first new position of the request (seq_len - q_len)
  int q0;       // first query token of the tile
  int ntok;     // valid query tokens of the tile
  int p_first;  // position of token q0
  int kv_end;   // keys the tile needs: 0 .. kv_end - 1
  int kt0, kt1; // K/V tiles of this unit (of ceil(kv_end / 128))
};

// Walks the unit list: request-major, then query tile, kv head, key split.
// Requests are found through the block's list of prefill requests (sequence
// ids and first tile indices, built once per CTA); when a batch holds more
// than kMaxListed of them the cursor walks the sequences instead.
template <int TM>
struct UnitCursor {
  const int* seq;   // listed requests, or nullptr
  const int* tbase; // first tile of each listed request; tbase[n] = all tiles
  int n;
  int i = 0;        // list position, or sequence when walking
  int base = 0, tiles = 0;
  __device__ __forceinline__ void init(const PrefillParams& p, const int* list_seq,
                                       const int* list_base, int listed) {
    seq = listed <= kMaxListed ? list_seq : nullptr;
    tbase = list_base;
    n = listed;
    i = 0;
    base = 0;
    tiles = (!seq && p.num_seqs > 0) ? prefill_tiles<TM>(p, 0, false) : 0;
  }
  __device__ __forceinline__ bool locate(const PrefillParams& p, long long u, Unit& U) {
    const long long per = (long long)p.n_kv * p.nsplit;
    const long long tile = u / per;
    const int rem = (int)(u % per);
    int s;
    if (seq) {
      while (i < n && tile >= tbase[i + 1]) ++i;
      if (i >= n) return false;
      s = seq[i];
      base = tbase[i];
    } else {
      while (i < p.num_seqs && tile >= (long long)base + tiles) {
        base += tiles;
        ++i;
        tiles = i < p.num_seqs ? prefill_tiles<TM>(p, i, false) : 0;
      }
      if (i >= p.num_seqs) return false;
      s = i;
    }
    const int a = __ldg(p.qsl + s), b = __ldg(p.qsl + s + 1);
    const int L = __ldg(p.seq_lens + s);
    const int ql = b - a;
    const int first = (int)(tile - base) * TM;
    U.s = s;
    U.a = a;
    U.c0 = L - ql;
    U.g = rem / p.nsplit;
    U.ks = rem % p.nsplit;
    U.q0 = a + first;
    U.ntok = min(TM, ql - first);
    U.p_first = L - ql + first;
    U.kv_end = U.p_first + U.ntok;
    const int nkt = (U.kv_end + kKeysPerTile - 1) / kKeysPerTile;
    U.kt0 = U.ks * nkt / p.nsplit;
    U.kt1 = (U.ks + 1) * nkt / p.nsplit;
    return true;
  }
};

struct PrefillShared {
  uint64_t q_full, q_empty;
  uint64_t q_land;  // 8-bit cache: the bf16 query tile has landed (then rewritten)
  uint64_t k_full[kStagesMax], k_empty[kStagesMax];
  uint64_t v_full[kStagesMax], v_empty[kStagesMax];
  uint64_t s_full[kSBufs], p_full[kSBufs], pv_done[kSBufs];
  uint64_t o_full, o_empty;
  uint64_t s_done, pv_done_all;  // each issuer's last products, before TMEM is freed
  uint64_t patch[kThreads / 32];  // per producer warp: a page to patch has landed
  uint32_t tmem_slot;
  int abort_flag;
  long long total_units;
  float xmax[2][2][kRows];  // partial row maxima: [tile parity][key half][row]
  float xsum[2][2][kRows];  // partial row sums: [unit parity][key half][row]
  int list_seq[kMaxListed];       // prefill requests in order
  int list_base[kMaxListed + 1];  // their first tile indices, then the tile count
  int listed;
  int warp_n[kThreads / 32], warp_tiles[kThreads / 32];
};

// acc += the two bf16 values of w (low half into x, high half into y),
// exactly as fp32 additions of the widened values.
__device__ __forceinline__ void add_bf16x2_to(float2& acc, uint32_t w) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
      : "+f"(acc.x), "+f"(acc.y)
      : "r"(w));
}

// acc += the two f16 values of w (low half into acc.x), in fp32.
__device__ __forceinline__ void add_f16x2_to(float2& acc, uint32_t w) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.f16 %0, lo, %0;\n\tadd.rn.f32.f16 %1, hi, %1;\n\t}"
      : "+f"(acc.x), "+f"(acc.y)
      : "r"(w));
}

// A bf16 pair times m, as an f16 pair (one rounding, of the fp32 product).
__device__ __forceinline__ uint32_t f16x2_from_bf16x2_mul(uint32_t w, float m) {
  const float2 f = bf16x2_to_float2(w);
  return f16x2_from_floats(f.x * m, f.y * m);
}

// Four E4M3 codes times a row scale given as an f16 pair (both halves the
// scale), as two f16 pairs: each value is f16(code * f16(scale)) (the codes
// convert exactly; one packed multiply per pair, round to nearest).
__device__ __forceinline__ void f16x4_from_e4m3x4_scaled(uint32_t w, uint32_t sc2, uint32_t& lo,
                                                         uint32_t& hi) {
  uint32_t a, b;
  f16x2x2_from_e4m3x4(w, a, b);
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(a), "r"(sc2));
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(b), "r"(sc2));
}

// Byte offset of 16-byte chunk c (0..7) of row r inside a [rows][64 x bf16]
// block stored with the 128-byte swizzle (8-row, 1024-byte atoms).
__device__ __forceinline__ uint32_t sw128_chunk(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

// Position in a ring of pipeline stages: the stage and the parity of its
// current use, which flips each time the ring wraps around.
//
// Every wait below is a phase-parity wait, which tells apart only the phase
// it names and the one before it.  So each wait carries, beside it, why its
// barrier is never still at the use before the one wanted (the wait would
// pass at once) nor already past the wanted use (it would wait for a
// completion that needs this thread).  The argument is the same shape each
// time: the waiter saw the previous use complete, or a product it already
// waited for needed it; and the next use needs something this thread does
// after the wait.  Stage and buffer counts are compile-time constants.
struct Ring {
  uint32_t stage = 0, phase = 0;
  __device__ __forceinline__ void next(uint32_t n) {
    if (++stage == n) {
      stage = 0;
      phase ^= 1u;
    }
  }
};

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            int z, int w, uint32_t mbar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(mbar)
      : "memory");
}

// S = Q K^T for the query tile and a K tile (128 x 128 x D), issued by one
// thread.  a, b: descriptors of the Q tile and the K tile; each K = 16 step
// advances both start addresses by a compile-time offset.  F16: f16 operands
// (the 8-bit cache's instance), else bf16.
template <int D, bool F16>
__device__ __forceinline__ void issue_s_mma(uint32_t d_tmem, tc::Desc a, tc::Desc b) {
  constexpr uint32_t HALF = kRows * 128;
  constexpr uint32_t IDESC_S = F16 ? tc::idesc_f16_f32(kRows, kKeysPerTile, 0, 0)
                                   : tc::idesc_bf16_f32(kRows, kKeysPerTile, 0, 0);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = ((kk >> 2) * HALF + (kk & 3) * 32) >> 4;
    if (kk == 0)
      tc::mma_bf16_pair<false>(d_tmem, a, off, b, off, IDESC_S);
    else
      tc::mma_bf16_pair<true>(d_tmem, a, off, b, off, IDESC_S);
  }
}

// O += P V: P (bf16 pairs) of keys 64h .. 64h + 63 sits in columns
// 64h .. 64h + 31 of the S buffer at p_tmem; V page kk of the tile
// (descriptor b) is one K = 16 step.
template <int D, bool F16>
__device__ __forceinline__ void issue_pv_mma(uint32_t o_tmem, uint32_t p_tmem, tc::Desc b,
                                             bool first) {
  constexpr uint32_t V_PAGE = (D / 64) * kBlock * 128;
  constexpr uint32_t IDESC_O =
      F16 ? tc::idesc_f16_f32(kRows, D, 0, 1) : tc::idesc_bf16_f32(kRows, D, 0, 1);
  if (first)
    tc::mma_bf16_tmem_a_pair<false>(o_tmem, p_tmem, b, 0, IDESC_O);
  else
    tc::mma_bf16_tmem_a_pair<true>(o_tmem, p_tmem, b, 0, IDESC_O);
#pragma unroll
  for (int kk = 1; kk < kPagesPerTile; ++kk)
    tc::mma_bf16_tmem_a_pair<true>(o_tmem, p_tmem + (kk >> 2) * 64 + (kk & 3) * 8, b,
                                   (kk * V_PAGE) >> 4, IDESC_O);
}

// Whether token t's slot is the slot of position pos of request U (the fused
// step's precondition), as a 64-bit slot or -1.
__device__ __forceinline__ int64_t fused_slot(const PrefillParams& p, const int32_t* table,
                                              int t, int pos) {
  const int64_t slot = __ldg(p.slot_mapping + t);
  const int lp = pos / kBlock;
  const int b = __ldg(table + (lp >> p.block_shift));
  const int64_t want =
      ((int64_t)((b << p.block_shift) + (lp & ((1 << p.block_shift) - 1)))) * kBlock +
      pos % kBlock;
  if (b < 0 || b >= p.num_blocks || slot != want) return -1;
  return slot;
}

// Fused step: store the new rows of kv head U.g of the unit's query tile
// (tokens q0 .. q0 + ntok - 1) from newrows to their slots in cache; warp
// idx of the nw warps doing it.  Eight 16-byte chunks per lane at a time,
// all their loads (row, slot, block-table entry) issued before any store,
// so one round trip covers a batch.  A token whose slot is not its
// position's slot is not stored and is flagged.
template <int D>
__device__ __forceinline__ void fused_store_rows(const PrefillParams& p, const Unit& U,
                                                 const int32_t* table, const uint16_t* newrows,
                                                 uint16_t* cache, int idx, int nw, int lane) {
  constexpr int PER_TOK = D / 8;  // 16-byte chunks of a row
  constexpr int NB = 8;
  const int n = U.ntok * PER_TOK;
  const int step = nw * 32;
  for (int e0 = idx * 32 + lane; e0 < n; e0 += NB * step) {
    uint4 v[NB];
    int64_t slot[NB];
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const int e = e0 + j * step;
      slot[j] = -1;
      v[j] = make_uint4(0u, 0u, 0u, 0u);
      if (e < n) {
        const int i = e / PER_TOK, c8 = e % PER_TOK;
        const int t = U.q0 + i;
        slot[j] = fused_slot(p, table, t, U.p_first + i);
        v[j] = __ldg(reinterpret_cast<const uint4*>(newrows + ((int64_t)t * p.n_kv + U.g) * D +
                                                    c8 * 8));
      }
    }
#pragma unroll
    for (int j = 0; j < NB; ++j) {
      const int e = e0 + j * step;
      if (e >= n) continue;
      const int c8 = e % PER_TOK;
      if (slot[j] < 0) {
        if (c8 == 0) flag_error(p.err, DEVERR_BOUNDS);
        continue;
      }
      *reinterpret_cast<uint4*>(cache + (slot[j] * p.n_kv + U.g) * D + c8 * 8) = v[j];
    }
  }
}

template <int D, int G, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap qmap,
                   const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap,
                   const __grid_constant__ CUtensorMap knmap,
                   const __grid_constant__ CUtensorMap vnmap) {
  constexpr bool FUSE = KIND == kKindFused;
  constexpr bool F8 = KIND == kKindFp8;
  // Stages: the 8-bit instance's V copies wait for a product two tiles
  // earlier with two V stages, and its producers take longer per page (code
  // conversion), so it trades a K stage for a V stage (same shared memory).
  constexpr int SK = F8 ? 2 : kStagesK;
  constexpr int SV = F8 ? 3 : kStagesV;
  static_assert(SK + SV == kStagesK + kStagesV && SK <= kStagesMax && SV <= kStagesMax,
                "shared memory holds kStagesK + kStagesV tiles");
  constexpr int TM = kRows / G;            // query tokens per tile
  constexpr int NH = D / 64;               // 64-element halves of head_dim
  constexpr uint32_t HALF = kRows * 128;   // bytes of one [128 rows][64] block
  constexpr uint32_t Q_BYTES = NH * HALF;  // the query tile
  constexpr uint32_t KV_BYTES = NH * HALF; // one K or V tile (128 keys)
  constexpr uint32_t V_PAGE = NH * kBlock * 128;  // V tile: [page][half][16][64]
  constexpr uint32_t TMEM_COLS = 512;
  constexpr uint32_t O_COL = kSBufs * kKeysPerTile;  // S buffers, then O
  static_assert(O_COL + D <= TMEM_COLS, "TMEM columns");

  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  unsigned char* q_s = base;
  unsigned char* k_s = q_s + Q_BYTES;
  unsigned char* v_s = k_s + SK * KV_BYTES;
  PrefillShared& B = *reinterpret_cast<PrefillShared*>(v_s + SV * KV_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the merge grid of split keys may start launching now
  asm volatile("griddepcontrol.launch_dependents;");
  // fetch the tensor maps this instance uses ahead of their first copy
  if (threadIdx.x == 32) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&qmap)) : "memory");
    if constexpr (!F8) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&kmap)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&vmap)) : "memory");
    }
    if constexpr (FUSE) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&knmap)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&vnmap)) : "memory");
    }
  }

  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&B.q_full), 1);
    mbar_init(smem_addr(&B.q_land), 1);
    mbar_init(smem_addr(&B.q_empty), 1);
    for (int i = 0; i < SK; ++i) {
      mbar_init(smem_addr(&B.k_full[i]), kKWarps);
      mbar_init(smem_addr(&B.k_empty[i]), 1);
    }
    for (int i = 0; i < SV; ++i) {
      mbar_init(smem_addr(&B.v_full[i]), kVWarps);
      mbar_init(smem_addr(&B.v_empty[i]), 1);
    }
    for (int i = 0; i < kSBufs; ++i) {
      mbar_init(smem_addr(&B.s_full[i]), 1);
      mbar_init(smem_addr(&B.p_full[i]), kSoftmaxWarps);
      mbar_init(smem_addr(&B.pv_done[i]), 1);
    }
    mbar_init(smem_addr(&B.o_full), 1);
    mbar_init(smem_addr(&B.o_empty), kSoftmaxWarps);
    mbar_init(smem_addr(&B.s_done), 1);
    mbar_init(smem_addr(&B.pv_done_all), 1);
    for (int w = 0; w < kThreads / 32; ++w) mbar_init(smem_addr(&B.patch[w]), 1);
    B.abort_flag = 0;
    fence_mbar_init();
  }
  {
    // list the requests with prefill rows (and their first tile index): one
    // pass over the sequences by the whole block, in order
    int listed = 0, tiles_so_far = 0;
    for (int s0 = 0; s0 < p.num_seqs; s0 += kThreads) {
      const int s = s0 + (int)threadIdx.x;
      const int t = s < p.num_seqs ? prefill_tiles<TM>(p, s, blockIdx.x == 0) : 0;
      const unsigned has = __ballot_sync(0xffffffffu, t > 0);
      int incl = t;  // inclusive scan of tiles over the warp
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (lane == 31) {
        B.warp_n[warp] = __popc(has);
        B.warp_tiles[warp] = incl;
      }
      __syncthreads();
      int n_before = 0, t_before = 0, n_all = 0, t_all = 0;
      for (int w = 0; w < kThreads / 32; ++w) {
        if (w < warp) {
          n_before += B.warp_n[w];
          t_before += B.warp_tiles[w];
        }
        n_all += B.warp_n[w];
        t_all += B.warp_tiles[w];
      }
      if (t > 0) {
        const int idx = listed + n_before + __popc(has & ((1u << lane) - 1u));
        if (idx < kMaxListed) {
          B.list_seq[idx] = s;
          B.list_base[idx] = tiles_so_far + t_before + incl - t;
        }
      }
      listed += n_all;
      tiles_so_far += t_all;
      __syncthreads();
    }
    if (threadIdx.x == 0) {
      B.listed = listed;
      if (listed <= kMaxListed) B.list_base[listed] = tiles_so_far;
      B.total_units = (long long)tiles_so_far * p.n_kv * p.nsplit;
    }
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_addr(&B.tmem_slot), TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = B.tmem_slot;
  const long long total_units = B.total_units;
  volatile int* abort_flag = &B.abort_flag;

  const bool k_warp = warp == 0 || (warp >= kWarpK1 && warp < kWarpK1 + kKWarps - 1);
  const bool v_warp = warp >= kWarpV0 && warp < kWarpV0 + kVWarps;
  if (k_warp || v_warp) {
    // ============================================================ producers
    // (lane 0 issues and waits; in the fused step the whole warp runs along
    // to patch pages and store the step's rows)
    if (FUSE || F8 || lane == 0) {
      // K warp k and V warp k load pages 3k .. 3k+2 of each tile (the last
      // two): 96 rows of 128 bytes per warp and tile either way
      const int idx = k_warp ? (warp == 0 ? 0 : warp - kWarpK1 + 1) : warp - kWarpV0;
      const int pg_lo = 3 * idx;
      const int pg_hi = min(pg_lo + 3, kPagesPerTile);
      const CUtensorMap* map = k_warp ? &kmap : &vmap;
      const CUtensorMap* nmap = k_warp ? &knmap : &vnmap;
      const uint16_t* newrows = k_warp ? p.k_new : p.v_new;
      unsigned char* ring = k_warp ? k_s : v_s;
      uint64_t* full = k_warp ? B.k_full : B.v_full;
      uint64_t* empty = k_warp ? B.k_empty : B.v_empty;
      const uint32_t nst = k_warp ? SK : SV;
      const uint32_t patch_bar = smem_addr(&B.patch[warp]);
      uint32_t n_patch = 0;
      UnitCursor<TM> cur;
      cur.init(p, B.list_seq, B.list_base, B.listed);
      int n_out = 0, c = 0;
      Ring pos;
      for (long long u = blockIdx.x; u < total_units; u += gridDim.x) {
        Unit U;
        if (!cur.locate(p, u, U)) break;
        if (U.kt0 == U.kt1) continue;
        if (warp == 0 && lane == 0) {
          // Q of the last unit released: this thread saw the release before
          // that (it loaded the last Q after it), and the next release needs
          // the S products of the Q loaded below
          if (n_out > 0) mbar_wait(smem_addr(&B.q_empty), (n_out - 1) & 1, p.err, abort_flag);
          const uint32_t qbar = smem_addr(F8 ? &B.q_land : &B.q_full);
          mbar_arrive_expect_tx(qbar, Q_BYTES);
#pragma unroll
          for (int h = 0; h < NH; ++h)
            tc::tma_load_3d(smem_addr(q_s + h * HALF), &qmap, h * 64, U.g * G, U.q0, qbar);
        }
        if constexpr (F8) {
          if (warp == 0) {
            // the bf16 query tile has landed (q_land: one use per unit, armed
            // above and waited for here before it is armed again); rewrite it
            // in place as f16(q * scale * log2 e) for the f16 products
            if (lane == 0) mbar_wait(smem_addr(&B.q_land), n_out & 1, p.err, abort_flag);
            __syncwarp();
            for (int e = lane; e < (int)(Q_BYTES / 16); e += 32) {
              uint4* qp = reinterpret_cast<uint4*>(q_s + e * 16);
              uint4 v = *qp;
              v.x = f16x2_from_bf16x2_mul(v.x, p.q_mul);
              v.y = f16x2_from_bf16x2_mul(v.y, p.q_mul);
              v.z = f16x2_from_bf16x2_mul(v.z, p.q_mul);
              v.w = f16x2_from_bf16x2_mul(v.w, p.q_mul);
              *qp = v;
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&B.q_full));
          }
        }
        ++n_out;
        const int pages = (U.kv_end + kBlock - 1) / kBlock;
        const int32_t* table = p.block_tables + (int64_t)U.s * p.max_blocks;
        for (int kt = U.kt0; kt < U.kt1; ++kt, ++c) {
          // per page: -1 (nothing to load), 0 (cached rows: the cache), 1
          // (new rows only: k_new / v_new), 2 (both: the cache, then the new
          // rows copied over)
          int phys[4], kind[4];
          uint32_t bytes = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int lp = kt * kPagesPerTile + pg_lo + i;  // logical page
            phys[i] = -1;
            kind[i] = -1;
            if (pg_lo + i < pg_hi && lp < pages) {
              const int pos0 = lp * kBlock;
              if (FUSE && pos0 >= U.c0) {
                kind[i] = 1;
                bytes += NH * (kBlock * 128);
                continue;
              }
              const int b = __ldg(table + (lp >> p.block_shift));
              if (b < 0 || b >= p.num_blocks) {
                if (lane == 0) flag_error(p.err, DEVERR_BOUNDS);
              } else {
                phys[i] = (b << p.block_shift) + (lp & ((1 << p.block_shift) - 1));
                kind[i] = (FUSE && pos0 + kBlock > U.c0) ? 2 : 0;
                if (kind[i] == 0) bytes += NH * (kBlock * 128);
              }
            }
          }
          const uint32_t st = pos.stage;
          if constexpr (F8) {
            // 8-bit cache: this warp's pages as codes and row scales, by
            // plain loads issued before the stage is free (their latency
            // overlaps the wait); lane j-th chunk: 16 codes of one row
            constexpr int CPR = D / 16;                  // chunks per row
            constexpr int NJ = 3 * kBlock * CPR / 32;    // chunks per lane
            const uint8_t* pages = k_warp ? p.k_codes : p.v_codes;
            const int64_t page_bytes = fp8_page_bytes(p.n_kv, D);
            const int64_t scales_at = fp8_scales_offset(p.n_kv, D);
            uint4 w8[NJ];
            float sc[NJ];
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
              const int pi = (32 * j) / D;  // page of the warp (D rows x chunks per page)
              const int rem = (32 * j) % D + lane;
              w8[j] = make_uint4(0u, 0u, 0u, 0u);
              sc[j] = 0.f;
              if (phys[pi] >= 0) {
                const uint8_t* page = pages + (int64_t)phys[pi] * page_bytes;
                const int row = (rem / CPR) * p.n_kv + U.g;  // (token row, head) in the page
                w8[j] = __ldg(reinterpret_cast<const uint4*>(page + (int64_t)row * D) + rem % CPR);
                sc[j] = __ldg(reinterpret_cast<const float*>(page + scales_at) + row);
              }
            }
            // the stage's last reader released it (as below)
            if (lane == 0 && c >= (int)nst)
              mbar_wait(smem_addr(&empty[st]), pos.phase ^ 1u, p.err, abort_flag);
            __syncwarp();
            unsigned char* stage = ring + st * KV_BYTES;
#pragma unroll
            for (int j = 0; j < NJ; ++j) {
              const int pi = (32 * j) / D;
              if (phys[pi] < 0) continue;  // no page there: nothing is read from it
              const int rem = (32 * j) % D + lane;
              const int r = rem / CPR, c16 = rem % CPR;
              const int pg = pg_lo + pi;
              uint32_t h[8];  // the chunk's 16 values, f16
              const uint32_t sc2 = f16x2_from_floats(sc[j], sc[j]);
              f16x4_from_e4m3x4_scaled(w8[j].x, sc2, h[0], h[1]);
              f16x4_from_e4m3x4_scaled(w8[j].y, sc2, h[2], h[3]);
              f16x4_from_e4m3x4_scaled(w8[j].z, sc2, h[4], h[5]);
              f16x4_from_e4m3x4_scaled(w8[j].w, sc2, h[6], h[7]);
              // elements 16 c16 .. +15: half c16 / 4, 16-byte chunks 2 (c16 % 4)
              // and the next of that half's 128-byte row
              const int hh = c16 >> 2, c8 = (c16 & 3) * 2;
              unsigned char* d0 =
                  k_warp ? stage + hh * HALF + sw128_chunk(pg * kBlock + r, c8)
                         : stage + pg * V_PAGE + hh * (kBlock * 128) + sw128_chunk(r, c8);
              unsigned char* d1 =
                  k_warp ? stage + hh * HALF + sw128_chunk(pg * kBlock + r, c8 + 1)
                         : stage + pg * V_PAGE + hh * (kBlock * 128) + sw128_chunk(r, c8 + 1);
              *reinterpret_cast<uint4*>(d0) = make_uint4(h[0], h[1], h[2], h[3]);
              *reinterpret_cast<uint4*>(d1) = make_uint4(h[4], h[5], h[6], h[7]);
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&full[st]));
            pos.next(nst);
            continue;
          }
          // the stage's last reader released it: one commit per use, and the
          // next commit needs this load, so never two completions behind
          if (lane == 0 && c >= (int)nst)
            mbar_wait(smem_addr(&empty[st]), pos.phase ^ 1u, p.err, abort_flag);
          if constexpr (FUSE) __syncwarp();
          bool patch = false;
#pragma unroll
          for (int i = 0; i < 4; ++i) patch |= FUSE && kind[i] == 2;
          if (lane == 0) {
            // with a page to patch, all of this warp's copies of the stage
            // land on its own barrier, and its arrival on the stage's
            // barrier waits until the new rows are in place
            if (patch)
              mbar_arrive_expect_tx(patch_bar, bytes + NH * (kBlock * 128));
            else
              mbar_arrive_expect_tx(smem_addr(&full[st]), bytes);
          }
          unsigned char* stage = ring + st * KV_BYTES;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (kind[i] < 0 || lane != 0) continue;
            const int pg = pg_lo + i;
            const uint32_t bar = patch ? patch_bar : smem_addr(&full[st]);
            // rows of the box: a cache page, or 16 new tokens of the request
            const CUtensorMap* m = kind[i] == 1 ? nmap : map;
            const int z = kind[i] == 1 ? U.a + (kt * kPagesPerTile + pg) * kBlock - U.c0
                                       : phys[i] * kBlock;
            if (k_warp) {
#pragma unroll
              for (int h = 0; h < NH; ++h)
                tc::tma_load_3d(smem_addr(stage + h * HALF + pg * (kBlock * 128)), m, h * 64, U.g,
                                z, bar);
            } else if (NH == 2) {
              tma_load_4d(smem_addr(stage + pg * V_PAGE), m, 0, U.g, z, 0, bar);
            } else {
              tc::tma_load_3d(smem_addr(stage + pg * V_PAGE), m, 0, U.g, z, bar);
            }
          }
          if (patch) {
            // the page with both kinds of rows: wait for its cache rows,
            // then copy its new rows over them (16-byte chunks, in the
            // stage's 128-byte-swizzled layout), visible to the products
            // one use of this warp's own barrier at a time: armed above,
            // completed here before it is armed again
            if (lane == 0) mbar_wait(patch_bar, n_patch & 1, p.err, abort_flag);
            ++n_patch;
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              if (kind[i] != 2) continue;
              const int pg = pg_lo + i;
              const int pos0 = (kt * kPagesPerTile + pg) * kBlock;
              const int r0 = U.c0 - pos0;  // first new row of the page
              // rows past the unit's keys are masked (and V rows cleared),
              // and past the request's tokens there is no new row to copy
              const int r1 = min(kBlock, U.kv_end - pos0);
              const int nchunks = max(0, r1 - r0) * NH * 8;
              for (int e = lane; e < nchunks; e += 32) {
                const int r = r0 + e / (NH * 8), h = (e / 8) % NH, c8 = e % 8;
                const int t = U.a + pos0 + r - U.c0;  // its token
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(
                    newrows + ((int64_t)t * p.n_kv + U.g) * D + h * 64 + c8 * 8));
                unsigned char* dst =
                    k_warp ? stage + h * HALF + sw128_chunk(pg * kBlock + r, c8)
                           : stage + pg * V_PAGE + h * (kBlock * 128) + sw128_chunk(r, c8);
                *reinterpret_cast<uint4*>(dst) = v;
              }
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_addr(&full[st]));
          }
          pos.next(nst);
        }
        // fused step: the unit of the query tile's last key piece (never
        // empty, unlike the first when a request has fewer key tiles than
        // pieces) stores the tile's new rows of its kv head (K by the K
        // warps, V by the V warps) to their slots.  No unit reads these rows
        // from the cache, so the stores need no place in the pipeline: after
        // the unit's last copies are issued, the products of the stages in
        // flight cover them
        if (FUSE && U.ks == p.nsplit - 1)
          fused_store_rows<D>(p, U, table, newrows, k_warp ? p.k_cache : p.v_cache, idx,
                              k_warp ? kKWarps : kVWarps, lane);
      }
      // never hand back shared memory with a TMA copy still landing in it:
      // the last use of each stage (the one before it was released by the
      // consumer that read it; no later use is ever issued)
      if (lane == 0) {
        for (int i = max(0, c - (int)nst); i < c; ++i)
          mbar_wait(smem_addr(&full[i % nst]), (i / nst) & 1, p.err, abort_flag);
        if (warp == 0 && n_out > 0)
          mbar_wait(smem_addr(&B.q_full), (n_out - 1) & 1, p.err, abort_flag);
      }
    }
  } else if (warp == 1 || warp == kWarpPV) {
    // ============================================================ MMA issuers
    // (waits spin without the suspend hint: these threads' latency is the
    // tensor pipe's)
    if (lane == 0) {
      UnitCursor<TM> cur;
      cur.init(p, B.list_seq, B.list_base, B.listed);
      int n_out = 0;
      uint32_t ntiles = 0;  // tiles of S (or P V) issued so far, all units
      Ring kv, sb;          // K (or V) stage; S buffer of the next S (or P V)
      if (warp == 1) {
        // S = Q K^T into the S buffer at sb, which held P three tiles back:
        // the P V of that tile must have run
        const tc::Desc qd = tc::sw128_desc_pair(smem_addr(q_s), 16, 1024);
        // stage i's descriptor: the start address (16-byte units, low word)
        // advanced by i tiles
        const tc::Desc kd0 = tc::sw128_desc_pair(smem_addr(k_s), 16, 1024);
        for (long long u = blockIdx.x; u < total_units; u += gridDim.x) {
          Unit U;
          if (!cur.locate(p, u, U)) break;
          if (U.kt0 == U.kt1) continue;
          // this unit's Q: the last unit's load was waited for here, and
          // the next load waits for q_empty, which this thread commits
          mbar_wait_spin(smem_addr(&B.q_full), n_out & 1, p.err, abort_flag);
          for (int kt = U.kt0; kt < U.kt1; ++kt, ++ntiles) {
            // K tile kt: this thread waited for the stage's last use, and
            // the stage's next copy waits for k_empty, committed below
            mbar_wait_spin(smem_addr(&B.k_full[kv.stage]), kv.phase, p.err, abort_flag);
            // P V of the tile that last used this S buffer: the one before
            // on the buffer was waited for here, and the next needs the P
            // of the S about to be issued into it
            if (ntiles >= kSBufs)
              mbar_wait_spin(smem_addr(&B.pv_done[sb.stage]), sb.phase ^ 1u, p.err, abort_flag);
            tc::fence_after_sync();
            issue_s_mma<D, F8>(tmem + sb.stage * kKeysPerTile, qd,
                           tc::Desc{kd0.lo + kv.stage * (KV_BYTES >> 4), kd0.hi});
            tc::commit(smem_addr(&B.s_full[sb.stage]));
            tc::commit(smem_addr(&B.k_empty[kv.stage]));
            if (kt == U.kt1 - 1) tc::commit(smem_addr(&B.q_empty));
            kv.next(SK);
            sb.next(kSBufs);
          }
          ++n_out;
        }
        if (ntiles > 0) {
          tc::commit(smem_addr(&B.s_done));  // its only use: phase 0
          mbar_wait_spin(smem_addr(&B.s_done), 0, p.err, abort_flag);
        }
      } else {
        // O += P V with P in the S buffer at sb and V at kv; the first tile of
        // a unit overwrites O once the previous unit's epilogue has read it
        const tc::Desc vd0 = tc::sw128_desc_pair(smem_addr(v_s), kBlock * 128, 1024);
        for (long long u = blockIdx.x; u < total_units; u += gridDim.x) {
          Unit U;
          if (!cur.locate(p, u, U)) break;
          if (U.kt0 == U.kt1) continue;
          for (int kt = U.kt0; kt < U.kt1; ++kt, ++ntiles) {
            const bool first = kt == U.kt0;
            // P of this tile: the buffer's last P was waited for here, and
            // its next P needs an S that waits for this P V (pv_done)
            mbar_wait_spin(smem_addr(&B.p_full[sb.stage]), sb.phase, p.err, abort_flag);
            // V tile kt: the stage's last use was waited for here, and its
            // next copy waits for v_empty, committed below
            mbar_wait_spin(smem_addr(&B.v_full[kv.stage]), kv.phase, p.err, abort_flag);
            // the last unit's O read out: the release before was waited for
            // here, and the next needs this unit's O (o_full)
            if (first && n_out > 0)
              mbar_wait_spin(smem_addr(&B.o_empty), (n_out - 1) & 1, p.err, abort_flag);
            tc::fence_after_sync();
            issue_pv_mma<D, F8>(tmem + O_COL, tmem + sb.stage * kKeysPerTile,
                                tc::Desc{vd0.lo + kv.stage * (KV_BYTES >> 4), vd0.hi},
                            first);
            tc::commit(smem_addr(&B.v_empty[kv.stage]));
            tc::commit(smem_addr(&B.pv_done[sb.stage]));
            kv.next(SV);
            sb.next(kSBufs);
          }
          tc::commit(smem_addr(&B.o_full));
          ++n_out;
        }
        if (ntiles > 0) {
          tc::commit(smem_addr(&B.pv_done_all));  // its only use: phase 0
          mbar_wait_spin(smem_addr(&B.pv_done_all), 0, p.err, abort_flag);
        }
      }
    }
  } else {
    // ============================================================ softmax
    const int quarter = warp & 3;    // TMEM lanes 32*quarter .. +31
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
    UnitCursor<TM> cur;
    cur.init(p, B.list_seq, B.list_base, B.listed);
    int n_out = 0;
    Ring sbr, prev, prev2, vr;  // S buffer of this tile, the last one and the one
                                // before; V stage of this tile
    uint32_t xpar = 0;          // exchange slot parity
    uint32_t nt = 0;            // tiles done by this CTA
    for (long long u = blockIdx.x; u < total_units; u += gridDim.x) {
      Unit U;
      if (!cur.locate(p, u, U)) break;
      const bool row_valid = tl < U.ntok;
      const int64_t row = (int64_t)(U.q0 + tl) * p.n_q + U.g * G + hl;
      if (U.kt0 == U.kt1) {
        // a key split with no tile (fewer tiles than splits): an empty piece
        if (kh == 0 && row_valid)
          *reinterpret_cast<float2*>(p.part_ml + (row * p.nsplit + U.ks) * 2) =
              make_float2(kNegInf, 0.f);
        continue;
      }
      const int p_row = row_valid ? U.p_first + tl : U.kv_end - 1;
      float m_ref = kNegInf, l = 0.f;
      for (int kt = U.kt0; kt < U.kt1; ++kt) {
        const uint32_t s_cols = tmem + lane_addr + sbr.stage * kKeysPerTile + kh * 64;
        // S of this tile: the buffer's last S was waited for here, and its
        // next S waits for the P V of this tile, which needs this P
        mbar_wait(smem_addr(&B.s_full[sbr.stage]), sbr.phase, p.err, abort_flag);
        tc::fence_after_sync();
        uint32_t sr[64];
        tc::tmem_ld32(s_cols, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tc::tmem_ld32(s_cols + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tc::tmem_wait_ld();

        // causal mask and the max of this half (three-input max, 4 chains)
        const int lim = p_row - (kt * kKeysPerTile + kh * 64);  // keys c <= lim visible
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
        float m4[4] = {kNegInf, kNegInf, kNegInf, kNegInf};
#pragma unroll
        for (int c = 0; c < 64; c += 8) {
          const int q = (c >> 3) & 3;
          m4[q] = fmax3(m4[q], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
          m4[q] = fmax3(m4[q], __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
          m4[q] = fmax3(m4[q], __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
          m4[q] = fmax3(m4[q], __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
        }
        const float mh = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        // swap the half maxima with the other warp on these rows (slots
        // alternate with the tile parity, so a slot is rewritten only after a
        // later barrier)
        B.xmax[xpar][kh][r] = mh;
        named_barrier(pair_bar, 64);
        float mx = fmaxf(mh, B.xmax[xpar][kh ^ 1][r]);
        mx = (mx == kNegInf) ? kNegInf : mx * emul;  // now in scaled base-2 units
        // both warps of the pair see the same maxima and take the same branch
        float alpha = 1.f;
        if (m_ref == kNegInf) {
          m_ref = mx;  // first tile with a visible key: O holds zeros so far
        } else if (mx > m_ref + kRescaleThreshold) {
          alpha = fast_exp2(m_ref - mx);
          l *= alpha;
          m_ref = mx;
        }
        // p = 2^(emul * s - m_ref), packed in bf16 pairs (f16 for the 8-bit
        // cache) in place (sr[j] holds keys 2j, 2j+1 of this half), stored over
        // the first 32 columns of the half; a row with no visible key so far
        // gets p = 0.  The row sum adds the rounded values the P V product
        // uses, so that the output is an exact
        // convex combination of V rows with those weights (summing the fp32
        // values instead leaves numerator and denominator 2^-9 apart, which
        // rows with few keys of large values showed as errors past 1e-2)
        const float mu = (m_ref == kNegInf) ? 0.f : m_ref;
        const float2 e2 = make_float2(emul, emul);
        const float2 nm2 = make_float2(-mu, -mu);
        float2 l4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) l4[j] = make_float2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float2 x = __ffma2_rn(
              make_float2(__uint_as_float(sr[2 * j]), __uint_as_float(sr[2 * j + 1])), e2, nm2);
          if constexpr (F8) {
            sr[j] = f16x2_from_floats(fast_exp2(x.x), fast_exp2(x.y));
            add_f16x2_to(l4[j & 3], sr[j]);
          } else {
            sr[j] = pack_bf16x2(fast_exp2(x.x), fast_exp2(x.y));
            add_bf16x2_to(l4[j & 3], sr[j]);
          }
        }
        tc::tmem_st32(s_cols, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        l += ((l4[0].x + l4[0].y) + (l4[1].x + l4[1].y)) +
             ((l4[2].x + l4[2].y) + (l4[3].x + l4[3].y));

        // rescale this half of the running output when the reference max moved
        // (rare); the P V product of the last tile must have landed first
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          // P V of the last tile: the buffer's use before (kSBufs tiles
          // earlier) was waited for by the S issued into this tile's buffer,
          // whose S these warps waited for; the next needs a later P
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
        // poisoned data; zero them so that P = 0 times V stays 0.  Thread r
        // clears half of the 16-byte chunks of V row 64 kh + r / 2.
        const int kv_local = U.kv_end - kt * kKeysPerTile;
        if (kv_local < kKeysPerTile) {
          // A parity wait tells apart only two phases in a row: the stage's
          // barrier must be at this tile's use or the one after, never still
          // at the use SV tiles back (its phase has this tile's parity, and
          // the wait would pass before this tile's V landed).  These warps
          // wait on V at tail tiles only, so nothing else keeps them from
          // running ahead of the V copies.  The P V product of that earlier
          // tile has read its use: with SV >= kSBufs the S of this tile
          // waited for it already (its buffer's last P V); with SV == 2 wait
          // for it here.  (The V barrier cannot be past this tile's use: the
          // next copy into the stage waits for this tile's P V, which waits
          // for this tile's P.)
          static_assert(SV >= kSBufs || (SV == 2 && kSBufs >= 3), "the P V SV tiles back");
          if constexpr (SV < kSBufs) {
            if (nt >= 2)
              mbar_wait(smem_addr(&B.pv_done[prev2.stage]), prev2.phase, p.err, abort_flag);
          }
          mbar_wait(smem_addr(&B.v_full[vr.stage]), vr.phase, p.err, abort_flag);
          const int key = kh * 64 + (r >> 1);
          if (key >= kv_local) {
            unsigned char* vpage = v_s + vr.stage * KV_BYTES + (key >> 4) * V_PAGE;
#pragma unroll
            for (int h = 0; h < NH; ++h)
#pragma unroll
              for (int c8 = 4 * (r & 1); c8 < 4 * (r & 1) + 4; ++c8)
                *reinterpret_cast<uint4*>(vpage + h * (kBlock * 128) + sw128_chunk(key & 15, c8)) =
                    make_uint4(0, 0, 0, 0);
          }
        }
        tc::tmem_wait_st();
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&B.p_full[sbr.stage]));
        prev2 = prev;
        prev = sbr;
        sbr.next(kSBufs);
        vr.next(SV);
        xpar ^= 1u;
        ++nt;
      }
      // epilogue: each warp of the pair handles half of d
      const uint32_t upar = n_out & 1;
      B.xsum[upar][kh][r] = l;
      named_barrier(pair_bar, 64);
      const float ltot = l + B.xsum[upar][kh ^ 1][r];
      const float inv = ltot > 0.f ? 1.f / ltot : 0.f;
      // this unit's O: the last unit's was waited for here, and the next
      // unit's first P V waits for o_empty, which these warps arrive on
      mbar_wait(smem_addr(&B.o_full), upar, p.err, abort_flag);
      tc::fence_after_sync();
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t o[32];
        tc::tmem_ld32(tmem + lane_addr + O_COL + kh * (D / 2) + c * 32, o);
        tc::tmem_wait_ld();
        if (!row_valid) continue;
        if (p.nsplit == 1) {
          uint16_t* orow = p.out + row * D + kh * (D / 2) + c * 32;
#pragma unroll
          for (int j = 0; j < 32; j += 8) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(o[j + 4]) * inv, __uint_as_float(o[j + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(o[j + 6]) * inv, __uint_as_float(o[j + 7]) * inv);
            *reinterpret_cast<uint4*>(orow + j) = w;
          }
        } else {
          float* prow = p.part_o + (row * p.nsplit + U.ks) * D + kh * (D / 2) + c * 32;
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(prow + j) =
                make_float4(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv,
                            __uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv);
        }
      }
      if (p.nsplit > 1 && kh == 0 && row_valid)
        *reinterpret_cast<float2*>(p.part_ml + (row * p.nsplit + U.ks) * 2) =
            make_float2(ltot > 0.f ? m_ref : kNegInf, ltot);
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&B.o_empty));
      ++n_out;
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

// Combines the key-split pieces of the prefill rows: one warp per (token, q
// head) of a request with q_len >= 2; out = sum_i w_i (O_i / l_i) / sum_i w_i
// with w_i = l_i 2^(m_i - max m).  Pieces with l = 0 saw no key.
template <int D>
__global__ void __launch_bounds__(256) prefill_merge_kernel(const PrefillParams p) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  constexpr int E = D / 32;  // columns per lane
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= (long long)p.num_tokens * p.n_q) return;
  const int token = (int)(row / p.n_q);
  if (token < __ldg(p.qsl) || token >= __ldg(p.qsl + p.num_seqs)) return;
  // the request of this token: the last s with qsl[s] <= token
  int lo = 0, hi = p.num_seqs;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(p.qsl + mid) <= token)
      lo = mid;
    else
      hi = mid;
  }
  int a, ql, L;
  if (!prefill_request(p, lo, a, ql, L, false)) return;
  const int ns = p.nsplit;
  float m[kMaxSplit], w[kMaxSplit];
  float mmax = kNegInf;
#pragma unroll
  for (int i = 0; i < kMaxSplit; ++i) {
    m[i] = kNegInf;
    w[i] = 0.f;
    if (i < ns) {
      const float2 ml = *reinterpret_cast<const float2*>(p.part_ml + (row * ns + i) * 2);
      if (ml.y > 0.f) {
        m[i] = ml.x;
        w[i] = ml.y;
        mmax = fmaxf(mmax, ml.x);
      }
    }
  }
  float wsum = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxSplit; ++i) {
    w[i] = w[i] > 0.f ? w[i] * fast_exp2(m[i] - mmax) : 0.f;
    wsum += w[i];
  }
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxSplit; ++i) {
    if (w[i] > 0.f) {
      const float* o = p.part_o + (row * ns + i) * D + lane * E;
#pragma unroll
      for (int e = 0; e < E; e += 2) {
        const float2 v = *reinterpret_cast<const float2*>(o + e);
        acc[e] = fmaf(w[i], v.x, acc[e]);
        acc[e + 1] = fmaf(w[i], v.y, acc[e + 1]);
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint16_t* orow = p.out + row * D + lane * E;
  if constexpr (E == 4) {
    *reinterpret_cast<uint2*>(orow) = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                                 pack_bf16x2(acc[2] * inv, acc[3] * inv));
  } else {
    *reinterpret_cast<uint32_t*>(orow) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
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

// bf16 tensor map with the 128-byte swizzle (the box's inner extent is 64).
cudaError_t make_map(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims,
                     const cuuint64_t* strides, const cuuint32_t* box) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return cudaErrorNotSupported;
  const cuuint32_t es[4] = {1, 1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), dims,
                         strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int D, int G>
size_t prefill_smem_bytes() {
  constexpr size_t half = kRows * 128;
  return 1024 + (size_t)(D / 64) * half * (1 + kStagesK + kStagesV) + sizeof(PrefillShared);
}

size_t split_bytes(int num_tokens, int num_q_heads, int head_dim, int nsplit) {
  if (nsplit <= 1) return 0;
  const size_t rows = (size_t)num_tokens * num_q_heads * nsplit;
  return ((rows * head_dim * sizeof(float) + 255) & ~size_t(255)) +
         ((rows * 2 * sizeof(float) + 255) & ~size_t(255));
}

template <int D, int G, int KIND>
cudaError_t launch_prefill_t(const AttnArgs& a, const PrefillPlan& plan, void* ws, int sm_count,
                             cudaStream_t stream) {
  constexpr bool FUSE = KIND == kKindFused;
  constexpr bool F8 = KIND == kKindFp8;
  constexpr int TM = kRows / G;
  PrefillParams p;
  p.k_new = a.fuse_k_new;
  p.v_new = a.fuse_v_new;
  p.slot_mapping = a.fuse_slot_mapping;
  p.k_cache = F8 ? nullptr : static_cast<uint16_t*>(const_cast<void*>(a.k_cache));
  p.v_cache = F8 ? nullptr : static_cast<uint16_t*>(const_cast<void*>(a.v_cache));
  p.k_codes = F8 ? static_cast<const uint8_t*>(a.k_cache) : nullptr;
  p.v_codes = F8 ? static_cast<const uint8_t*>(a.v_cache) : nullptr;
  p.block_tables = a.block_tables;
  p.seq_lens = a.seq_lens;
  p.qsl = a.query_start_loc;
  p.out = a.out;
  p.part_o = nullptr;
  p.part_ml = nullptr;
  p.err = a.err;
  p.num_blocks = a.num_blocks;
  p.max_blocks = a.max_blocks;
  p.num_seqs = a.num_seqs;
  p.num_tokens = a.num_tokens;
  p.n_q = a.num_q_heads;
  p.n_kv = a.num_kv_heads;
  p.max_seq_len = a.max_seq_len;
  p.block_shift = a.block_shift;
  p.no_decode = a.no_decode ? 1 : 0;
  p.nsplit = plan.nsplit;
  // the 8-bit instance scales the query tile itself (f16 operands), so its
  // scores arrive in base-2 units
  p.q_mul = a.scale * 1.4426950408889634f;
  p.scale_log2 = F8 ? 1.f : p.q_mul;
  if (plan.nsplit > 1) {
    const size_t rows = (size_t)a.num_tokens * a.num_q_heads * plan.nsplit;
    p.part_o = static_cast<float*>(ws);
    p.part_ml = reinterpret_cast<float*>(static_cast<unsigned char*>(ws) +
                                         ((rows * D * sizeof(float) + 255) & ~size_t(255)));
  }
  const cuuint64_t nkv = (cuuint64_t)a.num_kv_heads;
  const cuuint64_t rows = ((cuuint64_t)a.num_blocks << a.block_shift) * kBlock;
  CUtensorMap qm, km, vm, knm, vnm;
  {
    const cuuint64_t dims[3] = {D, (cuuint64_t)a.num_q_heads, (cuuint64_t)a.num_tokens};
    const cuuint64_t strides[2] = {D * 2, (cuuint64_t)a.num_q_heads * D * 2};
    const cuuint32_t box[3] = {64, G, TM};
    cudaError_t e = make_map(&qm, a.q, 3, dims, strides, box);
    if (e != cudaSuccess) return e;
  }
  // (the 8-bit instance reads its pages with plain loads: no cache maps)
  km = vm = qm;
  if (!F8) {
    const cuuint64_t dims[3] = {D, nkv, rows};
    const cuuint64_t strides[2] = {D * 2, nkv * D * 2};
    const cuuint32_t box[3] = {64, 1, kBlock};
    cudaError_t e = make_map(&km, a.k_cache, 3, dims, strides, box);
    if (e != cudaSuccess) return e;
    if (D == 64) {
      e = make_map(&vm, a.v_cache, 3, dims, strides, box);
      if (e != cudaSuccess) return e;
    }
  }
  if (!F8 && D == 128) {
    // one box per page with both 64-column halves, the half as the outermost
    // box dimension: shared-memory layout [half][16 tokens][64]
    const cuuint64_t dims[4] = {64, nkv, rows, 2};
    const cuuint64_t strides[3] = {D * 2, nkv * D * 2, 128};
    const cuuint32_t box[4] = {64, 1, kBlock, 2};
    cudaError_t e = make_map(&vm, a.v_cache, 4, dims, strides, box);
    if (e != cudaSuccess) return e;
  }
  knm = km;
  vnm = vm;
  if (FUSE) {
    // the step's new rows [num_tokens, n_kv, D], read with the caches' boxes:
    // 16 consecutive tokens of one kv head
    const cuuint64_t tok = (cuuint64_t)a.num_tokens;
    {
      const cuuint64_t dims[3] = {D, nkv, tok};
      const cuuint64_t strides[2] = {D * 2, nkv * D * 2};
      const cuuint32_t box[3] = {64, 1, kBlock};
      cudaError_t e = make_map(&knm, a.fuse_k_new, 3, dims, strides, box);
      if (e != cudaSuccess) return e;
      if (D == 64) {
        e = make_map(&vnm, a.fuse_v_new, 3, dims, strides, box);
        if (e != cudaSuccess) return e;
      }
    }
    if (D == 128) {
      const cuuint64_t dims[4] = {64, nkv, tok, 2};
      const cuuint64_t strides[3] = {D * 2, nkv * D * 2, 128};
      const cuuint32_t box[4] = {64, 1, kBlock, 2};
      cudaError_t e = make_map(&vnm, a.fuse_v_new, 4, dims, strides, box);
      if (e != cudaSuccess) return e;
    }
  }
  // upper bound of the number of units; the kernel reads the exact count
  const long long tiles_bound = (long long)a.num_tokens / TM + a.num_seqs;
  const long long units_bound = tiles_bound * a.num_kv_heads * plan.nsplit;
  const int grid = (int)(units_bound < sm_count ? units_bound : sm_count);
  if (grid <= 0) return cudaSuccess;
  const size_t smem = prefill_smem_bytes<D, G>();
  auto kern = prefill_kernel<D, G, KIND>;
  static int configured_device = -1;
  int dev = 0;
  cudaGetDevice(&dev);
  if (configured_device != dev) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured_device = dev;
  }
  kern<<<grid, kThreads, smem, stream>>>(p, qm, km, vm, knm, vnm);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || plan.nsplit == 1) return e;
  // the merge may launch while the prefill grid runs; it waits for that grid
  // with griddepcontrol.wait before reading a piece
  const long long mrows = (long long)a.num_tokens * a.num_q_heads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((mrows + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, prefill_merge_kernel<D>, p);
}

}  // namespace

// The 8-bit cache's instance (pa_prefill_fp8.cu).
cudaError_t launch_prefill_fp8(const AttnArgs& a, const PrefillPlan& plan, void* ws,
                               int sm_count, cudaStream_t stream);

}  // namespace pa
