/*
 * oracle.c -- plain, slow, fp64 CPU definition of attention over a paged KV
 * cache, of the slot scatter that fills the cache, and of the copy-on-write
 * block copy.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file.  It is used by the tests, by the smoke check and by the
 * benchmark's CPU-baseline / reference arm, and by nothing else.  It shares no
 * code, header, table or constant with the CUDA library: it decodes bfloat16
 * itself and computes everything in double precision with plain loops.
 *
 * Sources (the pages this follows, by title and section):
 *  [bxagent] "PagedAttention 显存分页与连续批处理(Continuous Batching)实战",
 *            "PagedAttention 核心机理" part 1 (logical vs physical blocks, the
 *            Block Table, a 48-token sequence = logical blocks 0..2) and
 *            part 2 (the kernel reads the Block Table and turns a logical
 *            index into a physical block pointer), and the comparison table
 *            there (on-demand block allocation, copy-on-write sharing).
 *  [guijiagi] "连续批处理：推理吞吐的范式革命", section 3.3 (preemption by
 *            swapping: a request's KV cache moves to CPU memory and comes back
 *            without recomputation), section 4.1 (the paged
 *            attention kernel: q [num_tokens, d], key/value caches
 *            [num_blocks, block_size, d], block_tables
 *            [num_requests, max_blocks], seq_lens [num_requests]; walk the
 *            request's blocks, score = q.k / sqrt(d_k), softmax, weighted sum
 *            of v, normalise), section 4.2 (prefix sharing).
 *
 * Readings taken where the pages are silent or inconsistent (each one is
 * listed with its reason in the design notes of the repository):
 *  - softmax is the textbook definition (max, exp, sum, divide); the page's
 *    online update is an implementation strategy and, as printed, forgets to
 *    rescale its running sum, so it is not followed;
 *  - the score scale is an argument (the page hard-codes 1/sqrt(d_k));
 *  - cache layout is [num_blocks, block_size, num_kv_heads, head_dim];
 *  - grouped-query attention maps q head h to kv head h / (n_q / n_kv);
 *  - seq_lens counts every cached token of the request including this step's
 *    new tokens; query row i of a request with q_len rows sits at position
 *    p = seq_len - q_len + i and attends to keys 0..p (bottom-right causal);
 *  - a negative slot in slot_mapping means "skip this token";
 *  - copy_blocks applies its (src, dst) pairs one after the other.
 *  - swap works on whole blocks ("vLLM中的PagedAttention机制与显存优化实践",
 *    section 2.1: swap is block-grained): swap-out packs the listed blocks,
 *    in list order, into host arrays [n, block_size, num_kv_heads, head_dim];
 *    swap-in writes the host arrays' blocks back at the listed block ids.
 *
 * The 8-bit cache variant is not on the pages.  It stores each cached key or
 * value row (one token, one kv head: head_dim values) as FP8 E4M3 codes plus
 * one fp32 scale, so that a cache of the same layout holds half the bytes.
 * Its definition, written out below: E4M3 is the 8-bit format with 1 sign
 * bit, 4 exponent bits of bias 7 and 3 mantissa bits, no infinities, the
 * all-ones exponent and mantissa pattern as NaN, largest finite magnitude 448
 * and subnormals m * 2^-9; a row x quantises to scale = max_c |x_c| / 448
 * (1 for an all-zero row) and codes round_e4m3(x_c / scale), rounding to
 * nearest with ties to even and saturating at +-448; the divisions are fp32,
 * which fixes every code; attention then uses code * scale in place of the
 * bfloat16 value.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
  ORACLE_OK = 0,
  ORACLE_ERR_ARG = 1,   /* a size or pointer argument is invalid          */
  ORACLE_ERR_INDEX = 2, /* a slot, block id or length is out of its range  */
  ORACLE_ERR_NOMEM = 3
};

/* bfloat16 is the top 16 bits of an IEEE-754 binary32 value. */
static double bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* E4M3 code -> value (exact in double). */
double oracle_e4m3_to_double(uint8_t code) {
  const int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m, -9); /* subnormal: m/8 * 2^(1-7) */
  else
    mag = ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -mag : mag;
}

/* fp32 value -> E4M3 code, rounding to nearest (ties to even), saturating at
 * the largest finite magnitude; NaN -> 0x7f.  The quantum (spacing of codes)
 * is 2^-9 below 2^-6 and 2^(e-3) in the binade [2^e, 2^(e+1)), so the value
 * rounds to an integer multiple of its binade's quantum; a value rounded up to
 * the next power of two is still a multiple of the new binade's quantum. */
uint8_t oracle_e4m3_from_float(float y) {
  if (isnan(y)) return 0x7f;
  const int sign = signbit(y) ? 1 : 0;
  double a = fabs((double)y);
  double q;
  if (a < ldexp(1.0, -6)) {
    q = ldexp(1.0, -9);
  } else {
    int e;
    frexp(a, &e); /* a = f * 2^e, f in [0.5, 1): a in [2^(e-1), 2^e) */
    q = ldexp(1.0, e - 1 - 3);
  }
  double v = nearbyint(a / q) * q; /* a / q is exact; nearbyint: ties to even */
  if (v > 448.0) v = 448.0;
  uint8_t bits;
  if (v < ldexp(1.0, -6)) {
    bits = (uint8_t)(v / ldexp(1.0, -9)); /* 0..8; 8 means 2^-6, the first normal */
    if (bits == 8) bits = (uint8_t)(1 << 3);
  } else {
    int e;
    double f = frexp(v, &e); /* v = f * 2^e, f in [0.5, 1) */
    int ebias = (e - 1) + 7;
    int m = (int)((f * 2.0 - 1.0) * 8.0);
    bits = (uint8_t)((ebias << 3) | m);
  }
  return (uint8_t)(bits | (sign << 7));
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Block addressing ([bxagent] part 1; [guijiagi] 4.1): logical position pos of
 * a request lives in logical block pos / block_size, which the Block Table
 * maps to a physical block; inside it, the token is row pos % block_size.
 * Returns the flat slot index phys * block_size + row. */
int64_t oracle_slot_of(const int32_t *block_table_row, int32_t pos,
                       int32_t block_size) {
  int32_t logical = pos / block_size;
  int32_t row = pos % block_size;
  return (int64_t)block_table_row[logical] * block_size + row;
}

/* Slot scatter: for each new token t with slot s = slot_mapping[t] >= 0, copy
 * its key and value rows (num_kv_heads * head_dim bfloat16 values each) to
 * slot s of the caches.  A bit copy. */
int oracle_reshape_and_cache(const uint16_t *k, const uint16_t *v,
                             int32_t num_tokens, uint16_t *k_cache,
                             uint16_t *v_cache, int32_t num_blocks,
                             int32_t block_size, int32_t num_kv_heads,
                             int32_t head_dim, const int32_t *slot_mapping) {
  if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 ||
      num_kv_heads <= 0 || head_dim <= 0)
    return ORACLE_ERR_ARG;
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  const int64_t num_slots = (int64_t)num_blocks * block_size;
  for (int32_t t = 0; t < num_tokens; ++t) {
    int64_t s = slot_mapping[t];
    if (s < 0) continue;
    if (s >= num_slots) return ORACLE_ERR_INDEX;
    for (int64_t c = 0; c < row; ++c) {
      k_cache[s * row + c] = k[(int64_t)t * row + c];
      v_cache[s * row + c] = v[(int64_t)t * row + c];
    }
  }
  return ORACLE_OK;
}

/* The 8-bit cache's scatter: like oracle_reshape_and_cache, but each
 * (token, kv head) row of head_dim values is quantised (see the header):
 * scale = max |x| / 448 in fp32 (1 if the row is all zero), code_c =
 * round_e4m3(x_c / scale) with the division in fp32.  Codes go to
 * k_cache / v_cache [num_blocks, block_size, num_kv_heads, head_dim] (bytes),
 * scales to k_scale / v_scale [num_blocks, block_size, num_kv_heads]. */
static void quantise_row(const uint16_t *x, int32_t n, uint8_t *codes, float *scale) {
  float amax = 0.0f;
  for (int32_t c = 0; c < n; ++c) {
    float a = fabsf((float)bf16_to_double(x[c]));
    if (a > amax) amax = a;
  }
  float sc = amax > 0.0f ? amax / 448.0f : 1.0f;
  for (int32_t c = 0; c < n; ++c)
    codes[c] = oracle_e4m3_from_float((float)bf16_to_double(x[c]) / sc);
  *scale = sc;
}

int oracle_reshape_and_cache_fp8(const uint16_t *k, const uint16_t *v, int32_t num_tokens,
                                 uint8_t *k_cache, uint8_t *v_cache, float *k_scale,
                                 float *v_scale, int32_t num_blocks, int32_t block_size,
                                 int32_t num_kv_heads, int32_t head_dim,
                                 const int32_t *slot_mapping) {
  if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 ||
      num_kv_heads <= 0 || head_dim <= 0)
    return ORACLE_ERR_ARG;
  const int64_t num_slots = (int64_t)num_blocks * block_size;
  for (int32_t t = 0; t < num_tokens; ++t) {
    int64_t s = slot_mapping[t];
    if (s < 0) continue;
    if (s >= num_slots) return ORACLE_ERR_INDEX;
    for (int32_t g = 0; g < num_kv_heads; ++g) {
      int64_t src = ((int64_t)t * num_kv_heads + g) * head_dim;
      int64_t dst = (s * num_kv_heads + g) * head_dim;
      quantise_row(k + src, head_dim, k_cache + dst, k_scale + s * num_kv_heads + g);
      quantise_row(v + src, head_dim, v_cache + dst, v_scale + s * num_kv_heads + g);
    }
  }
  return ORACLE_OK;
}

/* Copy-on-write block copy ([bxagent] comparison table, "Copy-on-Write";
 * [guijiagi] 4.2): for each pair, in order, physical block dst of both caches
 * becomes a bit copy of physical block src. */
int oracle_copy_blocks(uint16_t *k_cache, uint16_t *v_cache, int32_t num_blocks,
                       int32_t block_size, int32_t num_kv_heads,
                       int32_t head_dim, const int32_t *src_dst_pairs,
                       int32_t num_pairs) {
  if (num_pairs < 0 || num_blocks <= 0 || block_size <= 0 ||
      num_kv_heads <= 0 || head_dim <= 0)
    return ORACLE_ERR_ARG;
  const int64_t blk = (int64_t)block_size * num_kv_heads * head_dim;
  for (int32_t i = 0; i < num_pairs; ++i) {
    int64_t src = src_dst_pairs[2 * i];
    int64_t dst = src_dst_pairs[2 * i + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks)
      return ORACLE_ERR_INDEX;
    for (int64_t c = 0; c < blk; ++c) {
      k_cache[dst * blk + c] = k_cache[src * blk + c];
      v_cache[dst * blk + c] = v_cache[src * blk + c];
    }
  }
  return ORACLE_OK;
}

/* Swap-out: host_k[i], host_v[i] <- K and V of block ids[i], for i < n (a
 * bit copy of each block; ids may repeat). */
int oracle_swap_out(const uint16_t *k_cache, const uint16_t *v_cache, int32_t num_blocks,
                    int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                    const int32_t *ids, int32_t n, uint16_t *host_k, uint16_t *host_v) {
  if (n < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return ORACLE_ERR_ARG;
  const int64_t blk = (int64_t)block_size * num_kv_heads * head_dim;
  for (int32_t i = 0; i < n; ++i) {
    const int64_t b = ids[i];
    if (b < 0 || b >= num_blocks) return ORACLE_ERR_INDEX;
    for (int64_t c = 0; c < blk; ++c) {
      host_k[i * blk + c] = k_cache[b * blk + c];
      host_v[i * blk + c] = v_cache[b * blk + c];
    }
  }
  return ORACLE_OK;
}

/* Swap-in: K and V of block ids[i] <- host_k[i], host_v[i], for i < n in
 * order (ids should be distinct; with repeats the last one wins). */
int oracle_swap_in(uint16_t *k_cache, uint16_t *v_cache, int32_t num_blocks,
                   int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                   const int32_t *ids, int32_t n, const uint16_t *host_k,
                   const uint16_t *host_v) {
  if (n < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
    return ORACLE_ERR_ARG;
  const int64_t blk = (int64_t)block_size * num_kv_heads * head_dim;
  for (int32_t i = 0; i < n; ++i) {
    const int64_t b = ids[i];
    if (b < 0 || b >= num_blocks) return ORACLE_ERR_INDEX;
  }
  for (int32_t i = 0; i < n; ++i) {
    const int64_t b = ids[i];
    for (int64_t c = 0; c < blk; ++c) {
      k_cache[b * blk + c] = host_k[i * blk + c];
      v_cache[b * blk + c] = host_v[i * blk + c];
    }
  }
  return ORACLE_OK;
}

/* Geometry of one paged-attention call, as plain values. */
typedef struct {
  const uint16_t *q;       /* [num_tokens, num_q_heads, head_dim]             */
  const uint16_t *k_cache; /* [num_blocks, block_size, num_kv_heads, head_dim] */
  const uint16_t *v_cache; /* same layout as k_cache                           */
  int32_t num_blocks, block_size, num_q_heads, num_kv_heads, head_dim;
  const int32_t *block_tables; /* [num_seqs, max_blocks]                       */
  int32_t max_blocks;
  const int32_t *seq_lens;        /* [num_seqs]                                */
  const int32_t *query_start_loc; /* [num_seqs + 1]                            */
  int32_t num_seqs;
  double scale;
  /* 8-bit cache (k_cache / v_cache unused when k8 is set) */
  const uint8_t *k8, *v8;         /* codes, same layout as k_cache             */
  const float *k_scale, *v_scale; /* [num_blocks, block_size, num_kv_heads]   */
} oracle_geom;

/* Value c of the cached row (slot, kv head g) of the key (is_v = 0) or value
 * cache. */
static double cached(const oracle_geom *G, int is_v, int64_t slot, int32_t g, int32_t c) {
  const int64_t row = slot * G->num_kv_heads + g;
  if (G->k8) {
    const uint8_t *codes = is_v ? G->v8 : G->k8;
    const float *sc = is_v ? G->v_scale : G->k_scale;
    return oracle_e4m3_to_double(codes[row * G->head_dim + c]) * (double)sc[row];
  }
  const uint16_t *cache = is_v ? G->v_cache : G->k_cache;
  return bf16_to_double(cache[row * G->head_dim + c]);
}

/* One output row: sequence s, query row i of that sequence, q head h.
 * scratch holds at least seq_len doubles.  Writes head_dim doubles to out.
 *
 *   p      = seq_len - q_len + i
 *   x_j    = scale * sum_c q[t,h,c] * K[j,g,c],       j = 0..p
 *   w_j    = exp(x_j - max_j x_j)
 *   out_c  = sum_j w_j * V[j,g,c] / sum_j w_j
 *
 * with K[j] / V[j] read through the Block Table ([guijiagi] 4.1:
 * physical_block = block_tables[req][j / block_size], row j % block_size). */
static int attention_row(const oracle_geom *G, int32_t s, int32_t i, int32_t h,
                         double *scratch, double *out) {
  const int32_t q_len = G->query_start_loc[s + 1] - G->query_start_loc[s];
  const int32_t seq_len = G->seq_lens[s];
  if (i < 0 || i >= q_len) return ORACLE_ERR_INDEX;
  if (q_len > seq_len) return ORACLE_ERR_INDEX;
  if ((int64_t)seq_len > (int64_t)G->max_blocks * G->block_size)
    return ORACLE_ERR_INDEX;
  const int32_t group = G->num_q_heads / G->num_kv_heads;
  const int32_t g = h / group;
  const int32_t d = G->head_dim;
  const int64_t t = (int64_t)G->query_start_loc[s] + i;
  const int32_t p = seq_len - q_len + i;
  const uint16_t *qrow = G->q + (t * G->num_q_heads + h) * d;
  const int32_t *table = G->block_tables + (int64_t)s * G->max_blocks;

  /* scores */
  for (int32_t j = 0; j <= p; ++j) {
    int32_t phys = table[j / G->block_size];
    if (phys < 0 || phys >= G->num_blocks) return ORACLE_ERR_INDEX;
    int64_t slot = (int64_t)phys * G->block_size + j % G->block_size;
    double acc = 0.0;
    for (int32_t c = 0; c < d; ++c)
      acc += bf16_to_double(qrow[c]) * cached(G, 0, slot, g, c);
    scratch[j] = G->scale * acc;
  }
  /* softmax */
  double m = -INFINITY;
  for (int32_t j = 0; j <= p; ++j)
    if (scratch[j] > m) m = scratch[j];
  double denom = 0.0;
  for (int32_t j = 0; j <= p; ++j) {
    scratch[j] = exp(scratch[j] - m);
    denom += scratch[j];
  }
  /* weighted sum of values */
  for (int32_t c = 0; c < d; ++c) out[c] = 0.0;
  for (int32_t j = 0; j <= p; ++j) {
    int32_t phys = table[j / G->block_size];
    int64_t slot = (int64_t)phys * G->block_size + j % G->block_size;
    for (int32_t c = 0; c < d; ++c) out[c] += scratch[j] * cached(G, 1, slot, g, c);
  }
  for (int32_t c = 0; c < d; ++c) out[c] /= denom;
  return ORACLE_OK;
}

static int check_geom(const oracle_geom *G) {
  if (G->num_blocks <= 0 || G->block_size <= 0 || G->num_q_heads <= 0 ||
      G->num_kv_heads <= 0 || G->head_dim <= 0 || G->max_blocks < 0 ||
      G->num_seqs < 0)
    return ORACLE_ERR_ARG;
  if (G->num_q_heads % G->num_kv_heads != 0) return ORACLE_ERR_ARG;
  return ORACLE_OK;
}

/* Full paged attention: writes out[t, h, :] (fp64) for every query token t of
 * every sequence.  Rows of out that belong to no sequence are left untouched.
 * num_threads <= 0 means "all available". */
static int paged_attention(oracle_geom G, double *out, int32_t num_threads) {
  const int32_t num_q_heads = G.num_q_heads, head_dim = G.head_dim, num_seqs = G.num_seqs;
  const int32_t *query_start_loc = G.query_start_loc, *seq_lens = G.seq_lens;
  int st = check_geom(&G);
  if (st) return st;
  /* enumerate (sequence, row) pairs */
  int64_t rows = 0;
  int32_t max_len = 0;
  for (int32_t s = 0; s < num_seqs; ++s) {
    int32_t ql = query_start_loc[s + 1] - query_start_loc[s];
    if (ql < 0 || ql > seq_lens[s]) return ORACLE_ERR_INDEX;
    rows += ql;
    if (seq_lens[s] > max_len) max_len = seq_lens[s];
  }
  int32_t *row_seq = (int32_t *)malloc(sizeof(int32_t) * (rows ? rows : 1));
  int32_t *row_idx = (int32_t *)malloc(sizeof(int32_t) * (rows ? rows : 1));
  if (!row_seq || !row_idx) {
    free(row_seq);
    free(row_idx);
    return ORACLE_ERR_NOMEM;
  }
  int64_t r = 0;
  for (int32_t s = 0; s < num_seqs; ++s)
    for (int32_t i = 0; i < query_start_loc[s + 1] - query_start_loc[s]; ++i) {
      row_seq[r] = s;
      row_idx[r] = i;
      ++r;
    }
  const int64_t work = rows * num_q_heads;
  int status = ORACLE_OK;
#ifdef _OPENMP
  if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel num_threads(num_threads)
#endif
  {
    double *scratch = (double *)malloc(sizeof(double) * (max_len ? max_len : 1));
    if (!scratch) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      status = ORACLE_ERR_NOMEM;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 4)
#endif
      for (int64_t w = 0; w < work; ++w) {
        int64_t rr = w / num_q_heads;
        int32_t h = (int32_t)(w % num_q_heads);
        int32_t s = row_seq[rr];
        int32_t i = row_idx[rr];
        int64_t t = (int64_t)query_start_loc[s] + i;
        int e = attention_row(&G, s, i, h, scratch,
                              out + (t * num_q_heads + h) * head_dim);
        if (e) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
          status = e;
        }
      }
      free(scratch);
    }
  }
  free(row_seq);
  free(row_idx);
  return status;
}

int oracle_paged_attention(const uint16_t *q, const uint16_t *k_cache,
                           const uint16_t *v_cache, int32_t num_blocks,
                           int32_t block_size, int32_t num_q_heads,
                           int32_t num_kv_heads, int32_t head_dim,
                           const int32_t *block_tables, int32_t max_blocks,
                           const int32_t *seq_lens,
                           const int32_t *query_start_loc, int32_t num_seqs,
                           double scale, double *out, int32_t num_threads) {
  oracle_geom G = {q,          k_cache,       v_cache,         num_blocks,
                   block_size, num_q_heads,   num_kv_heads,    head_dim,
                   block_tables, max_blocks,  seq_lens,        query_start_loc,
                   num_seqs,   scale, NULL, NULL, NULL, NULL};
  return paged_attention(G, out, num_threads);
}

/* Paged attention over the 8-bit cache: every cached value is code * scale
 * of its row (see the header); the rest is oracle_paged_attention. */
int oracle_paged_attention_fp8(const uint16_t *q, const uint8_t *k_cache,
                               const uint8_t *v_cache, const float *k_scale,
                               const float *v_scale, int32_t num_blocks,
                               int32_t block_size, int32_t num_q_heads,
                               int32_t num_kv_heads, int32_t head_dim,
                               const int32_t *block_tables, int32_t max_blocks,
                               const int32_t *seq_lens, const int32_t *query_start_loc,
                               int32_t num_seqs, double scale, double *out,
                               int32_t num_threads) {
  oracle_geom G = {q,          NULL,          NULL,            num_blocks,
                   block_size, num_q_heads,   num_kv_heads,    head_dim,
                   block_tables, max_blocks,  seq_lens,        query_start_loc,
                   num_seqs,   scale, k_cache, v_cache, k_scale, v_scale};
  return paged_attention(G, out, num_threads);
}

/* Sampled paged attention: computes only the listed (sequence, row, head)
 * triples, so that very large calls can be checked one output row at a time.
 * out is [num_samples, head_dim]. */
int oracle_paged_attention_rows(const uint16_t *q, const uint16_t *k_cache,
                                const uint16_t *v_cache, int32_t num_blocks,
                                int32_t block_size, int32_t num_q_heads,
                                int32_t num_kv_heads, int32_t head_dim,
                                const int32_t *block_tables, int32_t max_blocks,
                                const int32_t *seq_lens,
                                const int32_t *query_start_loc, int32_t num_seqs,
                                double scale, const int32_t *samples /*[n,3]*/,
                                int32_t num_samples, double *out,
                                int32_t num_threads) {
  oracle_geom G = {q,          k_cache,       v_cache,         num_blocks,
                   block_size, num_q_heads,   num_kv_heads,    head_dim,
                   block_tables, max_blocks,  seq_lens,        query_start_loc,
                   num_seqs,   scale, NULL, NULL, NULL, NULL};
  int st = check_geom(&G);
  if (st) return st;
  int32_t max_len = 0;
  for (int32_t n = 0; n < num_samples; ++n) {
    int32_t s = samples[3 * n];
    if (s < 0 || s >= num_seqs) return ORACLE_ERR_INDEX;
    if (samples[3 * n + 2] < 0 || samples[3 * n + 2] >= num_q_heads)
      return ORACLE_ERR_INDEX;
    if (seq_lens[s] > max_len) max_len = seq_lens[s];
  }
  int status = ORACLE_OK;
#ifdef _OPENMP
  if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel num_threads(num_threads)
#endif
  {
    double *scratch = (double *)malloc(sizeof(double) * (max_len ? max_len : 1));
    if (!scratch) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
      status = ORACLE_ERR_NOMEM;
    } else {
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
      for (int32_t n = 0; n < num_samples; ++n) {
        int e = attention_row(&G, samples[3 * n], samples[3 * n + 1],
                              samples[3 * n + 2], scratch,
                              out + (int64_t)n * head_dim);
        if (e) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
          status = e;
        }
      }
      free(scratch);
    }
  }
  return status;
}
