/*
 * dsa_oracle.c -- plain, slow, single-threaded CPU oracle for the DSA sparse
 * attention hot path.  TEST INFRASTRUCTURE ONLY: nothing in the library's
 * product path may link, load or call this file.  It shares no code, header,
 * table or helper with the CUDA path; the two meet only through the seeded
 * inputs that tests and the benchmark hand to both.
 *
 * Sources followed (web pages on DSA sparse attention):
 *  [P1] "Day-0 Adaptation of Trillion-Parameter MoE Models on Domestic GPUs",
 *       section 3 "Adapting Sparse Attention (DSA)", items (1) Index Selection,
 *       (2) KV Cache Layout, (3) Two Compute Paths: Prefill and Decode.
 *  [P2] "Technical Path for Day-0 Adaptation of Trillion-Parameter Models on
 *       Domestic GPUs", section 3.1 "Implementing Sparse Attention".
 *  [P3] "Day-0 Adaptation of Ultra-Large-Scale MoE Models on Heterogeneous AI
 *       Accelerators", section 4 "Joint Debugging Essentials for the Sparse
 *       Attention Pipeline" (tie-break determinism, cache layout alignment).
 *
 * Arithmetic: every stored value is decoded exactly into a double; scores and
 * attention are accumulated in double.  The score of a position is rounded to
 * fp32 once, at the end, because the top-K decision is taken on fp32 scores
 * (the precision the scores are handed over in).  With the pages' integer
 * indexer inputs every score is an integer below 2^24, so the rounding is exact.
 *
 * Parity pins: see the "pins" tests; every function here is pinned by at least
 * one closed form, invariant, library special case or brute-force check.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR_ARG -1
#define OR_ERR_LAYOUT -2 /* block-table entry or position out of range */
#define OR_ERR_NAN -3    /* NaN score handed to the selector */

enum { OR_BF16 = 0, OR_FP8_E4M3 = 1 };

/* ---- exact decoders of the two storage formats ------------------------- */

/* bfloat16: the upper 16 bits of an IEEE-754 binary32. */
static double or_dec_bf16(uint16_t u) {
  uint32_t bits = (uint32_t)u << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* FP8 E4M3 (OCP 8-bit floating point, "fn" variant): 1 sign bit, 4 exponent
 * bits with bias 7, 3 mantissa bits; exponent field 0 encodes subnormals
 * m/8 * 2^-6; S.1111.111 is NaN; there are no infinities. */
static double or_dec_e4m3(uint8_t u) {
  int sign = (u >> 7) & 1;
  int e = (u >> 3) & 15;
  int m = u & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, 1 - 7);
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

static double or_load(const void* base, int dtype, int64_t i) {
  if (dtype == OR_BF16) return or_dec_bf16(((const uint16_t*)base)[i]);
  return or_dec_e4m3(((const uint8_t*)base)[i]);
}

/* Exported for the format pins. */
double oracle_decode(int dtype, uint32_t raw) {
  if (dtype == OR_BF16) return or_dec_bf16((uint16_t)raw);
  return or_dec_e4m3((uint8_t)raw);
}

/* ---- paged layout [P1 §3 (2)] ------------------------------------------
 * The cache is organised by page: a page holds `bs` consecutive positions
 * stored contiguously, and a per-sequence index table jumps between pages.
 * Position p of sequence b lives in physical row
 *     block_table[b][p / bs] * bs + p % bs.
 * Returns -1 when the table entry is outside [0, num_blocks). */
static int64_t or_phys_row(const int32_t* block_table, int max_blocks, int bs,
                           int num_blocks, int b, int64_t p) {
  int64_t slot = p / bs;
  if (slot >= max_blocks) return -1;
  int32_t page = block_table[(int64_t)b * max_blocks + slot];
  if (page < 0 || page >= num_blocks) return -1;
  return (int64_t)page * bs + (p % bs);
}

/* ---- stage 1: indexer score [P1 §3 (1); P2 §3.1 item 1] ----------------
 * Every cached position is scored by its similarity to the query, read as
 * the ReLU-weighted sum over indexer heads:
 *     s[r, p] = sum_h w[r, h] * max(0, sum_d q_idx[r, h, d] * k_idx[p, d])
 * for the positions p a query may attend to: p <= q_pos[r] and p < L_b
 * (causal: only historical positions, the current one included).  Every other
 * entry of the row, up to ld, is -inf.
 *
 * q_idx: [Nq][H][D] encoded (dtype); w: [Nq][H] fp32; kidx_pool:
 * [num_blocks][bs][D] encoded; scores: [Nq][ld] fp32 (output). */
int oracle_index_score(int batch, int bs, int num_blocks, int max_blocks,
                       const int32_t* block_table, const int32_t* seq_lens,
                       int Nq, const int32_t* q_seq, const int32_t* q_pos,
                       int H, int D, int dtype, const void* q_idx,
                       const float* w, const void* kidx_pool, int64_t ld,
                       float* scores) {
  if (batch <= 0 || bs <= 0 || Nq < 0 || H <= 0 || D <= 0 || ld <= 0)
    return OR_ERR_ARG;
  double* q = (double*)malloc(sizeof(double) * (size_t)H * D);
  double* k = (double*)malloc(sizeof(double) * (size_t)D);
  if (!q || !k) { free(q); free(k); return OR_ERR_ARG; }
  int rc = OR_OK;
  for (int r = 0; r < Nq; ++r) {
    int b = q_seq[r];
    if (b < 0 || b >= batch) { rc = OR_ERR_ARG; break; }
    int64_t L = seq_lens[b];
    int64_t last = q_pos[r]; /* inclusive */
    if (last > L - 1) last = L - 1;
    for (int h = 0; h < H; ++h)
      for (int d = 0; d < D; ++d)
        q[h * D + d] = or_load(q_idx, dtype, ((int64_t)r * H + h) * D + d);
    for (int64_t p = 0; p < ld; ++p) {
      float* out = &scores[(int64_t)r * ld + p];
      if (p > last) { *out = -INFINITY; continue; }
      int64_t row = or_phys_row(block_table, max_blocks, bs, num_blocks, b, p);
      if (row < 0) { *out = -INFINITY; rc = OR_ERR_LAYOUT; continue; }
      for (int d = 0; d < D; ++d) k[d] = or_load(kidx_pool, dtype, row * D + d);
      double s = 0.0;
      for (int h = 0; h < H; ++h) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += q[h * D + d] * k[d];
        if (dot > 0.0) s += (double)w[(int64_t)r * H + h] * dot;
      }
      *out = (float)s;
    }
  }
  free(q);
  free(k);
  return rc;
}

/* ---- stage 2: top-K [P1 §3 (1); P3 §4 "Determinism of index selection"] --
 * For each query row, among its first n_elig[r] positions, keep the K with the
 * largest score; equal scores are ordered by position, the lower position
 * winning (a fixed, reproducible tie rule).  Scores are compared as values,
 * so -0.0 and +0.0 tie.  The kept positions are written in ascending order
 * and the row is padded with -1 when fewer than K positions are eligible.
 * This is the plain definition: a full sort of (score desc, position asc). */
typedef struct {
  float s;
  int32_t p;
} or_cand;

static int or_cmp_cand(const void* a, const void* b) {
  const or_cand* x = (const or_cand*)a;
  const or_cand* y = (const or_cand*)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->p > y->p) - (x->p < y->p);
}

static int or_cmp_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

int oracle_topk(const float* scores, int64_t ld, const int32_t* n_elig, int Nq,
                int K, int32_t* idx) {
  if (K <= 0 || Nq < 0) return OR_ERR_ARG;
  or_cand* c = NULL;
  int64_t cap = 0;
  for (int r = 0; r < Nq; ++r) {
    int64_t n = n_elig[r];
    if (n < 0) n = 0;
    if (n > ld) { free(c); return OR_ERR_ARG; }
    if (n > cap) {
      free(c);
      cap = n;
      c = (or_cand*)malloc(sizeof(or_cand) * (size_t)cap);
      if (!c) return OR_ERR_ARG;
    }
    for (int64_t p = 0; p < n; ++p) {
      float s = scores[(int64_t)r * ld + p];
      if (isnan(s)) { free(c); return OR_ERR_NAN; }
      c[p].s = s;
      c[p].p = (int32_t)p;
    }
    qsort(c, (size_t)n, sizeof(or_cand), or_cmp_cand);
    int64_t m = n < K ? n : K;
    int32_t* out = &idx[(int64_t)r * K];
    for (int64_t j = 0; j < m; ++j) out[j] = c[j].p;
    qsort(out, (size_t)m, sizeof(int32_t), or_cmp_i32);
    for (int64_t j = m; j < K; ++j) out[j] = -1;
  }
  free(c);
  return OR_OK;
}

/* ---- stage 3: exact softmax attention over the selected rows -------------
 * [P1 §3 (3); P2 §3.1 item 3; P3 §4 execution chain, the step that gathers
 * the cached rows and attends over them].  For query r (of sequence q_seq[r]) and head h, over the
 * selected positions j (idx entries >= 0) whose rows are gathered through the
 * block table:
 *     z_j = sm_scale * sum_d q[r,h,d] * K[j,d]
 *     out[r,h,:] = sum_j exp(z_j - m) V[j,:] / sum_j exp(z_j - m),  m = max z
 *     lse[r,h]   = m + log(sum_j exp(z_j - m))
 * Two passes (max, then sums), all in double.  With no selected position the
 * output is 0 and lse is -inf.  q: [Nq][Hq][Dqk] bf16; K rows at
 * k_pool + row*k_row_stride (Dqk bf16 each); V rows at v_pool +
 * row*v_row_stride (Dv bf16 each); idx: [Nq][K]; out: [Nq][Hq][Dv];
 * lse: [Nq][Hq] (may be NULL). */
int oracle_sparse_attn(int batch, int bs, int num_blocks, int max_blocks,
                       const int32_t* block_table, const int32_t* seq_lens,
                       int Nq, const int32_t* q_seq, int Hq, int Dqk, int Dv,
                       const uint16_t* q, const uint16_t* k_pool,
                       int64_t k_row_stride, const uint16_t* v_pool,
                       int64_t v_row_stride, const int32_t* idx, int K,
                       double sm_scale, double* out, double* lse) {
  if (batch <= 0 || bs <= 0 || Nq < 0 || Hq <= 0 || Dqk <= 0 || Dv <= 0 ||
      K <= 0)
    return OR_ERR_ARG;
  int rc = OR_OK;
  /* the selected rows, decoded once: kk [K][Dqk], vv [K][Dv] */
  double* kk = (double*)malloc(sizeof(double) * (size_t)K * Dqk);
  double* vv = (double*)malloc(sizeof(double) * (size_t)K * Dv);
  double* z = (double*)malloc(sizeof(double) * (size_t)K);
  double* qh = (double*)malloc(sizeof(double) * (size_t)Dqk);
  if (!kk || !vv || !z || !qh) { free(kk); free(vv); free(z); free(qh); return OR_ERR_ARG; }
  for (int r = 0; r < Nq; ++r) {
    int b = q_seq[r];
    if (b < 0 || b >= batch) { rc = OR_ERR_ARG; break; }
    int n = 0;
    for (int j = 0; j < K; ++j) {
      int32_t p = idx[(int64_t)r * K + j];
      if (p < 0) continue;
      if (p >= seq_lens[b]) { rc = OR_ERR_LAYOUT; continue; }
      int64_t row = or_phys_row(block_table, max_blocks, bs, num_blocks, b, p);
      if (row < 0) { rc = OR_ERR_LAYOUT; continue; }
      for (int d = 0; d < Dqk; ++d) kk[(int64_t)n * Dqk + d] = or_dec_bf16(k_pool[row * k_row_stride + d]);
      for (int d = 0; d < Dv; ++d) vv[(int64_t)n * Dv + d] = or_dec_bf16(v_pool[row * v_row_stride + d]);
      ++n;
    }
    for (int h = 0; h < Hq; ++h) {
      double* o = &out[((int64_t)r * Hq + h) * Dv];
      for (int d = 0; d < Dqk; ++d)
        qh[d] = or_dec_bf16(q[((int64_t)r * Hq + h) * Dqk + d]);
      for (int d = 0; d < Dv; ++d) o[d] = 0.0;
      if (n == 0) {
        if (lse) lse[(int64_t)r * Hq + h] = -INFINITY;
        continue;
      }
      double m = -INFINITY;
      for (int j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int d = 0; d < Dqk; ++d) dot += qh[d] * kk[(int64_t)j * Dqk + d];
        z[j] = sm_scale * dot;
        if (z[j] > m) m = z[j];
      }
      double l = 0.0;
      for (int j = 0; j < n; ++j) {
        double e = exp(z[j] - m);
        l += e;
        for (int d = 0; d < Dv; ++d) o[d] += e * vv[(int64_t)j * Dv + d];
      }
      for (int d = 0; d < Dv; ++d) o[d] /= l;
      if (lse) lse[(int64_t)r * Hq + h] = m + log(l);
    }
  }
  free(kk);
  free(vv);
  free(z);
  free(qh);
  return rc;
}
