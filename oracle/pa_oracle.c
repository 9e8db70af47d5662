/*
 * CPU oracle for paged-attention decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the package smoke check and the bench's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library; the two meet only in the seeded inputs of workloads.py.
 *
 * What it computes.  The pages study paged-attention decode: new query tokens
 * attend over a KV cache that is stored in fixed-size physical pages and read
 * page by page through a per-sequence block table ("HSTU Paged Attention",
 * RecSDK issue 1281, background section; "Benchmark high-perf Paged
 * Attention", simpler issue 998, shape table b1_h16_kv1_s128_bs128_hd128).
 * The pages never print the attention formula, so this file writes out the
 * plain definition of scaled dot-product softmax attention, one query row at
 * a time:
 *
 *   g    = h / (Hq / Hkv)                       query head h reads KV head g
 *   L    = n - q_len + i + 1 if causal else n   keys 0..L-1 are visible
 *   k_j  = K[table[b][j / bs], j % bs, g, :]    (the same for v_j)
 *   s_j  = sm_scale * sum_d q[d] * k_j[d]
 *   m    = max_j s_j,  e_j = exp(s_j - m)
 *   out  = sum_j e_j v_j / sum_j e_j,  lse = m + log(sum_j e_j)
 *
 * Rows i >= q_len are padding: out = 0 and lse = -inf.  The LSE merge used
 * for split invariance is  m* = max_s lse_s, w_s = exp(lse_s - m*),
 * out = sum_s w_s o_s / sum_s w_s, lse = m* + log(sum_s w_s); a split with
 * lse = -inf has weight 0.  Work is split into per-range partials merged this
 * way in the split-KV decode of "Optimize paged-attention metadata decode"
 * (FlyDSL PR #910, Summary: persistent decode plus split reducer).
 *
 * Inputs are the stored bytes the GPU reads.  bf16 and fp16 are widened
 * exactly; an fp8 cache holds OCP E4M3 codes (bias 7, subnormals, no
 * infinities, S.1111.111 = NaN, max 448) that are decoded here bit by bit and
 * multiplied by their scale: one fp32 scalar per tensor, or one fp32 per
 * (block, slot, kv-head) row (FlyDSL PR #910, per_token_kv scale mode).
 *
 * Precision.  The pages' correctness check is against a CPU FP32 reference
 * (RecSDK issue 1281, correctness section).  This one source is compiled
 * twice: with ORACLE_F32 every sum, exp and log is in float (that reference),
 * and without it in double (used to pin the float build).  Softmax is the
 * two-pass form above; there is no blocking, fusion or reordering beyond it.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef ORACLE_F32
typedef float real;
#define R_EXP expf
#define R_LOG logf
#else
typedef double real;
#define R_EXP exp
#define R_LOG log
#endif

enum { OR_BF16 = 0, OR_FP16 = 1, OR_E4M3 = 2 };
enum { OR_SCALE_NONE = 0, OR_SCALE_TENSOR = 1, OR_SCALE_TOKEN = 2 };

typedef struct {
  int32_t batch, max_q_len, num_q_heads, num_kv_heads, head_dim, block_size;
  int32_t max_blocks_per_seq, num_blocks;
  int32_t q_dtype, kv_dtype, scale_mode, causal;
  double sm_scale;
} oracle_cfg;

/* Size of the real type, so the caller can check which build it loaded. */
int oracle_real_bytes(void) { return (int)sizeof(real); }

/* bf16 is the upper half of an IEEE binary32. */
real oracle_bf16(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (real)f;
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits. */
real oracle_fp16(uint16_t bits) {
  int sign = bits >> 15, e = (bits >> 10) & 0x1f, m = bits & 0x3ff;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24);
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + m), e - 25);
  return (real)(sign ? -v : v);
}

/* OCP FP8 E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent and
 * mantissa all ones is NaN; there is no infinity. */
real oracle_e4m3(uint8_t code) {
  int sign = code >> 7, e = (code >> 3) & 0xf, m = code & 0x7;
  double v;
  if (e == 15 && m == 7)
    v = NAN;
  else if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp((double)(8 + m), e - 10);
  return (real)(sign ? -v : v);
}

static real element(int dtype, const void *base, size_t idx) {
  switch (dtype) {
    case OR_BF16: return oracle_bf16(((const uint16_t *)base)[idx]);
    case OR_FP16: return oracle_fp16(((const uint16_t *)base)[idx]);
    default: return oracle_e4m3(((const uint8_t *)base)[idx]);
  }
}

typedef struct {
  const oracle_cfg *c;
  const void *q, *k, *v;
  const float *k_scale, *v_scale;
  const int32_t *block_tables, *context_lens, *q_lens;
} problem;

/* Scale of the (page, slot, kv-head) row of K (is_v = 0) or V (is_v = 1). */
static real row_scale(const problem *p, int is_v, int page, int slot, int g) {
  const float *s = is_v ? p->v_scale : p->k_scale;
  const oracle_cfg *c = p->c;
  if (c->scale_mode == OR_SCALE_TENSOR) return (real)s[0];
  if (c->scale_mode == OR_SCALE_TOKEN)
    return (real)s[((size_t)page * c->block_size + slot) * c->num_kv_heads + g];
  return 1;
}

/* Number of keys query row i of sequence b may see (0 for a padding row). */
static int visible_keys(const problem *p, int b, int i) {
  int n = p->context_lens[b], ql = p->q_lens[b];
  if (i >= ql) return 0;
  return p->c->causal ? n - ql + i + 1 : n;
}

/* Softmax attention of query row (b, i, h) over keys [j0, j1), the two-pass form.
 * Writes D values to o and the log-sum-exp to *lse; an empty range gives 0 and -inf.
 * Returns -1 if a page index is outside the pool. */
static int attend_range(const problem *p, int b, int i, int h, int j0, int j1, real *o,
                        real *lse) {
  const oracle_cfg *c = p->c;
  int D = c->head_dim, bs = c->block_size, G = c->num_q_heads / c->num_kv_heads;
  int g = h / G;
  for (int d = 0; d < D; ++d) o[d] = 0;
  *lse = -INFINITY;
  if (j1 <= j0) return 0;
  int nk = j1 - j0;
  real *s = (real *)malloc(sizeof(real) * (size_t)nk);
  real *qrow = (real *)malloc(sizeof(real) * (size_t)D);
  if (!s || !qrow) { free(s); free(qrow); return -2; }
  size_t qoff = (((size_t)b * c->max_q_len + i) * c->num_q_heads + h) * (size_t)D;
  for (int d = 0; d < D; ++d) qrow[d] = element(c->q_dtype, p->q, qoff + d);

  /* pass 1: scores and their maximum */
  real m = -INFINITY;
  for (int j = j0; j < j1; ++j) {
    int page = p->block_tables[(size_t)b * c->max_blocks_per_seq + j / bs];
    int slot = j % bs;
    if (page < 0 || page >= c->num_blocks) { free(s); free(qrow); return -1; }
    size_t koff = (((size_t)page * bs + slot) * c->num_kv_heads + g) * (size_t)D;
    real ks = row_scale(p, 0, page, slot, g);
    real dot = 0;
    for (int d = 0; d < D; ++d) dot += qrow[d] * (element(c->kv_dtype, p->k, koff + d) * ks);
    s[j - j0] = (real)c->sm_scale * dot;
    if (s[j - j0] > m) m = s[j - j0];
  }
  /* pass 2: exponentials, their sum and the weighted sum of values */
  real den = 0;
  for (int j = j0; j < j1; ++j) {
    int page = p->block_tables[(size_t)b * c->max_blocks_per_seq + j / bs];
    int slot = j % bs;
    size_t voff = (((size_t)page * bs + slot) * c->num_kv_heads + g) * (size_t)D;
    real vs = row_scale(p, 1, page, slot, g);
    real e = R_EXP(s[j - j0] - m);
    den += e;
    for (int d = 0; d < D; ++d) o[d] += e * (element(c->kv_dtype, p->v, voff + d) * vs);
  }
  for (int d = 0; d < D; ++d) o[d] /= den;
  *lse = m + R_LOG(den);
  free(s);
  free(qrow);
  return 0;
}

/* LSE merge of n partial results (o_s: n rows of D, lse_s: n values). */
void oracle_merge(int n, int D, const real *o_s, const real *lse_s, real *o, real *lse) {
  real mx = -INFINITY;
  for (int s = 0; s < n; ++s)
    if (lse_s[s] > mx) mx = lse_s[s];
  for (int d = 0; d < D; ++d) o[d] = 0;
  if (mx == -INFINITY) { *lse = -INFINITY; return; }
  real wsum = 0;
  for (int s = 0; s < n; ++s) {
    real w = (lse_s[s] == -INFINITY) ? 0 : R_EXP(lse_s[s] - mx);
    wsum += w;
    for (int d = 0; d < D; ++d) o[d] += w * o_s[(size_t)s * D + d];
  }
  for (int d = 0; d < D; ++d) o[d] /= wsum;
  *lse = mx + R_LOG(wsum);
}

/* One query row: the whole visible range at once (nsplit <= 1), or nsplit
 * contiguous ranges of ceil(L / nsplit) keys each, merged by oracle_merge. */
static int one_row(const problem *p, int b, int i, int h, int nsplit, real *o, real *lse) {
  int D = p->c->head_dim;
  int L = visible_keys(p, b, i);
  if (nsplit <= 1) return attend_range(p, b, i, h, 0, L, o, lse);
  real *os = (real *)malloc(sizeof(real) * (size_t)nsplit * D);
  real *ls = (real *)malloc(sizeof(real) * (size_t)nsplit);
  if (!os || !ls) { free(os); free(ls); return -2; }
  int chunk = (L + nsplit - 1) / nsplit;
  int rc = 0;
  for (int s = 0; s < nsplit && rc == 0; ++s) {
    int j0 = s * chunk, j1 = (s + 1) * chunk;
    if (j0 > L) j0 = L;
    if (j1 > L) j1 = L;
    rc = attend_range(p, b, i, h, j0, j1, os + (size_t)s * D, ls + s);
  }
  if (rc == 0) oracle_merge(nsplit, D, os, ls, o, lse);
  free(os);
  free(ls);
  return rc;
}

static int check_lengths(const oracle_cfg *c, const int32_t *context_lens,
                         const int32_t *q_lens) {
  for (int b = 0; b < c->batch; ++b) {
    if (q_lens[b] < 0 || q_lens[b] > c->max_q_len) return -3;
    if (context_lens[b] < q_lens[b]) return -3;
    if (context_lens[b] > c->max_blocks_per_seq * c->block_size) return -3;
  }
  return 0;
}

/* Every output row: out[B, Sq, Hq, D], lse[B, Sq, Hq].  Returns 0, or a negative
 * code for an invalid problem (-1 page outside the pool, -3 bad lengths). */
int oracle_decode(const oracle_cfg *c, const void *q, const void *k, const void *v,
                  const float *k_scale, const float *v_scale, const int32_t *block_tables,
                  const int32_t *context_lens, const int32_t *q_lens, int nsplit, real *out,
                  real *lse) {
  problem p = {c, q, k, v, k_scale, v_scale, block_tables, context_lens, q_lens};
  int rc = check_lengths(c, context_lens, q_lens);
  if (rc) return rc;
  long rows = (long)c->batch * c->max_q_len * c->num_q_heads;
  int fail = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : fail)
  for (long r = 0; r < rows; ++r) {
    int h = (int)(r % c->num_q_heads);
    int i = (int)((r / c->num_q_heads) % c->max_q_len);
    int b = (int)(r / ((long)c->num_q_heads * c->max_q_len));
    if (one_row(&p, b, i, h, nsplit, out + (size_t)r * c->head_dim, lse + r) != 0) fail = 1;
  }
  return fail ? -1 : 0;
}

/* A chosen subset of rows: rows_bih holds n triples (b, i, h); row t of out/lse
 * receives that row's result. */
int oracle_decode_rows(const oracle_cfg *c, const void *q, const void *k, const void *v,
                       const float *k_scale, const float *v_scale,
                       const int32_t *block_tables, const int32_t *context_lens,
                       const int32_t *q_lens, int n, const int32_t *rows_bih, real *out,
                       real *lse) {
  problem p = {c, q, k, v, k_scale, v_scale, block_tables, context_lens, q_lens};
  int rc = check_lengths(c, context_lens, q_lens);
  if (rc) return rc;
  int fail = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : fail)
  for (int t = 0; t < n; ++t) {
    if (one_row(&p, rows_bih[3 * t], rows_bih[3 * t + 1], rows_bih[3 * t + 2], 0,
                out + (size_t)t * c->head_dim, lse + t) != 0)
      fail = 1;
  }
  return fail ? -1 : 0;
}

/* Attention of row (b, i, h) over an explicit key range [j0, j1) of its visible
 * keys (the range is clipped to them): the partial result one split produces. */
int oracle_attend_range(const oracle_cfg *c, const void *q, const void *k, const void *v,
                        const float *k_scale, const float *v_scale,
                        const int32_t *block_tables, const int32_t *context_lens,
                        const int32_t *q_lens, int b, int i, int h, int j0, int j1, real *o,
                        real *lse) {
  problem p = {c, q, k, v, k_scale, v_scale, block_tables, context_lens, q_lens};
  int L = visible_keys(&p, b, i);
  if (j1 > L) j1 = L;
  if (j0 > j1) j0 = j1;
  return attend_range(&p, b, i, h, j0, j1, o, lse);
}

/* ------------------------------------------------------------------------------------
 * KV append with quantise-on-write: the step that fills the paged cache the decode reads.
 *
 * A decode step's q_len new tokens of sequence b are the last q_len positions of its
 * context_len cached tokens (the convention of the decode above), so new row i of
 * sequence b is stored at position pos = context_len - q_len + i, which is slot pos % bs
 * of physical block block_tables[b][pos / bs] ("HSTU Paged Attention", RecSDK issue 1281,
 * background: K/V live in a paged cache read through per-sequence page lists).  A 16-bit
 * cache receives the new row's bits unchanged.  An fp8 cache receives E4M3 codes of the
 * row divided by its scale, one of the scale modes of "Optimize paged-attention metadata
 * decode" (FlyDSL PR #910, Breaking Changes: per_token_kv): per-token, the scale of the
 * (block, slot, kv-head) row is its largest magnitude over 448 (the E4M3 maximum), or 1
 * for an all-zero row, and is written next to the codes; per-tensor, the one scale the
 * caller holds is used as it is; with no scale the values are encoded directly.
 *
 * The scale and the quotient are float (binary32) operations, as the scales are stored
 * in float; the code is the E4M3 value nearest to the quotient clamped to [-448, 448],
 * ties to the even code.  These are float in both builds of this file, so a code is the
 * same integer decision whatever `real` is.
 * ------------------------------------------------------------------------------------ */

/* Round-half-to-even of t >= 0 to an integer (kept in a double). */
static double round_half_even(double t) {
  double fl = floor(t), fr = t - fl;
  if (fr > 0.5 || (fr == 0.5 && fmod(fl, 2.0) == 1.0)) fl += 1.0;
  return fl;
}

/* OCP E4M3 code of x: magnitude clamped to 448, rounded to the nearest point of the E4M3
 * grid (ties to even), NaN to 0x7f.  In the binade [2^e, 2^(e+1)), e >= -6, the grid
 * spacing is 2^(e-3); below 2^-6 (subnormals) it is 2^-9. */
uint8_t oracle_e4m3_encode(float x) {
  if (isnan(x)) return 0x7f;
  int sign = signbit(x) ? 1 : 0;
  double a = fabs((double)x);
  if (a > 448.0) a = 448.0;
  int e = -6;
  if (a >= ldexp(1.0, -6)) {
    (void)frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;             /* a in [2^e, 2^(e+1)) */
  }
  double step = ldexp(1.0, e - 3);
  double v = round_half_even(a / step) * step; /* a / step is exact: step is a power of 2 */
  int efield = 0, mant = 0;
  if (v >= ldexp(1.0, -6)) {
    int ev;
    double f = frexp(v, &ev); /* v = f * 2^ev = (2f) * 2^(ev-1) */
    efield = ev - 1 + 7;
    mant = (int)((2.0 * f - 1.0) * 8.0);
  } else {
    mant = (int)(v / ldexp(1.0, -9));
  }
  return (uint8_t)((sign << 7) | (efield << 3) | mant);
}

/* Append every sequence's q_lens[b] new rows of k_new / v_new ([B, max_q_len, Hkv, D] in
 * q_dtype) into k_cache / v_cache ([num_blocks, block_size, Hkv, D] in kv_dtype), and for
 * per-token fp8 their scales into k_scale / v_scale ([num_blocks, block_size, Hkv]).  For
 * per-tensor fp8, k_scale[0] / v_scale[0] are read.  Nothing is written when a length or a
 * block id in use is invalid: returns -3 (lengths) or -1 (block id), 0 otherwise. */
int oracle_append_kv(const oracle_cfg *c, const void *k_new, const void *v_new,
                     const int32_t *block_tables, const int32_t *context_lens,
                     const int32_t *q_lens, void *k_cache, void *v_cache, float *k_scale,
                     float *v_scale) {
  int rc = check_lengths(c, context_lens, q_lens);
  if (rc) return rc;
  int bs = c->block_size, D = c->head_dim, H = c->num_kv_heads;
  for (int b = 0; b < c->batch; ++b) {
    int n = context_lens[b], ql = q_lens[b];
    for (int i = 0; i < ql; ++i) {
      int pos = n - ql + i;
      int page = block_tables[(size_t)b * c->max_blocks_per_seq + pos / bs];
      if (page < 0 || page >= c->num_blocks) return -1;
    }
  }
  float *x = (float *)malloc(sizeof(float) * (size_t)D);
  if (!x) return -2;
  for (int b = 0; b < c->batch; ++b) {
    int n = context_lens[b], ql = q_lens[b];
    for (int i = 0; i < ql; ++i) {
      int pos = n - ql + i;
      int page = block_tables[(size_t)b * c->max_blocks_per_seq + pos / bs];
      int slot = pos % bs;
      for (int g = 0; g < H; ++g) {
        size_t src = (((size_t)b * c->max_q_len + i) * H + g) * (size_t)D;
        size_t row = ((size_t)page * bs + slot) * H + g;
        for (int t = 0; t < 2; ++t) { /* K, then V */
          const void *nw = t ? v_new : k_new;
          void *cache = t ? v_cache : k_cache;
          float *scales = t ? v_scale : k_scale;
          if (c->kv_dtype != OR_E4M3) {
            memcpy((uint16_t *)cache + row * D, (const uint16_t *)nw + src, sizeof(uint16_t) * D);
            continue;
          }
          for (int d = 0; d < D; ++d) x[d] = (float)element(c->q_dtype, nw, src + d);
          float s = 1.0f;
          if (c->scale_mode == OR_SCALE_TOKEN) {
            float amax = 0.0f;
            for (int d = 0; d < D; ++d)
              if (fabsf(x[d]) > amax) amax = fabsf(x[d]);
            s = amax > 0.0f ? amax / 448.0f : 1.0f;
            scales[row] = s;
          } else if (c->scale_mode == OR_SCALE_TENSOR) {
            s = scales[0];
          }
          uint8_t *codes = (uint8_t *)cache + row * D;
          for (int d = 0; d < D; ++d) codes[d] = oracle_e4m3_encode(x[d] / s);
        }
      }
    }
  }
  free(x);
  return 0;
}
