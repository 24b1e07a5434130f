/*
 * CPU oracle for paged multi-token attention and the paged KV append.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What it computes (plainest reading of "Stateful Large Language Model
 * Serving with Pensieve", abstract: the PagedAttention kernel generalised to
 * attention between multiple input tokens, with the GPU cache spread over
 * non-contiguous memory; and of the PagedAttention description in the
 * "LLM上下文缓存与状态复用机制的分析和探索" blog, section 3.1: the KV cache is cut
 * into fixed-size blocks that may sit anywhere in physical memory):
 *
 *   For request r, query token t at absolute position p_t and query head h,
 *   with KV head g = h / G (G = Hq / Hkv):
 *     Kc[j] = Kpool[bt[r][j / B]][g][j % B][:]           (gather, j in [0, ctx_r))
 *     s_j   = scale * sum_d q[t][h][d] * Kc[j][d]        for every j <= p_t
 *     m     = max_j s_j ;  l = sum_j exp(s_j - m)
 *     O[t][h][:] = sum_j exp(s_j - m) * Vc[j][:] / l
 *     LSE[t][h]  = m + ln(l)                               (natural log)
 *   Keys with j > p_t are not part of the sum at all.
 *
 *   Append: for token t of request r at position p, for every KV head g,
 *     Kpool[bt[r][p / B]][g][p % B][:] = Knew[t][g][:]  (bit copy), same for V.
 *
 *   Swap: copy whole physical blocks (all KV heads, K then V) between the
 *   pool and a host buffer laid out [n][2][Hkv][B][D].
 *
 * Arithmetic is fp64 throughout; bf16 inputs are widened exactly.
 * Pool layout: [num_blocks][num_kv_heads][block_size][head_dim], bf16 bits.
 *
 * FP8 KV cache (the "_fp8" entry points): the pools hold OCP FP8 E4M3 codes
 * (sign, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 is
 * subnormal; S.1111.111 is NaN; no infinities; largest finite 448).  A code
 * stands for e4m3(c) * scale with one scale per pool for K and one for V.
 * Append quantises a bf16 element x to the code nearest to the fp32 quotient
 * x / scale, ties to the even code, finite values beyond 448 saturating to
 * +-448 and NaN to NaN.  Attention then runs on the dequantised values.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1

static double bf16_to_f64(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Value of an E4M3 code, from the format's definition. */
double oracle_e4m3_decode(uint8_t c) {
  int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m / 8.0, -6);          /* subnormal: 0.m * 2^(1-7) */
  else v = ldexp(1.0 + (double)m / 8.0, e - 7);         /* normal: 1.m * 2^(e-7) */
  return sign ? -v : v;
}

/* Nearest E4M3 code to the float x (ties to the even code, i.e. the one with
 * an even mantissa), finite values beyond the largest code saturating. */
uint8_t oracle_e4m3_encode(float x) {
  if (isnan(x)) return 0x7F;
  uint8_t sign = signbit(x) ? 0x80 : 0;
  double a = fabs((double)x);
  if (a >= 448.0) return sign | 0x7E;                  /* 448 = 1.75 * 2^8, code 0.1111.110 */
  if (a < ldexp(1.0, -6)) {
    /* subnormal range: multiples of 2^-9; 8 * 2^-9 = 2^-6 is the smallest normal, code 8 */
    double n = rint(ldexp(a, 9));                       /* round half to even (default mode) */
    return sign | (uint8_t)n;
  }
  int k;
  double f = frexp(a, &k);                              /* a = f * 2^k, f in [0.5, 1) */
  int E = k - 1;                                        /* a = (2f) * 2^E, 2f in [1, 2) */
  double mm = rint((2.0 * f - 1.0) * 8.0);              /* mantissa steps of 1/8, ties to even */
  if (mm == 8.0) { mm = 0.0; E += 1; }
  /* a < 448 keeps the result at or below 1.75 * 2^8 */
  return sign | (uint8_t)(((E + 7) << 3) | (int)mm);
}

/* Request owning token t: the r with cu_q_lens[r] <= t < cu_q_lens[r+1]. */
static int owner_of(const int32_t* cu_q_lens, int num_reqs, int t) {
  for (int r = 0; r < num_reqs; ++r)
    if (t >= cu_q_lens[r] && t < cu_q_lens[r + 1]) return r;
  return -1;
}

/* Element idx of a pool: a bf16 value, or an E4M3 code times the pool's scale. */
static double pool_value(const void* pool, size_t idx, int fp8, double scale) {
  if (fp8) return oracle_e4m3_decode(((const uint8_t*)pool)[idx]) * scale;
  return bf16_to_f64(((const uint16_t*)pool)[idx]);
}

/* One output row (token t, query head h).  Returns 0 or ORACLE_EINVAL. */
static int attn_row(const uint16_t* q, const void* k_pool, const void* v_pool, int fp8, double k_scale, double v_scale,
                    int num_blocks, int hkv, int bs, int d, int hq,
                    const int32_t* bt, int max_blocks, const int32_t* ctx_lens,
                    const int32_t* cu_q_lens, const int32_t* q_pos, int num_reqs,
                    double scale, int t, int h, double* out, double* lse) {
  int r = owner_of(cu_q_lens, num_reqs, t);
  if (r < 0) return ORACLE_EINVAL;
  int group = hq / hkv;
  int g = h / group;
  int p = q_pos[t];
  int ctx = ctx_lens[r];
  if (p < 0 || p >= ctx) return ORACLE_EINVAL;
  int nvis = p + 1;                      /* keys 0..p are visible */
  double* kc = (double*)malloc(sizeof(double) * (size_t)nvis * d);
  double* vc = (double*)malloc(sizeof(double) * (size_t)nvis * d);
  double* s = (double*)malloc(sizeof(double) * (size_t)nvis);
  if (!kc || !vc || !s) { free(kc); free(vc); free(s); return ORACLE_EINVAL; }
  /* gather: logical key j lives in physical block bt[r][j / bs], slot j % bs */
  for (int j = 0; j < nvis; ++j) {
    int lb = j / bs;
    if (lb >= max_blocks) { free(kc); free(vc); free(s); return ORACLE_EINVAL; }
    int pb = bt[(size_t)r * max_blocks + lb];
    if (pb < 0 || pb >= num_blocks) { free(kc); free(vc); free(s); return ORACLE_EINVAL; }
    size_t base = (((size_t)pb * hkv + g) * bs + (j % bs)) * (size_t)d;
    for (int e = 0; e < d; ++e) {
      kc[(size_t)j * d + e] = pool_value(k_pool, base + e, fp8, k_scale);
      vc[(size_t)j * d + e] = pool_value(v_pool, base + e, fp8, v_scale);
    }
  }
  const uint16_t* qrow = q + ((size_t)t * hq + h) * d;
  double m = -INFINITY;
  for (int j = 0; j < nvis; ++j) {
    double acc = 0.0;
    for (int e = 0; e < d; ++e) acc += bf16_to_f64(qrow[e]) * kc[(size_t)j * d + e];
    s[j] = scale * acc;
    if (s[j] > m) m = s[j];
  }
  double l = 0.0;
  for (int e = 0; e < d; ++e) out[e] = 0.0;
  for (int j = 0; j < nvis; ++j) {
    double w = exp(s[j] - m);
    l += w;
    for (int e = 0; e < d; ++e) out[e] += w * vc[(size_t)j * d + e];
  }
  for (int e = 0; e < d; ++e) out[e] /= l;
  *lse = m + log(l);
  free(kc); free(vc); free(s);
  return ORACLE_OK;
}

/*
 * Attention for a list of (token, query head) rows.
 *   q [T][hq][d], pools [num_blocks][hkv][bs][d] (bf16 bits)
 *   bt [num_reqs][max_blocks], ctx_lens [num_reqs], cu_q_lens [num_reqs+1], q_pos [T]
 *   rows_t / rows_h [n_rows]; out [n_rows][d] fp64, lse [n_rows] fp64.
 * Returns 0, or ORACLE_EINVAL if any row violates a precondition.
 */
static int attn_rows(const uint16_t* q, const void* k_pool, const void* v_pool, int fp8, double k_scale,
                     double v_scale, int num_blocks, int num_kv_heads, int block_size, int head_dim,
                     int num_q_heads, const int32_t* block_tables, int max_blocks,
                     const int32_t* ctx_lens, const int32_t* cu_q_lens,
                     const int32_t* q_positions, int num_reqs, double scale,
                     const int32_t* rows_t, const int32_t* rows_h, int n_rows,
                     double* out, double* lse) {
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || block_size <= 0 || head_dim <= 0)
    return ORACLE_EINVAL;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int i = 0; i < n_rows; ++i) {
    int rc = attn_row(q, k_pool, v_pool, fp8, k_scale, v_scale, num_blocks, num_kv_heads, block_size, head_dim,
                      num_q_heads, block_tables, max_blocks, ctx_lens, cu_q_lens, q_positions,
                      num_reqs, scale, rows_t[i], rows_h[i], out + (size_t)i * head_dim, lse + i);
    if (rc) bad |= 1;
  }
  return bad ? ORACLE_EINVAL : ORACLE_OK;
}

int oracle_paged_attn_rows(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                           int num_blocks, int num_kv_heads, int block_size, int head_dim,
                           int num_q_heads, const int32_t* block_tables, int max_blocks,
                           const int32_t* ctx_lens, const int32_t* cu_q_lens,
                           const int32_t* q_positions, int num_reqs, double scale,
                           const int32_t* rows_t, const int32_t* rows_h, int n_rows,
                           double* out, double* lse) {
  return attn_rows(q, k_pool, v_pool, 0, 1.0, 1.0, num_blocks, num_kv_heads, block_size, head_dim,
                   num_q_heads, block_tables, max_blocks, ctx_lens, cu_q_lens, q_positions, num_reqs,
                   scale, rows_t, rows_h, n_rows, out, lse);
}

/* The same rows over FP8 pools (E4M3 codes) with dequantisation scales. */
int oracle_paged_attn_rows_fp8(const uint16_t* q, const uint8_t* k_pool, const uint8_t* v_pool,
                               double k_scale, double v_scale,
                               int num_blocks, int num_kv_heads, int block_size, int head_dim,
                               int num_q_heads, const int32_t* block_tables, int max_blocks,
                               const int32_t* ctx_lens, const int32_t* cu_q_lens,
                               const int32_t* q_positions, int num_reqs, double scale,
                               const int32_t* rows_t, const int32_t* rows_h, int n_rows,
                               double* out, double* lse) {
  return attn_rows(q, k_pool, v_pool, 1, k_scale, v_scale, num_blocks, num_kv_heads, block_size,
                   head_dim, num_q_heads, block_tables, max_blocks, ctx_lens, cu_q_lens, q_positions,
                   num_reqs, scale, rows_t, rows_h, n_rows, out, lse);
}

/* Attention for every row: out [T][hq][d], lse [T][hq]. */
int oracle_paged_attn(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                      int num_blocks, int num_kv_heads, int block_size, int head_dim,
                      int num_q_heads, const int32_t* block_tables, int max_blocks,
                      const int32_t* ctx_lens, const int32_t* cu_q_lens,
                      const int32_t* q_positions, int num_reqs, int num_tokens, double scale,
                      double* out, double* lse) {
  size_t n = (size_t)num_tokens * num_q_heads;
  int32_t* rt = (int32_t*)malloc(sizeof(int32_t) * (n ? n : 1));
  int32_t* rh = (int32_t*)malloc(sizeof(int32_t) * (n ? n : 1));
  if (!rt || !rh) { free(rt); free(rh); return ORACLE_EINVAL; }
  for (int t = 0; t < num_tokens; ++t)
    for (int h = 0; h < num_q_heads; ++h) {
      rt[(size_t)t * num_q_heads + h] = t;
      rh[(size_t)t * num_q_heads + h] = h;
    }
  int rc = oracle_paged_attn_rows(q, k_pool, v_pool, num_blocks, num_kv_heads, block_size,
                                  head_dim, num_q_heads, block_tables, max_blocks, ctx_lens,
                                  cu_q_lens, q_positions, num_reqs, scale, rt, rh, (int)n, out, lse);
  free(rt); free(rh);
  return rc;
}

/*
 * Append: scatter k_new / v_new [T][hkv][d] into the pools at each token's slot.
 * Every token is checked before anything is written; returns ORACLE_EINVAL and
 * writes nothing if any slot is out of range.
 */
int oracle_append(uint16_t* k_pool, uint16_t* v_pool, int num_blocks, int num_kv_heads,
                  int block_size, int head_dim, const int32_t* block_tables, int max_blocks,
                  const int32_t* cu_q_lens, const int32_t* positions, int num_reqs,
                  int num_tokens, const uint16_t* k_new, const uint16_t* v_new) {
  for (int t = 0; t < num_tokens; ++t) {
    int r = owner_of(cu_q_lens, num_reqs, t);
    if (r < 0) return ORACLE_EINVAL;
    int p = positions[t];
    if (p < 0 || p / block_size >= max_blocks) return ORACLE_EINVAL;
    int pb = block_tables[(size_t)r * max_blocks + p / block_size];
    if (pb < 0 || pb >= num_blocks) return ORACLE_EINVAL;
  }
  size_t row = (size_t)head_dim * sizeof(uint16_t);
  for (int t = 0; t < num_tokens; ++t) {
    int r = owner_of(cu_q_lens, num_reqs, t);
    int p = positions[t];
    int pb = block_tables[(size_t)r * max_blocks + p / block_size];
    for (int g = 0; g < num_kv_heads; ++g) {
      size_t dst = (((size_t)pb * num_kv_heads + g) * block_size + (p % block_size)) * head_dim;
      size_t src = ((size_t)t * num_kv_heads + g) * head_dim;
      memcpy(k_pool + dst, k_new + src, row);
      memcpy(v_pool + dst, v_new + src, row);
    }
  }
  return ORACLE_OK;
}

/*
 * FP8 append: the same scatter, each bf16 element x of k_new / v_new stored as
 * the E4M3 code of the fp32 quotient x / k_scale (x / v_scale).
 */
int oracle_append_fp8(uint8_t* k_pool, uint8_t* v_pool, float k_scale, float v_scale,
                      int num_blocks, int num_kv_heads, int block_size, int head_dim,
                      const int32_t* block_tables, int max_blocks, const int32_t* cu_q_lens,
                      const int32_t* positions, int num_reqs, int num_tokens,
                      const uint16_t* k_new, const uint16_t* v_new) {
  for (int t = 0; t < num_tokens; ++t) {
    int r = owner_of(cu_q_lens, num_reqs, t);
    if (r < 0) return ORACLE_EINVAL;
    int p = positions[t];
    if (p < 0 || p / block_size >= max_blocks) return ORACLE_EINVAL;
    int pb = block_tables[(size_t)r * max_blocks + p / block_size];
    if (pb < 0 || pb >= num_blocks) return ORACLE_EINVAL;
  }
  for (int t = 0; t < num_tokens; ++t) {
    int r = owner_of(cu_q_lens, num_reqs, t);
    int p = positions[t];
    int pb = block_tables[(size_t)r * max_blocks + p / block_size];
    for (int g = 0; g < num_kv_heads; ++g) {
      size_t dst = (((size_t)pb * num_kv_heads + g) * block_size + (p % block_size)) * head_dim;
      size_t src = ((size_t)t * num_kv_heads + g) * head_dim;
      for (int e = 0; e < head_dim; ++e) {
        float kx = (float)bf16_to_f64(k_new[src + e]);
        float vx = (float)bf16_to_f64(v_new[src + e]);
        float kq = kx / k_scale;   /* one IEEE fp32 division */
        float vq = vx / v_scale;
        k_pool[dst + e] = oracle_e4m3_encode(kq);
        v_pool[dst + e] = oracle_e4m3_encode(vq);
      }
    }
  }
  return ORACLE_OK;
}

/* Swap out: host[i] = (K block ids[i], V block ids[i]); host layout [n][2][hkv][bs][d]. */
int oracle_swap_out(const uint16_t* k_pool, const uint16_t* v_pool, int num_blocks,
                    int num_kv_heads, int block_size, int head_dim, const int32_t* ids, int n,
                    uint16_t* host) {
  size_t blk = (size_t)num_kv_heads * block_size * head_dim;
  for (int i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= num_blocks) return ORACLE_EINVAL;
  for (int i = 0; i < n; ++i) {
    memcpy(host + (size_t)i * 2 * blk, k_pool + (size_t)ids[i] * blk, blk * sizeof(uint16_t));
    memcpy(host + ((size_t)i * 2 + 1) * blk, v_pool + (size_t)ids[i] * blk, blk * sizeof(uint16_t));
  }
  return ORACLE_OK;
}

/* Swap in: the reverse copy, host [n][2][hkv][bs][d] into blocks ids[i]. */
int oracle_swap_in(uint16_t* k_pool, uint16_t* v_pool, int num_blocks, int num_kv_heads,
                   int block_size, int head_dim, const int32_t* ids, int n, const uint16_t* host) {
  size_t blk = (size_t)num_kv_heads * block_size * head_dim;
  for (int i = 0; i < n; ++i)
    if (ids[i] < 0 || ids[i] >= num_blocks) return ORACLE_EINVAL;
  for (int i = 0; i < n; ++i) {
    memcpy(k_pool + (size_t)ids[i] * blk, host + (size_t)i * 2 * blk, blk * sizeof(uint16_t));
    memcpy(v_pool + (size_t)ids[i] * blk, host + ((size_t)i * 2 + 1) * blk, blk * sizeof(uint16_t));
  }
  return ORACLE_OK;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
