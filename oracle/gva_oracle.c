/*
 * gva_oracle.c -- plain fp64 CPU oracle for the Grouped Value Attention (GVA) decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The CUDA library shares no code,
 * header, table or helper with it, and neither calls the other.  Everything here is
 * written for a reader to check against the pages by eye: no blocking, no fusion, no
 * reordering beyond what the definitions state.  All arithmetic is fp64.
 *
 * Sources (page title, section):
 *   [ABS]  "Grouped Value Attention: Efficient KV Caching via On-Demand Key Reconstruction"
 *          (abstract, huggingface.co/papers/2609.13285).
 *   [SUM]  ai-feeds.com summary "Grouped Value Attention:通过按需 key 重建实现高效 KV 缓存",
 *          sections 方法 (GVA 核心流程) and 核心洞察.
 *   [EXP]  m.szthrk.cn explainer, sections "GVA 的正式方案", "位置信息怎么办",
 *          "省下来的到底是多少".
 *   [REV]  review "[논문리뷰] Grouped Value Attention ...", section 3 (Methodology,
 *          Decoupled RoPE).
 *   [GQA]  explainer "GQA 分组查询注意力：KV Cache 与模型质量的折中", sections
 *          "MHA、MQA 与 GQA 的结构关系", "KV Cache 为什么会不断变大",
 *          "与位置编码和 KV Cache 的关系".
 *
 * What the method computes, per sequence b and query head h, at decode time:
 *   g      = g(h), the value group of head h                       [REV §3; GQA §结构关系]
 *   q'     = M_h q_c            (content key K_h = V_g M_h absorbed) [SUM §方法; EXP §正式方案]
 *   q~_r   = RoPE(q_r, p_q)     (decoupled positional slice)       [REV §3 Decoupled RoPE]
 *   s_j    = scale * (q' . v_j + q~_r . k~_r,j)   for j < T_b      [REV §3; SUM §方法]
 *   o      = sum_j softmax(s)_j v_j                                [SUM §方法 (value-weighted sum)]
 * The persistent cache holds per token only the G grouped values and ONE positional key
 * shared by all heads, stored already rotated [EXP §位置信息怎么办; REV §3].
 *
 * Readings taken where the pages are silent:
 *   - M_h is d_v x d_n and the column form of the absorbed query is q' = M_h q_c (the row
 *     form Q' = Q M^T of [SUM §方法]); K_h = V_g M_h means k_c,j = M_h^T v_j.
 *   - g(h) = floor(h / (H/G)): contiguous head blocks, as drawn in [GQA §结构关系].
 *   - RoPE: interleaved pairs (2i, 2i+1), theta_i = base^(-2i/d_r), rotation by +p*theta_i.
 *   - scale = 1/sqrt(d_n + d_r) unless the caller gives one.
 *   - The query sits at position T_b - 1 and attends to positions 0..T_b-1, itself
 *     included [GQA §KV Cache 为什么会不断变大, §与位置编码和 KV Cache 的关系].
 *   - Paged layout, 64-token blocks:  V element (blk, g, o, i) at ((blk*G+g)*64+o)*d_v+i,
 *     k_r element (blk, o, c) at (blk*64+o)*d_r+c, blk = table[b][p/64], o = p%64.
 *
 * Low-precision value cache (not on the pages; a reading of this library's own): the
 * value heads may be stored as OCP FP8 E4M3 codes (1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits; no infinities; S.1111.111 is NaN; largest finite 448), with one
 * power-of-two scale 2^e per (token, group).  e is the smallest integer with
 * max_i |v_i| <= 448 * 2^e, clamped to [-126, 120] (e = -126 for an all-zero row); each code
 * is v_i * 2^-e rounded once to the nearest E4M3 value (ties to even, magnitudes beyond 448
 * clamped to 448).  The stored value is code * 2^e, exact in fp64.  Pool layout: the codes
 * [NB][G][64][d_v] (one byte each) followed by the exponents [NB][G][64] (int8); the
 * positional keys stay bf16.
 *
 * Every function below is pinned by a CPU test against something other than itself
 * (closed forms, hand cases, library routines, invariants); see tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <fenv.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_F32 0
#define OR_BF16 1
#define OR_FP8 2 /* E4M3 value codes + per-(token, group) exponents; bf16 positional keys */
#define OR_BLOCK 64
#define OR_E4M3_MAX 448.0
#define OR_FP8_EMIN (-126)
#define OR_FP8_EMAX 120

#define OR_OK 0
#define OR_ERR_ARG 1
#define OR_ERR_INDEX 5

/* ------------------------------------------------------------------------------------ */
/* Number formats                                                                        */
/* ------------------------------------------------------------------------------------ */

/* bf16 is the top 16 bits of an IEEE binary32; widening is exact. */
double oracle_bf16_to_double(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a double to the nearest bf16 value, ties to even, in ONE rounding (no detour
 * through binary32, which could round twice).  bf16 has 8 significand bits and the
 * binary32 exponent range: normal numbers have spacing 2^(e-8) for |x| in [2^(e-1), 2^e),
 * subnormals have spacing 2^-133. */
uint16_t oracle_double_to_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  if (isinf(x)) return x > 0 ? 0x7F80 : 0xFF80;
  if (x == 0.0) return signbit(x) ? 0x8000 : 0x0000;
  int e;
  frexp(x, &e);                       /* |x| = m * 2^e, m in [0.5, 1) */
  int ulp_exp = e - 8;
  if (ulp_exp < -133) ulp_exp = -133; /* subnormal spacing */
  double q = ldexp(x, -ulp_exp);      /* exact: scaling by a power of two */
  int old = fegetround();
  fesetround(FE_TONEAREST);
  double r = nearbyint(q);            /* round half to even */
  fesetround(old);
  double y = ldexp(r, ulp_exp);
  float f = (float)y;                 /* exact unless it overflows to inf */
  if (isinf((double)f) || fabs(y) > 3.3895313892515355e38) return x > 0 ? 0x7F80 : 0xFF80;
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

/* E4M3 code -> value (exact).  Normal: (-1)^s (1 + m/8) 2^(E-7); subnormal (E = 0):
 * (-1)^s m 2^-9; S.1111.111 is NaN. */
double oracle_e4m3_to_double(uint8_t c) {
  int sgn = c >> 7, E = (c >> 3) & 15, m = c & 7;
  if (E == 15 && m == 7) return NAN;
  double mag = E == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, E - 7);
  return sgn ? -mag : mag;
}

/* Value -> E4M3 code, one rounding to nearest (ties to even); magnitudes that round beyond
 * 448 give +-448 (saturation), NaN gives 0x7F. */
uint8_t oracle_double_to_e4m3(double x) {
  if (isnan(x)) return 0x7F;
  uint8_t sgn = signbit(x) ? 0x80 : 0x00;
  double a = fabs(x);
  if (a == 0.0) return sgn;
  if (a > OR_E4M3_MAX) return (uint8_t)(sgn | 0x7E);  /* saturates (also infinities) */
  int e;
  frexp(a, &e);                      /* a = f * 2^e, f in [0.5, 1): spacing 2^(e-4) */
  int ulp_exp = e - 4;
  if (ulp_exp < -9) ulp_exp = -9;    /* subnormal spacing */
  int old = fegetround();
  fesetround(FE_TONEAREST);
  double r = nearbyint(ldexp(a, -ulp_exp)); /* exact scaling, then round half to even */
  fesetround(old);
  double y = ldexp(r, ulp_exp);
  if (y > OR_E4M3_MAX) y = OR_E4M3_MAX;
  if (y < ldexp(1.0, -6)) return (uint8_t)(sgn | (uint8_t)ldexp(y, 9)); /* subnormal or 0 */
  int ey;
  double fy = frexp(y, &ey);         /* y = fy * 2^ey: E = ey + 6, mantissa (2 fy - 1) * 8 */
  return (uint8_t)(sgn | ((ey + 6) << 3) | (int)((2.0 * fy - 1.0) * 8.0));
}

/* Exponent of the power-of-two scale of a row whose largest magnitude is amax: the smallest
 * e with amax <= 448 * 2^e, clamped to [-126, 120]; -126 for amax = 0. */
int oracle_fp8_exponent(double amax) {
  if (!(amax > 0.0)) return OR_FP8_EMIN;
  int E;
  double f = frexp(amax, &E);        /* amax = f * 2^E; 448 = 0.875 * 2^9 */
  int e = E - 9 + (f > 0.875 ? 1 : 0);
  if (e < OR_FP8_EMIN) e = OR_FP8_EMIN;
  if (e > OR_FP8_EMAX) e = OR_FP8_EMAX;
  return e;
}

static double load_elem(const void* base, int dtype, int64_t idx) {
  if (dtype == OR_F32) return (double)((const float*)base)[idx];
  return oracle_bf16_to_double(((const uint16_t*)base)[idx]);
}

/* Dtype of the positional-key pool: the fp8 cache keeps its keys in bf16. */
static int kr_dtype(int dtype) { return dtype == OR_FP8 ? OR_BF16 : dtype; }

/* Value element (blk, g, o, i) of a pool of num_blocks blocks. */
static double load_v(const void* v_pool, int dtype, int G, int d_v, int num_blocks, int64_t blk,
                     int g, int o, int i) {
  int64_t idx = (((blk * G + g) * OR_BLOCK) + o) * (int64_t)d_v + i;
  if (dtype != OR_FP8) return load_elem(v_pool, dtype, idx);
  const uint8_t* codes = (const uint8_t*)v_pool;
  const int8_t* exps = (const int8_t*)(codes + (int64_t)num_blocks * G * OR_BLOCK * d_v);
  return ldexp(oracle_e4m3_to_double(codes[idx]), exps[(blk * G + g) * OR_BLOCK + o]);
}

static void store_elem(void* base, int dtype, int64_t idx, double v) {
  if (dtype == OR_F32)
    ((float*)base)[idx] = (float)v; /* C conversion: round to nearest even */
  else
    ((uint16_t*)base)[idx] = oracle_double_to_bf16(v);
}

static int elem_size(int dtype) { return dtype == OR_F32 ? 4 : 2; }

/* Offset of the exponent of (blk, g, o) in an fp8 value pool (after all the codes). */
int64_t oracle_fp8_exp_offset(int G, int d_v, int num_blocks, int64_t blk, int g, int o) {
  return (int64_t)num_blocks * G * OR_BLOCK * d_v + (blk * G + g) * OR_BLOCK + o;
}

/* ------------------------------------------------------------------------------------ */
/* Decoupled RoPE on the positional slice  [REV §3 Decoupled RoPE; EXP §位置信息怎么办]     */
/* ------------------------------------------------------------------------------------ */

/* y = R(pos) x for a d_r-wide vector: pair (x_2i, x_2i+1) is turned by the angle
 * pos * base^(-2i/d_r).  x and y may alias. */
void oracle_rope(const double* x, int d_r, double pos, double base, double* y) {
  for (int i = 0; i < d_r / 2; ++i) {
    double theta = pow(base, -2.0 * (double)i / (double)d_r);
    double a = pos * theta;
    double c = cos(a), s = sin(a);
    double x0 = x[2 * i], x1 = x[2 * i + 1];
    y[2 * i] = x0 * c - x1 * s;
    y[2 * i + 1] = x0 * s + x1 * c;
  }
}

/* ------------------------------------------------------------------------------------ */
/* Query absorption  q' = M_h q_c  and query rotation  [SUM §方法; EXP §正式方案; REV §3]   */
/* ------------------------------------------------------------------------------------ */

/* q_c [B,H,d_n], q_r [B,H,d_r], pos_q [B], M [H,d_v,d_n] (M[h][i][k])
 * -> q_abs [B,H,d_v], q_rot [B,H,d_r]. */
int oracle_absorb(int B, int H, int d_v, int d_n, int d_r, double base, const double* q_c,
                  const double* q_r, const int32_t* pos_q, const double* M, double* q_abs,
                  double* q_rot) {
  if (B < 0 || H <= 0 || d_v <= 0 || d_n <= 0 || d_r < 0 || (d_r % 2) != 0) return OR_ERR_ARG;
  for (int b = 0; b < B; ++b) {
    for (int h = 0; h < H; ++h) {
      const double* qc = q_c + ((int64_t)b * H + h) * d_n;
      const double* Mh = M + (int64_t)h * d_v * d_n;
      double* qa = q_abs + ((int64_t)b * H + h) * d_v;
      for (int i = 0; i < d_v; ++i) {
        double acc = 0.0;
        for (int k = 0; k < d_n; ++k) acc += Mh[(int64_t)i * d_n + k] * qc[k];
        qa[i] = acc;
      }
      if (d_r > 0)
        oracle_rope(q_r + ((int64_t)b * H + h) * d_r, d_r, (double)pos_q[b], base,
                    q_rot + ((int64_t)b * H + h) * d_r);
    }
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------------------ */
/* Paged cache layout and append  [EXP §位置信息怎么办; GQA §与位置编码和 KV Cache 的关系]  */
/* ------------------------------------------------------------------------------------ */

int64_t oracle_v_offset(int G, int d_v, int64_t blk, int g, int o, int i) {
  return (((blk * G + g) * OR_BLOCK) + o) * (int64_t)d_v + i;
}

int64_t oracle_kr_offset(int d_r, int64_t blk, int o, int c) {
  return (blk * OR_BLOCK + o) * (int64_t)d_r + c;
}

/* Physical block holding position p of sequence b, or -1 when the table cannot hold it. */
int64_t oracle_block_of(const int32_t* block_table, int max_blocks, int num_blocks, int b,
                        int64_t p) {
  if (p < 0) return -1;
  int64_t lb = p / OR_BLOCK;
  if (lb >= max_blocks) return -1;
  int64_t blk = block_table[(int64_t)b * max_blocks + lb];
  if (blk < 0 || blk >= num_blocks) return -1;
  return blk;
}

/* Writes n new tokens per sequence at positions pos[b] .. pos[b]+n-1.
 * v_new [B,n,G,d_v] and kr_new [B,n,d_r] hold cache-dtype values; V is copied bit for bit,
 * the positional key is rotated to its own position in fp64 and rounded (nearest even)
 * to the cache dtype.  Tokens whose slot cannot be resolved are skipped and make the
 * call return OR_ERR_INDEX. */
int oracle_append(int dtype, int B, int n, int G, int d_v, int d_r, double base,
                  const void* v_new, const void* kr_new, const int32_t* pos,
                  const int32_t* block_table, int max_blocks, int num_blocks, void* v_pool,
                  void* kr_pool) {
  if ((dtype != OR_F32 && dtype != OR_BF16 && dtype != OR_FP8) || B < 0 || n < 0 || G <= 0 ||
      d_v <= 0 || d_r < 0 || (d_r % 2) != 0)
    return OR_ERR_ARG;
  int es = elem_size(kr_dtype(dtype)); /* the fp8 cache takes its new values in bf16 */
  int status = OR_OK;
  double* x = (double*)malloc(sizeof(double) * (d_r > 0 ? d_r : 1));
  for (int b = 0; b < B; ++b) {
    for (int t = 0; t < n; ++t) {
      int64_t p = (int64_t)pos[b] + t;
      int64_t blk = oracle_block_of(block_table, max_blocks, num_blocks, b, p);
      if (blk < 0) {
        status = OR_ERR_INDEX;
        continue;
      }
      int o = (int)(p % OR_BLOCK);
      for (int g = 0; g < G; ++g) {
        int64_t src_idx = (((int64_t)b * n + t) * G + g) * d_v;
        if (dtype == OR_FP8) {
          /* quantise the row: the scale exponent from its largest magnitude, then each value
           * times 2^-e (exact) rounded once to E4M3 */
          double amax = 0.0;
          for (int i = 0; i < d_v; ++i) {
            double v = fabs(load_elem(v_new, OR_BF16, src_idx + i));
            if (v > amax) amax = v;
          }
          int e = oracle_fp8_exponent(amax);
          uint8_t* codes = (uint8_t*)v_pool;
          for (int i = 0; i < d_v; ++i)
            codes[oracle_v_offset(G, d_v, blk, g, o, i)] =
                oracle_double_to_e4m3(ldexp(load_elem(v_new, OR_BF16, src_idx + i), -e));
          ((int8_t*)v_pool)[oracle_fp8_exp_offset(G, d_v, num_blocks, blk, g, o)] = (int8_t)e;
        } else {
          const char* src = (const char*)v_new + src_idx * es;
          char* dst = (char*)v_pool + oracle_v_offset(G, d_v, blk, g, o, 0) * es;
          memcpy(dst, src, (size_t)d_v * es);
        }
      }
      for (int c = 0; c < d_r; ++c)
        x[c] = load_elem(kr_new, kr_dtype(dtype), ((int64_t)b * n + t) * d_r + c);
      oracle_rope(x, d_r, (double)p, base, x);
      for (int c = 0; c < d_r; ++c)
        store_elem(kr_pool, kr_dtype(dtype), oracle_kr_offset(d_r, blk, o, c), x[c]);
    }
  }
  free(x);
  return status;
}

/* Cache scalars per token per layer, GVA over GQA with the same G and head width
 * [EXP §省下来的到底是多少]: (G*d_v + d_r) / (2*G*d_v). */
double oracle_cache_ratio(int G, int d_v, int d_r) {
  return ((double)G * d_v + d_r) / (2.0 * G * d_v);
}

/* Persistent cache bytes per token per layer: values and positional key in the cache dtype;
 * the fp8 cache holds G*d_v codes, G exponents and d_r bf16 key elements. */
double oracle_cache_bytes_per_token(int dtype, int G, int d_v, int d_r) {
  if (dtype == OR_FP8) return (double)G * d_v + G + 2.0 * d_r;
  return (double)elem_size(dtype) * ((double)G * d_v + d_r);
}

/* ------------------------------------------------------------------------------------ */
/* Decode attention over the compact cache  [SUM §方法; REV §3]                           */
/* ------------------------------------------------------------------------------------ */

/* Token range [j0, j1) of (b, h): running-free two-pass softmax pieces.
 * Writes m = max_j s_j, l = sum_j exp(s_j - m), u[i] = sum_j exp(s_j - m) v_j[i]. */
static int partial_bh(int dtype, int H, int G, int d_v, int d_r, double scale,
                      const void* v_pool, const void* kr_pool, const int32_t* block_table,
                      int max_blocks, int num_blocks, int b, int h, int64_t j0, int64_t j1,
                      const double* qa, const double* qr, double* m_out, double* l_out,
                      double* u) {
  int r = H / G;
  int g = h / r;
  int64_t len = j1 - j0;
  double* s = (double*)malloc(sizeof(double) * (len > 0 ? len : 1));
  for (int64_t j = j0; j < j1; ++j) {
    int64_t blk = oracle_block_of(block_table, max_blocks, num_blocks, b, j);
    if (blk < 0) {
      free(s);
      return OR_ERR_INDEX;
    }
    int o = (int)(j % OR_BLOCK);
    double content = 0.0, positional = 0.0;
    for (int i = 0; i < d_v; ++i)
      content += qa[i] * load_v(v_pool, dtype, G, d_v, num_blocks, blk, g, o, i);
    for (int c = 0; c < d_r; ++c)
      positional += qr[c] * load_elem(kr_pool, kr_dtype(dtype), oracle_kr_offset(d_r, blk, o, c));
    s[j - j0] = scale * (content + positional);
  }
  double m = -INFINITY;
  for (int64_t j = 0; j < len; ++j)
    if (s[j] > m) m = s[j];
  double l = 0.0;
  for (int i = 0; i < d_v; ++i) u[i] = 0.0;
  for (int64_t j = j0; j < j1; ++j) {
    double w = exp(s[j - j0] - m);
    l += w;
    int64_t blk = oracle_block_of(block_table, max_blocks, num_blocks, b, j);
    int o = (int)(j % OR_BLOCK);
    for (int i = 0; i < d_v; ++i)
      u[i] += w * load_v(v_pool, dtype, G, d_v, num_blocks, blk, g, o, i);
  }
  free(s);
  *m_out = m;
  *l_out = l;
  return OR_OK;
}

static double g_scale(int d_n, int d_r, double scale) {
  return scale > 0.0 ? scale : 1.0 / sqrt((double)(d_n + d_r));
}

/* One (b, h) output row: o = softmax(s) V over positions 0..seq_len-1. */
int oracle_decode_one(int dtype, int H, int G, int d_v, int d_n, int d_r, double scale,
                      const void* v_pool, const void* kr_pool, const int32_t* block_table,
                      int max_blocks, int num_blocks, const int32_t* seq_lens, int b, int h,
                      const double* q_abs, const double* q_rot, double* out_row) {
  if (H <= 0 || G <= 0 || H % G != 0 || d_v <= 0 || d_r < 0) return OR_ERR_ARG;
  int64_t T = seq_lens[b];
  if (T <= 0) return OR_ERR_ARG;
  double sc = g_scale(d_n, d_r, scale);
  const double* qa = q_abs + ((int64_t)b * H + h) * d_v;
  const double* qr = q_rot + ((int64_t)b * H + h) * (d_r > 0 ? d_r : 0);
  double m, l;
  int st = partial_bh(dtype, H, G, d_v, d_r, sc, v_pool, kr_pool, block_table, max_blocks,
                      num_blocks, b, h, 0, T, qa, qr, &m, &l, out_row);
  if (st != OR_OK) return st;
  for (int i = 0; i < d_v; ++i) out_row[i] /= l;
  return OR_OK;
}

/* Full output [B,H,d_v].  Parallel over (b, h) pairs when built with OpenMP. */
int oracle_decode(int dtype, int B, int H, int G, int d_v, int d_n, int d_r, double scale,
                  const void* v_pool, const void* kr_pool, const int32_t* block_table,
                  int max_blocks, int num_blocks, const int32_t* seq_lens, const double* q_abs,
                  const double* q_rot, double* out) {
  if (B < 0 || H <= 0 || G <= 0 || H % G != 0) return OR_ERR_ARG;
  int status = OR_OK;
  int64_t pairs = (int64_t)B * H;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < pairs; ++bh) {
    int b = (int)(bh / H), h = (int)(bh % H);
    int st = oracle_decode_one(dtype, H, G, d_v, d_n, d_r, scale, v_pool, kr_pool, block_table,
                               max_blocks, num_blocks, seq_lens, b, h, q_abs, q_rot,
                               out + bh * d_v);
    if (st != OR_OK) {
#pragma omp critical
      status = st;
    }
  }
  return status;
}

/* Several query tokens per sequence: the last n_q positions of the context (the tokens
 * just appended).  Query i of sequence b sits at position p = seq_lens[b] - n_q + i and reads
 * the cache up to and including its own position [GQA §与位置编码和 KV Cache 的关系], so
 * its output is the single-query definition over positions 0..p.
 * q_abs [B][n_q][H][d_v], q_rot [B][n_q][H][d_r], out [B][n_q][H][d_v].  Every seq_lens[b]
 * must be at least n_q. */
int oracle_decode_multi(int dtype, int B, int n_q, int H, int G, int d_v, int d_n, int d_r,
                        double scale, const void* v_pool, const void* kr_pool,
                        const int32_t* block_table, int max_blocks, int num_blocks,
                        const int32_t* seq_lens, const double* q_abs, const double* q_rot,
                        double* out) {
  if (B < 0 || n_q < 1 || H <= 0 || G <= 0 || H % G != 0 || d_v <= 0 || d_r < 0) return OR_ERR_ARG;
  for (int b = 0; b < B; ++b)
    if (seq_lens[b] < n_q) return OR_ERR_ARG;
  double sc = g_scale(d_n, d_r, scale);
  int status = OR_OK;
  int64_t rows = (int64_t)B * n_q * H;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t row = 0; row < rows; ++row) {
    int h = (int)(row % H);
    int64_t bi = row / H;
    int b = (int)(bi / n_q), i = (int)(bi % n_q);
    int64_t p = (int64_t)seq_lens[b] - n_q + i; /* the query's own position */
    const double* qa = q_abs + row * d_v;
    const double* qr = q_rot + row * (d_r > 0 ? d_r : 0);
    double m, l;
    double* o = out + row * d_v;
    int st = partial_bh(dtype, H, G, d_v, d_r, sc, v_pool, kr_pool, block_table, max_blocks,
                        num_blocks, b, h, 0, p + 1, qa, qr, &m, &l, o);
    if (st != OR_OK) {
#pragma omp critical
      status = st;
    } else {
      for (int k = 0; k < d_v; ++k) o[k] /= l;
    }
  }
  return status;
}

/* Split-T form: positions 0..T-1 cut into S contiguous ranges of near-equal length, one
 * partial (m, l, u) per range, then merged:  M = max m_s,  o = sum e^(m_s-M) u_s /
 * sum e^(m_s-M) l_s.  Must equal the unsplit result up to rounding. */
int oracle_decode_split(int dtype, int H, int G, int d_v, int d_n, int d_r, double scale,
                        const void* v_pool, const void* kr_pool, const int32_t* block_table,
                        int max_blocks, int num_blocks, const int32_t* seq_lens, int b, int h,
                        const double* q_abs, const double* q_rot, int S, double* out_row) {
  int64_t T = seq_lens[b];
  if (S <= 0 || T <= 0 || S > T) return OR_ERR_ARG;
  double sc = g_scale(d_n, d_r, scale);
  const double* qa = q_abs + ((int64_t)b * H + h) * d_v;
  const double* qr = q_rot + ((int64_t)b * H + h) * d_r;
  double* ms = (double*)malloc(sizeof(double) * S);
  double* ls = (double*)malloc(sizeof(double) * S);
  double* us = (double*)malloc(sizeof(double) * S * d_v);
  int status = OR_OK;
  for (int sidx = 0; sidx < S && status == OR_OK; ++sidx) {
    int64_t j0 = T * sidx / S, j1 = T * (sidx + 1) / S;
    status = partial_bh(dtype, H, G, d_v, d_r, sc, v_pool, kr_pool, block_table, max_blocks,
                        num_blocks, b, h, j0, j1, qa, qr, &ms[sidx], &ls[sidx], us + (int64_t)sidx * d_v);
  }
  if (status == OR_OK) {
    double Mx = -INFINITY;
    for (int sidx = 0; sidx < S; ++sidx)
      if (ms[sidx] > Mx) Mx = ms[sidx];
    double L = 0.0;
    for (int i = 0; i < d_v; ++i) out_row[i] = 0.0;
    for (int sidx = 0; sidx < S; ++sidx) {
      double w = exp(ms[sidx] - Mx);
      L += w * ls[sidx];
      for (int i = 0; i < d_v; ++i) out_row[i] += w * us[(int64_t)sidx * d_v + i];
    }
    for (int i = 0; i < d_v; ++i) out_row[i] /= L;
  }
  free(ms);
  free(ls);
  free(us);
  return status;
}

/* ------------------------------------------------------------------------------------ */
/* Unabsorbed form: materialise K_h = V_g M_h and score with the full key [k_c ; k~_r]     */
/* [SUM §方法; EXP §正式方案; REV §3].  Raw query inputs, not the absorbed ones.             */
/* ------------------------------------------------------------------------------------ */

int oracle_decode_unabsorbed(int dtype, int B, int H, int G, int d_v, int d_n, int d_r,
                             double scale, double base, const void* v_pool, const void* kr_pool,
                             const int32_t* block_table, int max_blocks, int num_blocks,
                             const int32_t* seq_lens, const double* q_c, const double* q_r,
                             const int32_t* pos_q, const double* M, double* out) {
  if (B < 0 || H <= 0 || G <= 0 || H % G != 0) return OR_ERR_ARG;
  double sc = g_scale(d_n, d_r, scale);
  int r = H / G;
  double* qrot = (double*)malloc(sizeof(double) * (d_r > 0 ? d_r : 1));
  double* kc = (double*)malloc(sizeof(double) * d_n);
  double* v = (double*)malloc(sizeof(double) * d_v);
  int status = OR_OK;
  for (int b = 0; b < B && status == OR_OK; ++b) {
    int64_t T = seq_lens[b];
    if (T <= 0) { status = OR_ERR_ARG; break; }
    double* s = (double*)malloc(sizeof(double) * T);
    for (int h = 0; h < H && status == OR_OK; ++h) {
      int g = h / r;
      const double* qc = q_c + ((int64_t)b * H + h) * d_n;
      const double* Mh = M + (int64_t)h * d_v * d_n;
      if (d_r > 0) oracle_rope(q_r + ((int64_t)b * H + h) * d_r, d_r, (double)pos_q[b], base, qrot);
      double m = -INFINITY;
      for (int64_t j = 0; j < T; ++j) {
        int64_t blk = oracle_block_of(block_table, max_blocks, num_blocks, b, j);
        if (blk < 0) { status = OR_ERR_INDEX; break; }
        int o = (int)(j % OR_BLOCK);
        for (int i = 0; i < d_v; ++i) v[i] = load_v(v_pool, dtype, G, d_v, num_blocks, blk, g, o, i);
        /* row vector k_c = v^T M_h, i.e. kc[k] = sum_i v[i] M_h[i][k] */
        for (int k = 0; k < d_n; ++k) {
          double acc = 0.0;
          for (int i = 0; i < d_v; ++i) acc += v[i] * Mh[(int64_t)i * d_n + k];
          kc[k] = acc;
        }
        double dot = 0.0;
        for (int k = 0; k < d_n; ++k) dot += qc[k] * kc[k];
        for (int c = 0; c < d_r; ++c)
          dot += qrot[c] * load_elem(kr_pool, kr_dtype(dtype), oracle_kr_offset(d_r, blk, o, c));
        s[j] = sc * dot;
        if (s[j] > m) m = s[j];
      }
      if (status != OR_OK) break;
      double l = 0.0;
      double* orow = out + ((int64_t)b * H + h) * d_v;
      for (int i = 0; i < d_v; ++i) orow[i] = 0.0;
      for (int64_t j = 0; j < T; ++j) {
        double w = exp(s[j] - m);
        l += w;
        int64_t blk = oracle_block_of(block_table, max_blocks, num_blocks, b, j);
        int o = (int)(j % OR_BLOCK);
        for (int i = 0; i < d_v; ++i) orow[i] += w * load_v(v_pool, dtype, G, d_v, num_blocks, blk, g, o, i);
      }
      for (int i = 0; i < d_v; ++i) orow[i] /= l;
    }
    free(s);
  }
  free(qrot);
  free(kc);
  free(v);
  return status;
}

/* ------------------------------------------------------------------------------------ */
/* Matching GQA decode (comparison workload): a key cache and a value cache, each         */
/* [NB][G][64][d], s_j = scale q_h . k_g(h),j   [GQA §一次 GQA 计算如何展开]              */
/* ------------------------------------------------------------------------------------ */

int oracle_gqa_decode_one(int dtype, int H, int G, int d, double scale, const void* k_pool,
                          const void* v_pool, const int32_t* block_table, int max_blocks,
                          int num_blocks, const int32_t* seq_lens, int b, int h, const double* q,
                          double* out_row) {
  if (H <= 0 || G <= 0 || H % G != 0 || d <= 0 || (dtype != OR_F32 && dtype != OR_BF16)) return OR_ERR_ARG;
  int64_t T = seq_lens[b];
  if (T <= 0) return OR_ERR_ARG;
  double sc = scale > 0.0 ? scale : 1.0 / sqrt((double)d);
  int g = h / (H / G);
  const double* qh = q + ((int64_t)b * H + h) * d;
  double* s = (double*)malloc(sizeof(double) * T);
  double m = -INFINITY;
  for (int64_t j = 0; j < T; ++j) {
    int64_t blk = oracle_block_of(block_table, max_blocks, num_blocks, b, j);
    if (blk < 0) { free(s); return OR_ERR_INDEX; }
    int o = (int)(j % OR_BLOCK);
    double dot = 0.0;
    for (int i = 0; i < d; ++i) dot += qh[i] * load_elem(k_pool, dtype, oracle_v_offset(G, d, blk, g, o, i));
    s[j] = sc * dot;
    if (s[j] > m) m = s[j];
  }
  double l = 0.0;
  for (int i = 0; i < d; ++i) out_row[i] = 0.0;
  for (int64_t j = 0; j < T; ++j) {
    double w = exp(s[j] - m);
    l += w;
    int64_t blk = oracle_block_of(block_table, max_blocks, num_blocks, b, j);
    int o = (int)(j % OR_BLOCK);
    for (int i = 0; i < d; ++i) out_row[i] += w * load_elem(v_pool, dtype, oracle_v_offset(G, d, blk, g, o, i));
  }
  for (int i = 0; i < d; ++i) out_row[i] /= l;
  free(s);
  return OR_OK;
}

/* ------------------------------------------------------------------------------------ */
/* Threads used by oracle_decode (reported with CPU timings).                             */
/* ------------------------------------------------------------------------------------ */

void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int oracle_get_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
