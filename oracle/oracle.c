/*
 * oracle.c -- plain, slow CPU oracle for the CSA / HCA attention hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent definition that the
 * CUDA library is checked against.  Only the test suite, the smoke entry and
 * the benchmark's CPU-baseline leg may load it; the product path never does.
 * It shares no code, header, table or constant generator with the CUDA
 * sources, and it includes nothing from them.
 *
 * Every quantity is computed in fp64 from the exact values of the stored
 * inputs (bf16 or OCP FP8 E4M3 codes, decoded by the codecs below, which are
 * written from the format definitions).  Loops follow the method's steps in
 * order, with no blocking, fusion or reordering; OpenMP only spreads
 * independent queries / blocks over cores.
 *
 * Sources (page title, section):
 *  - "DeepSeek-V4: Towards Highly Efficient Million-Token Context
 *    Intelligence" (hyper.ai paper page), Method, CSA paragraph: every m
 *    tokens compressed into one entry with learnable compression weights and
 *    positional biases; a Lightning Indexer picks the top-k compressed entries;
 *    core attention is MQA over shared keys and values.
 *  - same page, Method, HCA paragraph: m' >> m, no overlapping compression,
 *    dense attention over all compressed entries; both branches add a
 *    sliding-window attention branch.
 *  - same page, Method: FP8 storage for non-RoPE KV, low precision indexer.
 *  - "DeepSeek-V4" (aiboss88 news page), Technical Principles: indexer score
 *    then top-k; sliding window and attention sink combined; FP8 range
 *    extension for the low-precision indexer QK path.
 *  - elamur.ai summary of the same paper, Summary: CSA "runs DeepSeek Sparse
 *    Attention" -- read here as the indexer form
 *    I(t,s) = sum_h w[t][h] * ReLU(q[t][h] . k[s]).
 *  - same page, References [95] (attention sinks): a per-head sink logit that
 *    joins the softmax denominator with a zero value vector.
 *
 * Readings where the pages are silent are listed in the design notes of the
 * repository (compression operator, visibility rule, window extent, FP8
 * scale rule, tie rule); each function below states the one it uses.
 *
 * Parity status: every function here is pinned by tests that do not re-type
 * it (closed forms, library routines on special cases, exhaustive checks);
 * see tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_RANGE 2
#define ORC_ERR_NOMEM 3

enum { ORC_BF16 = 0, ORC_FP8_E4M3 = 1, ORC_FP4_E2M1 = 2 };

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Number formats                                                           */
/* ------------------------------------------------------------------------ */

/* bf16: 1 sign bit, 8 exponent bits (bias 127), 7 stored mantissa bits; the
 * upper half of an IEEE binary32. */
double orc_bf16_to_f64(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round a double to the nearest bf16, ties to even, in one step (no detour
 * through binary32, which would round twice).  Results beyond the largest
 * finite value become infinity, as IEEE round-to-nearest prescribes. */
uint16_t orc_f64_to_bf16(double x) {
  if (isnan(x)) return 0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (isinf(a)) return sign | 0x7F80;
  if (a == 0.0) return sign;
  int e;
  frexp(a, &e);            /* a in [2^(e-1), 2^e) */
  int E = e - 1;
  int q = (E < -126) ? -133 : E - 7; /* exponent of one unit in the last place */
  double r = rint(ldexp(a, -q));     /* default rounding mode: nearest, ties to even */
  double v = ldexp(r, q);
  if (v >= ldexp(1.0, 128)) return sign | 0x7F80;
  float f = (float)v;                /* exact: v has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return sign | (uint16_t)(u >> 16);
}

/* OCP FP8 E4M3 ("E4M3FN"): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits, no infinities; S.1111.111 is NaN; largest finite 1.75 * 2^8 = 448;
 * exponent field 0 holds subnormals m * 2^-9. */
double orc_e4m3_to_f64(uint8_t c) {
  int s = c >> 7, E = (c >> 3) & 15, mnt = c & 7;
  double v;
  if (E == 15 && mnt == 7) return NAN;
  if (E == 0)
    v = ldexp((double)mnt, -9);
  else
    v = ldexp(1.0 + mnt / 8.0, E - 7);
  return s ? -v : v;
}

/* Nearest E4M3 value, ties to even; magnitudes beyond 448 saturate to 448
 * (the format has no infinity). */
uint8_t orc_f64_to_e4m3(double x) {
  if (isnan(x)) return 0x7F;
  uint8_t s = signbit(x) ? 0x80 : 0;
  double a = fabs(x);
  if (a >= 448.0) return s | 0x7E;
  if (a == 0.0) return s;
  int e;
  frexp(a, &e);
  int E = e - 1;
  int q = (E < -6) ? -9 : E - 3;
  double v = ldexp(rint(ldexp(a, -q)), q);
  if (v > 448.0) v = 448.0;
  if (v == 0.0) return s;
  frexp(v, &e);
  E = e - 1;
  if (E < -6) return s | (uint8_t)ldexp(v, 9);         /* subnormal */
  int mnt = (int)(ldexp(v, -E) * 8.0 - 8.0);            /* (v / 2^E - 1) * 8 */
  return s | (uint8_t)(((E + 7) << 3) | mnt);
}

void orc_bf16_decode_array(const uint16_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16_to_f64(in[i]);
}
void orc_bf16_encode_array(const double* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_bf16(in[i]);
}
void orc_e4m3_decode_array(const uint8_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_to_f64(in[i]);
}
void orc_e4m3_encode_array(const double* in, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_f64_to_e4m3(in[i]);
}

/* Per-row FP8 quantisation of compressed entries.  Reading of the pages'
 * "FP8 dynamic range" remark: one fp32 scale per entry, scale = amax / 448
 * (amax = 0 gives scale 1), stored as binary32; each channel is coded as the
 * nearest E4M3 value of y / scale, using the stored (binary32) scale. */
void orc_quantize_e4m3_rows(const double* y, int64_t rows, int d, uint8_t* codes,
                            float* scales) {
  for (int64_t r = 0; r < rows; ++r) {
    const double* yr = y + r * d;
    double amax = 0.0;
    for (int c = 0; c < d; ++c)
      if (fabs(yr[c]) > amax) amax = fabs(yr[c]);
    float sc = (amax > 0.0) ? (float)(amax / 448.0) : 1.0f;
    scales[r] = sc;
    for (int c = 0; c < d; ++c) codes[r * d + c] = orc_f64_to_e4m3(yr[c] / (double)sc);
  }
}

/* OCP FP4 E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit, no
 * infinities or NaN; exponent field 0 holds the subnormal m * 0.5.  The
 * magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double orc_e2m1_to_f64(uint8_t c) {
  int s = (c >> 3) & 1, E = (c >> 1) & 3, mnt = c & 1;
  double v = E == 0 ? 0.5 * mnt : ldexp(1.0 + 0.5 * mnt, E - 1);
  return s ? -v : v;
}

/* Nearest E2M1 value, ties to the even code (mantissa bit 0); magnitudes
 * beyond 6 saturate to 6. */
uint8_t orc_f64_to_e2m1(double x) {
  uint8_t s = signbit(x) ? 8 : 0;
  double a = fabs(x);
  if (isnan(x)) return 7;
  int best = 0;
  double bd = INFINITY;
  for (int c = 0; c < 8; ++c) {
    double d = fabs(a - orc_e2m1_to_f64((uint8_t)c));
    if (d < bd || (d == bd && (c & 1) == 0)) {
      bd = d;
      best = c;
    }
  }
  return s | (uint8_t)best;
}

void orc_e2m1_decode_array(const uint8_t* in, double* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_e2m1_to_f64(in[i]);
}

/* FP4 storage of indexer vectors.  Reading of the pages' FP4 indexer QK path
 * whose "dynamic range" is "extended with FP8": per block of 16 consecutive
 * channels one E4M3 scale, the nearest E4M3 value of amax / 6 (amax = 0
 * gives scale 1; a positive amax whose scale would round to 0 gets the
 * smallest positive E4M3 value, 2^-9); each channel is the nearest E2M1 value
 * of y / scale (ties to even, saturating at 6), using the decoded scale.
 * codes: rows of d/2 bytes, channel 2i in the low nibble of byte i;
 * scales: rows of d/16 E4M3 bytes.  d a multiple of 16. */
void orc_quantize_fp4_rows(const double* y, int64_t rows, int d, uint8_t* codes,
                           uint8_t* scales) {
  for (int64_t r = 0; r < rows; ++r) {
    const double* yr = y + r * d;
    for (int b = 0; b < d / 16; ++b) {
      double amax = 0.0;
      for (int c = 16 * b; c < 16 * b + 16; ++c)
        if (fabs(yr[c]) > amax) amax = fabs(yr[c]);
      uint8_t sc = amax > 0.0 ? orc_f64_to_e4m3(amax / 6.0) : orc_f64_to_e4m3(1.0);
      if (orc_e4m3_to_f64(sc) == 0.0) sc = 1;
      scales[r * (d / 16) + b] = sc;
      const double scv = orc_e4m3_to_f64(sc);
      for (int c = 16 * b; c < 16 * b + 16; ++c) {
        const uint8_t q = orc_f64_to_e2m1(yr[c] / scv);
        uint8_t* byte = codes + r * (d / 2) + c / 2;
        *byte = (c & 1) ? (uint8_t)((*byte & 0x0F) | (q << 4)) : (uint8_t)((*byte & 0xF0) | q);
      }
    }
  }
}

/* Values of FP4-stored vectors: rows of d channels from packed codes and
 * block scales (layout of orc_quantize_fp4_rows). */
void orc_fp4_dequantize_rows(const uint8_t* codes, const uint8_t* scales, int64_t rows, int d,
                             double* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int c = 0; c < d; ++c) {
      const uint8_t byte = codes[r * (d / 2) + c / 2];
      const uint8_t q = (c & 1) ? (byte >> 4) : (byte & 0x0F);
      out[r * d + c] = orc_e2m1_to_f64(q) * orc_e4m3_to_f64(scales[r * (d / 16) + c / 16]);
    }
}

/* ------------------------------------------------------------------------ */
/* Step a1: block compression                                               */
/* ------------------------------------------------------------------------ */

/* Compress blocks [block_begin, block_begin + n_blocks) of every sequence.
 * Block j (stride m) is compressed from the `span` raw tokens that end at its
 * last token, positions P(j) = { j*m + m - span + i : 0 <= i < span } minus the
 * negative ones (span = m: the non-overlapping blocks j*m .. j*m+m-1; span > m:
 * overlapping compression, the reading of the HCA paragraph's "without
 * overlapping compression" as setting HCA apart from CSA).  For each channel c
 * (the operator is the build's reading of "learnable compression weights and
 * positional biases"), over the positions p = j*m + m - span + i in P(j):
 *     g[i][c] = sum_e W[c][e] * x[p][e] + pos_bias[i][c]
 *     a[.][c] = softmax over those i of g[.][c]
 *     y[j][c] = sum_i a[i][c] * x[p][c]
 * raw: bf16 [B][raw_bstride] with token rows of d; W: bf16 [d][d] (row =
 * output channel); pos_bias: fp32 [span][d].  y: fp64 [B][n_blocks][d]. */
int orc_compress_span(const uint16_t* raw, int64_t raw_bstride, int B, int d, int m, int span,
                      int block_begin, int n_blocks, const uint16_t* W, const float* pos_bias,
                      double* y) {
  if (!raw || !W || !pos_bias || !y || B < 0 || d <= 0 || m <= 0 || span < m ||
      block_begin < 0 || n_blocks < 0)
    return ORC_ERR_ARG;
  if ((int64_t)(block_begin + n_blocks) * m * d > raw_bstride) return ORC_ERR_RANGE;
  double* Wd = (double*)malloc(sizeof(double) * (size_t)d * d);
  if (!Wd) return ORC_ERR_NOMEM;
  orc_bf16_decode_array(W, Wd, (int64_t)d * d);
  int err = ORC_OK;
#pragma omp parallel
  {
    double* x = (double*)malloc(sizeof(double) * (size_t)span * d);
    double* g = (double*)malloc(sizeof(double) * (size_t)span);
    if (!x || !g) {
#pragma omp atomic write
      err = ORC_ERR_NOMEM;
    }
#pragma omp for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
      for (int jj = 0; jj < n_blocks; ++jj) {
        if (!x || !g) continue;
        const int64_t j = block_begin + jj;
        const int64_t p0 = j * m + m - span;  /* position of bias row 0 */
        const int i0 = p0 < 0 ? (int)(-p0) : 0; /* first bias row with a token */
        const int n = span - i0;
        const uint16_t* xb = raw + (int64_t)b * raw_bstride + (p0 + i0) * d;
        orc_bf16_decode_array(xb, x, (int64_t)n * d);
        double* yo = y + ((int64_t)b * n_blocks + jj) * d;
        for (int c = 0; c < d; ++c) {
          for (int k = 0; k < n; ++k) {
            double s = 0.0;
            for (int e = 0; e < d; ++e) s += Wd[(int64_t)c * d + e] * x[(int64_t)k * d + e];
            g[k] = s + (double)pos_bias[(int64_t)(i0 + k) * d + c];
          }
          double gmax = g[0];
          for (int k = 1; k < n; ++k)
            if (g[k] > gmax) gmax = g[k];
          double den = 0.0, num = 0.0;
          for (int k = 0; k < n; ++k) {
            double a = exp(g[k] - gmax);
            den += a;
            num += a * x[(int64_t)k * d + c];
          }
          yo[c] = num / den;
        }
      }
    }
    free(x);
    free(g);
  }
  free(Wd);
  return err;
}

/* The non-overlapping blocks: span = m (pos_bias [m][d]). */
int orc_compress(const uint16_t* raw, int64_t raw_bstride, int B, int d, int m,
                 int block_begin, int n_blocks, const uint16_t* W, const float* pos_bias,
                 double* y) {
  return orc_compress_span(raw, raw_bstride, B, d, m, m, block_begin, n_blocks, W, pos_bias, y);
}

/* ------------------------------------------------------------------------ */
/* Step a2: Lightning-Indexer scores                                        */
/* ------------------------------------------------------------------------ */

/* Visible compressed entries for a query at absolute position t (block j is
 * visible iff it ends at or before t: j*m + m - 1 <= t), capped by the
 * number of entries present. */
static int64_t visible(int64_t t, int m, int64_t present) {
  int64_t nv = (t + 1) / m;
  return nv < present ? nv : present;
}

/* I(t,s) = sum_h w[t][h] * ReLU(q[t][h] . k[s]) for s < n_vis(t).
 * bf16: q, k are bf16 codes.  FP8: q, k are E4M3 codes and
 *     q[t][h] . k[s] = q_scale[t][h] * k_scale[s] * sum_d q8[d] * k8[d].
 * FP4: q, k are packed E2M1 codes (rows of dI/2 bytes) with E4M3 block
 *     scales (q_scale, k_scale then point to bytes: [B][T][H][dI/16] and
 *     [B][ks_bstride][dI/16]); the dot product is over the values
 *     code * block scale (orc_fp4_dequantize_rows).  k_bstride counts
 *     channels (elements) in every format.
 * q: [B][T][H][dI]; w, q_scale: [B][T][H]; k: [B][k_bstride] rows of dI;
 * k_scale: [B][ks_bstride].  scores: fp64 [B][T][N_out]; entries at and
 * beyond n_vis are -inf.  n_vis_out: [B][T]. */
int orc_indexer_scores(const void* q, const float* q_scale, const float* w, const void* k,
                       int64_t k_bstride, const float* k_scale, int64_t ks_bstride, int dtype,
                       const int32_t* q_pos, const int32_t* n_cmp, int B, int T, int H,
                       int dI, int m, int64_t N_out, double* scores, int32_t* n_vis_out) {
  if (!q || !w || !k || !q_pos || !n_cmp || !scores || B < 0 || T < 0 || H <= 0 ||
      dI <= 0 || m <= 0)
    return ORC_ERR_ARG;
  if (dtype != ORC_BF16 && dtype != ORC_FP8_E4M3 && dtype != ORC_FP4_E2M1) return ORC_ERR_ARG;
  if (dtype != ORC_BF16 && (!q_scale || !k_scale)) return ORC_ERR_ARG;
  if (dtype == ORC_FP4_E2M1 && (dI % 16 != 0 || k_bstride % 2 != 0)) return ORC_ERR_ARG;
  int err = ORC_OK;
#pragma omp parallel
  {
    double* qv = (double*)malloc(sizeof(double) * (size_t)H * dI);
    double* kv = (double*)malloc(sizeof(double) * (size_t)dI);
#pragma omp for collapse(2) schedule(dynamic)
    for (int b = 0; b < B; ++b) {
      for (int t = 0; t < T; ++t) {
        if (!qv || !kv) {
#pragma omp atomic write
          err = ORC_ERR_NOMEM;
          continue;
        }
        int64_t bt = (int64_t)b * T + t;
        int64_t tabs = q_pos[bt];
        if (tabs < 0 || n_cmp[b] < 0 || n_cmp[b] > N_out) {
#pragma omp atomic write
          err = ORC_ERR_RANGE;
          continue;
        }
        int64_t nv = visible(tabs, m, n_cmp[b]);
        if (n_vis_out) n_vis_out[bt] = (int32_t)nv;
        if (dtype == ORC_FP4_E2M1)
          orc_fp4_dequantize_rows((const uint8_t*)q + bt * H * (dI / 2),
                                  (const uint8_t*)q_scale + bt * H * (dI / 16), H, dI, qv);
        else
          for (int h = 0; h < H; ++h)
            for (int e = 0; e < dI; ++e) {
              int64_t o = (bt * H + h) * dI + e;
              qv[h * dI + e] = dtype == ORC_BF16 ? orc_bf16_to_f64(((const uint16_t*)q)[o])
                                                 : orc_e4m3_to_f64(((const uint8_t*)q)[o]);
            }
        double* out = scores + bt * N_out;
        for (int64_t s = 0; s < nv; ++s) {
          int64_t ko = (int64_t)b * k_bstride + s * dI;
          if (dtype == ORC_FP4_E2M1)
            orc_fp4_dequantize_rows((const uint8_t*)k + ko / 2,
                                    (const uint8_t*)k_scale +
                                        ((int64_t)b * ks_bstride + s) * (dI / 16),
                                    1, dI, kv);
          else
            for (int e = 0; e < dI; ++e)
              kv[e] = dtype == ORC_BF16 ? orc_bf16_to_f64(((const uint16_t*)k)[ko + e])
                                        : orc_e4m3_to_f64(((const uint8_t*)k)[ko + e]);
          double I = 0.0;
          for (int h = 0; h < H; ++h) {
            double dot = 0.0;
            for (int e = 0; e < dI; ++e) dot += qv[h * dI + e] * kv[e];
            if (dtype == ORC_FP8_E4M3)
              dot *= (double)q_scale[bt * H + h] * (double)k_scale[(int64_t)b * ks_bstride + s];
            I += (double)w[bt * H + h] * (dot > 0.0 ? dot : 0.0);
          }
          out[s] = I;
        }
        for (int64_t s = nv; s < N_out; ++s) out[s] = -INFINITY;
      }
    }
    free(qv);
    free(kv);
  }
  return err;
}

/* ------------------------------------------------------------------------ */
/* Step a3: top-k selection                                                 */
/* ------------------------------------------------------------------------ */

typedef struct {
  double s;
  int32_t i;
} scored_t;

/* Higher score first; equal scores: lower index first (the tie rule). */
static int by_score_then_index(const void* pa, const void* pb) {
  const scored_t* a = (const scored_t*)pa;
  const scored_t* b = (const scored_t*)pb;
  if (a->s > b->s) return -1;
  if (a->s < b->s) return 1;
  return (a->i > b->i) - (a->i < b->i);
}
static int ascending_i32(const void* pa, const void* pb) {
  int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
  return (a > b) - (a < b);
}

/* For each of Q queries: the min(k, n_vis) best entries by a full sort on
 * (-score, index), returned in ascending index order and padded with -1. */
int orc_topk(const double* scores, int64_t stride, const int32_t* n_vis, int64_t Q, int k,
             int32_t* idx_out) {
  if (!scores || !n_vis || !idx_out || Q < 0 || k < 0) return ORC_ERR_ARG;
  int err = ORC_OK;
#pragma omp parallel for schedule(dynamic)
  for (int64_t qq = 0; qq < Q; ++qq) {
    int64_t nv = n_vis[qq];
    int32_t* out = idx_out + qq * k;
    if (nv < 0 || nv > stride) {
#pragma omp atomic write
      err = ORC_ERR_RANGE;
      continue;
    }
    scored_t* arr = (scored_t*)malloc(sizeof(scored_t) * (size_t)(nv > 0 ? nv : 1));
    if (!arr) {
#pragma omp atomic write
      err = ORC_ERR_NOMEM;
      continue;
    }
    for (int64_t s = 0; s < nv; ++s) {
      arr[s].s = scores[qq * stride + s];
      arr[s].i = (int32_t)s;
    }
    qsort(arr, (size_t)nv, sizeof(scored_t), by_score_then_index);
    int64_t take = nv < k ? nv : k;
    for (int64_t r = 0; r < take; ++r) out[r] = arr[r].i;
    qsort(out, (size_t)take, sizeof(int32_t), ascending_i32);
    for (int64_t r = take; r < k; ++r) out[r] = -1;
    free(arr);
  }
  return err;
}

/* ------------------------------------------------------------------------ */
/* Steps a4 / a5: attention over compressed entries + window + sink          */
/* ------------------------------------------------------------------------ */

/* For query qq (sequence qb[qq], absolute position qt[qq]) and each head h,
 * over the key set
 *     S = { compressed rows sel[qq][i] for i < n_sel, sel >= 0 }
 *       u { raw rows p in [max(0, t - window + 1), t] }
 * (both parts count, even where a compressed entry summarises raw tokens that
 * are also in the window):
 *     l_j = scale * q_h . K_j
 *     M   = max(max_j l_j, sink_h)
 *     Z   = exp(sink_h - M) + sum_j exp(l_j - M)
 *     o_h = sum_j exp(l_j - M) * V_j / Z,      lse_h = M + ln Z
 * The sink term is absent when sink is NULL.  Empty S without a sink gives
 * o = 0 and lse = -inf.  MQA: one K and one V stream shared by all heads.
 * q: bf16 [Q][H][D].  k_cmp/v_cmp: bf16 [B][cmp_bstride] rows of D, with
 * n_cmp_rows valid rows per sequence.  k_raw/v_raw: bf16 [B][raw_bstride]
 * rows of D, row r holding absolute position raw_base + r, raw_rows rows.
 * out: fp64 [Q][H][D]; lse: fp64 [Q][H]. */
/* One stored K or V element: bf16 bits (raw rows, bf16 compressed rows) or an
 * already-decoded fp64 value (FP8-stored compressed rows, see
 * orc_kv8_dequantize). */
typedef struct {
  const void* row;
  int f64;
} orc_row;

static double orc_elem(orc_row r, int e) {
  return r.f64 ? ((const double*)r.row)[e] : orc_bf16_to_f64(((const uint16_t*)r.row)[e]);
}

static int attend_rows(const uint16_t* q, const int32_t* qb, const int32_t* qt, int64_t Q, int H,
                       int D, const void* k_cmp, const void* v_cmp, int cmp_f64,
                       int64_t cmp_bstride, int64_t n_cmp_rows, const int32_t* sel,
                       int64_t sel_stride, int n_sel, const uint16_t* k_raw,
                       const uint16_t* v_raw, int64_t raw_bstride, int64_t raw_base,
                       int64_t raw_rows, int window, const float* sink, double scale,
                       double* out, double* lse) {
  if (!q || !qb || !qt || !out || !lse || Q < 0 || H <= 0 || D <= 0 || n_sel < 0 ||
      window < 0)
    return ORC_ERR_ARG;
  if (n_sel > 0 && (!sel || !k_cmp || !v_cmp)) return ORC_ERR_ARG;
  if (window > 0 && (!k_raw || !v_raw)) return ORC_ERR_ARG;
  int err = ORC_OK;
  int64_t max_keys = (int64_t)n_sel + window;
#pragma omp parallel
  {
    double* qv = (double*)malloc(sizeof(double) * (size_t)D);
    orc_row* kr = (orc_row*)malloc(sizeof(orc_row) * (size_t)(max_keys + 1));
    orc_row* vr = (orc_row*)malloc(sizeof(orc_row) * (size_t)(max_keys + 1));
    double* l = (double*)malloc(sizeof(double) * (size_t)(max_keys + 1));
    double* acc = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic)
    for (int64_t qq = 0; qq < Q; ++qq) {
      if (!qv || !kr || !vr || !l || !acc) {
#pragma omp atomic write
        err = ORC_ERR_NOMEM;
        continue;
      }
      int64_t b = qb[qq], t = qt[qq];
      int64_t n = 0;
      int bad = 0;
      for (int i = 0; i < n_sel; ++i) {
        int64_t j = sel[qq * sel_stride + i];
        if (j < 0) continue;
        if (j >= n_cmp_rows) {
          bad = 1;
          break;
        }
        const int64_t off = b * cmp_bstride + j * D;
        kr[n].f64 = vr[n].f64 = cmp_f64;
        kr[n].row = cmp_f64 ? (const void*)((const double*)k_cmp + off)
                            : (const void*)((const uint16_t*)k_cmp + off);
        vr[n].row = cmp_f64 ? (const void*)((const double*)v_cmp + off)
                            : (const void*)((const uint16_t*)v_cmp + off);
        ++n;
      }
      int64_t p0 = t - window + 1;
      if (p0 < 0) p0 = 0;
      for (int64_t p = p0; window > 0 && p <= t; ++p) {
        int64_t r = p - raw_base;
        if (r < 0 || r >= raw_rows) {
          bad = 1;
          break;
        }
        kr[n].f64 = vr[n].f64 = 0;
        kr[n].row = k_raw + b * raw_bstride + r * D;
        vr[n].row = v_raw + b * raw_bstride + r * D;
        ++n;
      }
      if (bad) {
#pragma omp atomic write
        err = ORC_ERR_RANGE;
        continue;
      }
      for (int h = 0; h < H; ++h) {
        for (int e = 0; e < D; ++e) qv[e] = orc_bf16_to_f64(q[(qq * H + h) * D + e]);
        double M = -INFINITY;
        for (int64_t j = 0; j < n; ++j) {
          double s = 0.0;
          for (int e = 0; e < D; ++e) s += qv[e] * orc_elem(kr[j], e);
          l[j] = scale * s;
          if (l[j] > M) M = l[j];
        }
        double sk = sink ? (double)sink[h] : -INFINITY;
        if (sink && sk > M) M = sk;
        double* o = out + (qq * H + h) * D;
        if (M == -INFINITY) { /* empty set, no sink */
          for (int e = 0; e < D; ++e) o[e] = 0.0;
          lse[qq * H + h] = -INFINITY;
          continue;
        }
        double Z = sink ? exp(sk - M) : 0.0;
        for (int e = 0; e < D; ++e) acc[e] = 0.0;
        for (int64_t j = 0; j < n; ++j) {
          double p = exp(l[j] - M);
          Z += p;
          for (int e = 0; e < D; ++e) acc[e] += p * orc_elem(vr[j], e);
        }
        for (int e = 0; e < D; ++e) o[e] = acc[e] / Z;
        lse[qq * H + h] = M + log(Z);
      }
    }
    free(qv);
    free(kr);
    free(vr);
    free(l);
    free(acc);
  }
  return err;
}

int orc_attend(const uint16_t* q, const int32_t* qb, const int32_t* qt, int64_t Q, int H, int D,
               const uint16_t* k_cmp, const uint16_t* v_cmp, int64_t cmp_bstride,
               int64_t n_cmp_rows, const int32_t* sel, int64_t sel_stride, int n_sel,
               const uint16_t* k_raw, const uint16_t* v_raw, int64_t raw_bstride,
               int64_t raw_base, int64_t raw_rows, int window, const float* sink, double scale,
               double* out, double* lse) {
  return attend_rows(q, qb, qt, Q, H, D, k_cmp, v_cmp, 0, cmp_bstride, n_cmp_rows, sel,
                     sel_stride, n_sel, k_raw, v_raw, raw_bstride, raw_base, raw_rows, window,
                     sink, scale, out, lse);
}

/* The same with the compressed rows given as fp64 values (FP8-stored entries
 * decoded by orc_kv8_dequantize); the raw window rows stay bf16. */
int orc_attend_f64cmp(const uint16_t* q, const int32_t* qb, const int32_t* qt, int64_t Q, int H,
                      int D, const double* k_cmp, const double* v_cmp, int64_t cmp_bstride,
                      int64_t n_cmp_rows, const int32_t* sel, int64_t sel_stride, int n_sel,
                      const uint16_t* k_raw, const uint16_t* v_raw, int64_t raw_bstride,
                      int64_t raw_base, int64_t raw_rows, int window, const float* sink,
                      double scale, double* out, double* lse) {
  return attend_rows(q, qb, qt, Q, H, D, k_cmp, v_cmp, 1, cmp_bstride, n_cmp_rows, sel,
                     sel_stride, n_sel, k_raw, v_raw, raw_bstride, raw_base, raw_rows, window,
                     sink, scale, out, lse);
}

/* ------------------------------------------------------------------------ */
/* Mixed-precision storage of the compressed KV cache                       */
/* ------------------------------------------------------------------------ */

/* The hyper.ai DeepSeek-V4 page (Method) keeps the RoPE dimensions of the KV
 * entries in BF16 and stores the rest in FP8.  Reading: of a compressed
 * entry's d channels, the last n_rope are the RoPE channels (bf16); the first
 * d - n_rope are E4M3 codes with one fp32 scale per entry (the FP8 rule of
 * the indexer keys: scale = amax / 448 over those channels).  A V entry has no
 * RoPE channels (n_rope = 0).  Decoded value of channel c:
 *     c <  d - n_rope:  e4m3(codes[r][c]) * scale[r]
 *     c >= d - n_rope:  bf16(rope[r][c - (d - n_rope)])
 * codes: uint8 [rows][d - n_rope]; scale: fp32 [rows]; rope: bf16 bits
 * [rows][n_rope] (NULL when n_rope = 0); out: fp64 [rows][d]. */
int orc_kv8_dequantize(const uint8_t* codes, const float* scale, const uint16_t* rope,
                       int64_t rows, int d, int n_rope, double* out) {
  if (!codes || !scale || !out || rows < 0 || d <= 0 || n_rope < 0 || n_rope > d ||
      (n_rope > 0 && !rope))
    return ORC_ERR_ARG;
  const int dn = d - n_rope;
  for (int64_t r = 0; r < rows; ++r) {
    for (int c = 0; c < dn; ++c)
      out[r * d + c] = orc_e4m3_to_f64(codes[r * dn + c]) * (double)scale[r];
    for (int c = 0; c < n_rope; ++c) out[r * d + dn + c] = orc_bf16_to_f64(rope[r * n_rope + c]);
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Grouped output projection after the MQA core attention                   */
/* ------------------------------------------------------------------------ */

/* The hyper.ai DeepSeek-V4 page (Method, CSA paragraph) follows the MQA core
 * attention with "a grouped output projection".  Reading: the H heads of a
 * query's attention output are split into G groups of H/G consecutive heads;
 * group g's K = (H/G)*D values o_g (heads in order, D channels each) are
 * projected by its own matrix W_g (d_g rows of K):
 *     y[q][g*d_g + r] = sum_{j < K} W[g][r][j] * o[q][g*K + j]
 * o: bf16 [n][H*D]; W: bf16 [G][d_g][K]; y: fp64 [n][G*d_g]. */
int orc_grouped_out_proj(const uint16_t* o, const uint16_t* W, int64_t n, int H, int D, int G,
                         int d_g, double* y) {
  if (!o || !W || !y || n < 0 || H <= 0 || D <= 0 || G <= 0 || d_g <= 0 || H % G != 0)
    return ORC_ERR_ARG;
  const int K = (H / G) * D;
  int err = ORC_OK;
#pragma omp parallel
  {
    double* ov = (double*)malloc(sizeof(double) * (size_t)K);
    double* wv = (double*)malloc(sizeof(double) * (size_t)K);
#pragma omp for collapse(2) schedule(dynamic)
    for (int64_t q = 0; q < n; ++q) {
      for (int g = 0; g < G; ++g) {
        if (!ov || !wv) {
#pragma omp atomic write
          err = ORC_ERR_NOMEM;
          continue;
        }
        orc_bf16_decode_array(o + q * (int64_t)H * D + (int64_t)g * K, ov, K);
        for (int r = 0; r < d_g; ++r) {
          orc_bf16_decode_array(W + ((int64_t)g * d_g + r) * K, wv, K);
          double s = 0.0;
          for (int j = 0; j < K; ++j) s += wv[j] * ov[j];
          y[q * (int64_t)G * d_g + (int64_t)g * d_g + r] = s;
        }
      }
    }
    free(ov);
    free(wv);
  }
  return err;
}
