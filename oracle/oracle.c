/* oracle.c -- CPU oracle for the GGUF block-dequant GEMV and MoE path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or calls this
 * file; only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It is
 * plain C11 with float64 accumulation, written from the definitions of the block formats
 * and operations, with no blocking, fusion or reordering beyond what they state.  It
 * shares no code, header, table or constant with the CUDA library.
 *
 * Sources (the engine pages of the diskformer npm package, each a whole engine file):
 *  - ternary_bonsai_2_dflash.js (diskformer 0.5.4 -> 0.6.6), section "gguf.js": f16ToF32,
 *    the K-quant block layouts "follow ggml-quants.c", dequantQ4K / scaleMinK4, dequantQ6K.
 *  - gemma4_moe_ssd.js (diskformer 0.5.4 -> 0.6.6), WGSL preamble: Q4_0 value
 *    (nibble - 8) * scale, byte j holds values j and j + 16; Q6P / q6v per-index Q6_K decode.
 *  - qwen3_moe_ssd.js (diskformer 0.0.1 -> 0.3.0): header comment (Q8_0 = f16 scale + 32
 *    int8, kept bit-exact); WGSL kernels matmulQ8 (row dot), matmulF32 (router logits),
 *    topk (softmax, greedy top-k with ties to the lowest index, renormalised weights),
 *    expertQ8 (slot-indexed expert rows), siluMulMoe (SiLU(gate) * up), moeAccum
 *    (sum_j w_j * out_j in pick order, then the residual add).
 *  - qwen35_moe_ssd.js (diskformer 0.5.4 -> 0.6.6), BATCH_KERNELS: token-major batches,
 *    y[t*M + m] = sum_k x[t*N + k] * W[m][k] (matmulQ8T).
 *
 * Readings where the pages leave a step open:
 *  - raw byte order of Q8_0 / Q4_0 blocks: f16 d first, then the codes (ggml block_q8_0 /
 *    block_q4_0); the pages only show the split planes.
 *  - Q4_K element value: the exact real d*sc*q - dmin*m rounded once to f32 (RNE).  Both
 *    products are exact in f32, so the f32 subtraction below is that single rounding.
 *  - router: selection on the logits (softmax is monotone), ties to the lowest index;
 *    weights exp(l_j - lmax) / sum_picked exp(l_i - lmax), equal to p_j / sum p_picked.
 *  - MoE combine: out = x + sum_j w_j dn_j with the sum in pick order, then the residual.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OG_Q4_0 2
#define OG_Q8_0 8
#define OG_Q4_K 12
#define OG_Q6_K 14

#define OG_OK 0
#define OG_EBADTYPE (-1)
#define OG_EBADSHAPE (-2)
#define OG_ENOMEM (-3)

int og_version(void) { return 1; }

int og_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Elements and bytes per block of each type (ggml-quants block structs). */
static int og_block_shape(int type, int *qk, int *bb) {
  switch (type) {
    case OG_Q8_0: *qk = 32; *bb = 34; return 0;
    case OG_Q4_0: *qk = 32; *bb = 18; return 0;
    case OG_Q4_K: *qk = 256; *bb = 144; return 0;
    case OG_Q6_K: *qk = 256; *bb = 210; return 0;
    default: return -1;
  }
}

/* IEEE 754 binary16 -> value, by the definition of the format:
 *   e == 0:  (-1)^s * m * 2^-24            (zero and subnormals)
 *   e == 31: (-1)^s * inf, or NaN when m != 0
 *   else:    (-1)^s * (1024 + m) * 2^(e - 25)
 * The result is exact in float (and in double).  Follows f16ToF32 in ternary_bonsai_2_dflash.js. */
double og_f16_value(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp((double)(1024 + m), e - 25);
  return s ? -v : v;
}

float og_f16_to_f32(uint16_t h) { return (float)og_f16_value(h); }

static uint16_t le16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* Q4_K: 6-bit scale and min of sub-block j (0..7) from the 12 packed bytes
 * (get_scale_min_k4 in ggml-quants; scaleMinK4 in ternary_bonsai_2_dflash.js).
 * Sub-blocks 0..3 keep their scale in the low 6 bits of byte j and their min in the low 6
 * bits of byte j+4.  Sub-blocks 4..7 keep the low 4 bits of scale / min in the low / high
 * nibble of byte j+4, and the top 2 bits in the top 2 bits of byte j-4 (scale) / byte j (min). */
static void q4k_scale_min(const uint8_t *sc, int j, int *scale, int *min) {
  if (j < 4) {
    *scale = sc[j] & 63;
    *min = sc[j + 4] & 63;
  } else {
    *scale = (sc[j + 4] & 15) | ((sc[j - 4] >> 6) << 4);
    *min = (sc[j + 4] >> 4) | ((sc[j] >> 6) << 4);
  }
}

/* Value of element i of one block, as f32.  This is the dequantized weight. */
float og_block_value(int type, const uint8_t *blk, int i) {
  switch (type) {
    case OG_Q8_0: {
      /* d = f16 at bytes 0..1; element i is the int8 at byte 2 + i; value d * q (exact in f32) */
      double d = og_f16_value(le16(blk));
      int q = (int)(int8_t)blk[2 + i];
      return (float)(d * q);
    }
    case OG_Q4_0: {
      /* d = f16 at bytes 0..1; byte 2 + j holds element j (low nibble) and j + 16 (high) */
      double d = og_f16_value(le16(blk));
      int byte = blk[2 + (i & 15)];
      int nib = (i < 16) ? (byte & 15) : (byte >> 4);
      return (float)(d * (nib - 8));
    }
    case OG_Q4_K: {
      /* d, dmin = f16 at 0..1 and 2..3; scales at 4..15; nibbles at 16..143.  Element i lies
       * in 64-wide chunk c = i / 64: the first 32 take the low nibbles of bytes 32c..32c+31
       * (sub-block 2c), the next 32 the high nibbles of the same bytes (sub-block 2c + 1). */
      double d = og_f16_value(le16(blk)), dmin = og_f16_value(le16(blk + 2));
      int c = i / 64, r = i % 64;
      int byte = blk[16 + 32 * c + (r % 32)];
      int q = (r < 32) ? (byte & 15) : (byte >> 4);
      int scale, min;
      q4k_scale_min(blk + 4, 2 * c + (r >= 32), &scale, &min);
      float a = (float)(d * scale * q);  /* <= 21 significant bits: exact */
      float b = (float)(dmin * min);     /* <= 17 significant bits: exact */
      return a - b;                      /* one IEEE rounding of the exact difference */
    }
    case OG_Q6_K: {
      /* ql[128] at 0, qh[64] at 128, int8 scales[16] at 192, f16 d at 208.  Element i: half
       * n = i / 128, quarter qd = (i % 128) / 32, l = i % 32.  Low 4 bits from
       * ql[64n + l + 32 (qd & 1)] (low nibble for qd < 2, high nibble otherwise); high 2
       * bits from qh[32n + l] at bit 2 qd; scale index 8n + l / 16 + 2 qd; value
       * d * scale * (q - 32).  This is the per-index form of q6v (gemma4_moe_ssd.js). */
      double d = og_f16_value(le16(blk + 208));
      int n = i / 128, r = i % 128, qd = r / 32, l = r % 32;
      int lob = blk[64 * n + l + 32 * (qd & 1)];
      int lo = (qd < 2) ? (lob & 15) : (lob >> 4);
      int hi = (blk[128 + 32 * n + l] >> (2 * qd)) & 3;
      int q = lo | (hi << 4);
      int scale = (int)(int8_t)blk[192 + 8 * n + l / 16 + 2 * qd];
      return (float)(d * scale * (q - 32)); /* <= 23 significant bits: exact */
    }
    default:
      return NAN;
  }
}

/* Dequantize a [rows][n] tensor of raw blocks into f32. */
int og_dequant(int type, const uint8_t *w, int64_t rows, int64_t n, float *out) {
  int qk, bb;
  if (og_block_shape(type, &qk, &bb)) return OG_EBADTYPE;
  if (n % qk) return OG_EBADSHAPE;
  int64_t nb = n / qk;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < nb; ++b) {
      const uint8_t *blk = w + (r * nb + b) * bb;
      for (int i = 0; i < qk; ++i) out[r * n + b * qk + i] = og_block_value(type, blk, i);
    }
  return OG_OK;
}

/* Token-major quantized GEMV / GEMM (matmulQ8 for T = 1, matmulQ8T for T tokens):
 *   y[t][m] = sum_k w[m][k] * x[t][k],   bound[t][m] = sum_k |w[m][k] * x[t][k]|
 * w: raw blocks [M][N]; x: f32 [T][N]; y, bound: f64 [T][M] (bound may be NULL).
 * Each row is dequantized with og_block_value, then summed in float64 in index order. */
int og_gemv(int type, const uint8_t *w, int64_t M, int64_t N, const float *x, int64_t T,
            double *y, double *bound, int nthreads) {
  int qk, bb;
  if (og_block_shape(type, &qk, &bb)) return OG_EBADTYPE;
  if (N % qk || M < 0 || T < 0) return OG_EBADSHAPE;
  if (M == 0 || T == 0) return OG_OK;
  int64_t nb = N / qk;
  int failed = 0;
  if (nthreads < 1) nthreads = 1;
#pragma omp parallel num_threads(nthreads)
  {
    float *row = (float *)malloc((size_t)(N > 0 ? N : 1) * sizeof(float));
    if (!row) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
      if (!row) continue;
      for (int64_t b = 0; b < nb; ++b)
        for (int i = 0; i < qk; ++i) row[b * qk + i] = og_block_value(type, w + (m * nb + b) * bb, i);
      for (int64_t t = 0; t < T; ++t) {
        double s = 0.0, a = 0.0;
        const float *xt = x + t * N;
        for (int64_t k = 0; k < N; ++k) {
          double p = (double)row[k] * (double)xt[k];
          s += p;
          a += fabs(p);
        }
        y[t * M + m] = s;
        if (bound) bound[t * M + m] = a;
      }
    }
    free(row);
  }
  return failed ? OG_ENOMEM : OG_OK;
}

/* Router logits (matmulF32 / matmulF32T): l[t][e] = sum_h wr[e][h] * xn[t][h], f32 weights. */
int og_router_logits(const float *xn, const float *wr, int64_t T, int64_t H, int64_t E,
                     double *logits, double *bound) {
  for (int64_t t = 0; t < T; ++t)
    for (int64_t e = 0; e < E; ++e) {
      double s = 0.0, a = 0.0;
      for (int64_t h = 0; h < H; ++h) {
        double p = (double)wr[e * H + h] * (double)xn[t * H + h];
        s += p;
        a += fabs(p);
      }
      logits[t * E + e] = s;
      if (bound) bound[t * E + e] = a;
    }
  return OG_OK;
}

/* Router selection (topk / topkB): k rounds, each picking the largest remaining logit, ties
 * to the lowest expert index; weights are the softmax probabilities of the picks
 * renormalised over the picks, w_j = exp(l_j - lmax) / sum_{picked i} exp(l_i - lmax).
 * ids: int32 [T][k] in pick order; weights: f64 [T][k]. */
int og_topk(const double *logits, int64_t T, int64_t E, int k, int32_t *ids, double *weights) {
  if (k < 1 || k > E) return OG_EBADSHAPE;
  char *taken = (char *)malloc((size_t)E);
  if (!taken) return OG_ENOMEM;
  for (int64_t t = 0; t < T; ++t) {
    const double *l = logits + t * E;
    memset(taken, 0, (size_t)E);
    double lmax = l[0];
    for (int64_t e = 1; e < E; ++e)
      if (l[e] > lmax) lmax = l[e];
    double den = 0.0;
    for (int j = 0; j < k; ++j) {
      int64_t best = -1;
      for (int64_t e = 0; e < E; ++e)
        if (!taken[e] && (best < 0 || l[e] > l[best])) best = e;
      taken[best] = 1;
      ids[t * k + j] = (int32_t)best;
      den += exp(l[best] - lmax);
    }
    for (int j = 0; j < k; ++j) weights[t * k + j] = exp(l[ids[t * k + j]] - lmax) / den;
  }
  free(taken);
  return OG_OK;
}

/* SiLU(g) * u (siluMulMoe): g / (1 + e^-g) * u, as written on the page. */
double og_swiglu1(double g, double u) { return g / (1.0 + exp(-g)) * u; }

static const uint8_t *expert_base(const uint8_t *base, int64_t stride, const int32_t *slots, int32_t e) {
  int64_t slot = slots ? slots[e] : e;
  return base + slot * stride;
}

/* Slot-indexed gate/up expert rows and SwiGLU (expertQ8 with a shared input, siluMulMoe).
 * For pick z = t*k + j with expert e = ids[z] and slot s = slots[e] (identity when slots is
 * NULL): gate[z][i] = dot(Wg[s] row i, xn[t]), up[z][i] = dot(Wu[s] row i, xn[t]),
 * act[z][i] = SiLU(gate) * up.  Bounds are the sums of |products| of each dot. */
int og_moe_gate_up(int type, const uint8_t *w_gate, const uint8_t *w_up, int64_t expert_stride,
                   const int32_t *slots, const int32_t *ids, const float *xn, int64_t T, int k,
                   int64_t H, int64_t F, double *gate, double *up, double *act, double *bound_gate,
                   double *bound_up, int nthreads) {
  int qk, bb;
  if (og_block_shape(type, &qk, &bb)) return OG_EBADTYPE;
  if (H % qk) return OG_EBADSHAPE;
  int rc = OG_OK;
  for (int64_t z = 0; z < T * k && rc == OG_OK; ++z) {
    int64_t t = z / k;
    const uint8_t *g = expert_base(w_gate, expert_stride, slots, ids[z]);
    const uint8_t *u = expert_base(w_up, expert_stride, slots, ids[z]);
    rc = og_gemv(type, g, F, H, xn + t * H, 1, gate + z * F, bound_gate ? bound_gate + z * F : NULL, nthreads);
    if (rc == OG_OK)
      rc = og_gemv(type, u, F, H, xn + t * H, 1, up + z * F, bound_up ? bound_up + z * F : NULL, nthreads);
    for (int64_t i = 0; rc == OG_OK && i < F; ++i) act[z * F + i] = og_swiglu1(gate[z * F + i], up[z * F + i]);
  }
  return rc;
}

/* Down rows per pick and the weighted combine (expertQ8 with a per-pick input, moeAccum):
 *   dn[z][h] = dot(Wd[s] row h, act[z])
 *   out[t][h] = (add_residual ? x[t][h] : 0) + sum_{j=0..k-1} w[t][j] * dn[t*k + j][h]
 * with the sum taken in pick order and the residual added last.  act and w are float64
 * inputs so that either the oracle's own or another path's intermediates can be fed in.
 * bound_out[t][h] = |x| + sum_j |w_j| * sum_f |Wd[s][h][f] * act[z][f]|. */
int og_moe_down_combine(int type, const uint8_t *w_down, int64_t expert_stride, const int32_t *slots,
                        const int32_t *ids, const double *wts, const double *act, const float *x_in,
                        int64_t T, int k, int64_t H, int64_t F, int add_residual, double *dn,
                        double *bound_dn, double *out, double *bound_out, int nthreads) {
  int qk, bb;
  if (og_block_shape(type, &qk, &bb)) return OG_EBADTYPE;
  if (F % qk) return OG_EBADSHAPE;
  int64_t nb = F / qk;
  int failed = 0;
  if (nthreads < 1) nthreads = 1;
  for (int64_t z = 0; z < T * k; ++z) {
    const uint8_t *wd = expert_base(w_down, expert_stride, slots, ids[z]);
#pragma omp parallel num_threads(nthreads)
    {
      float *row = (float *)malloc((size_t)(F > 0 ? F : 1) * sizeof(float));
      if (!row) {
#pragma omp atomic write
        failed = 1;
      }
#pragma omp for schedule(static)
      for (int64_t h = 0; h < H; ++h) {
        if (!row) continue;
        for (int64_t b = 0; b < nb; ++b)
          for (int i = 0; i < qk; ++i) row[b * qk + i] = og_block_value(type, wd + (h * nb + b) * bb, i);
        double s = 0.0, a = 0.0;
        for (int64_t f = 0; f < F; ++f) {
          double p = (double)row[f] * act[z * F + f];
          s += p;
          a += fabs(p);
        }
        dn[z * H + h] = s;
        if (bound_dn) bound_dn[z * H + h] = a;
      }
      free(row);
    }
  }
  if (failed) return OG_ENOMEM;
  for (int64_t t = 0; t < T; ++t)
    for (int64_t h = 0; h < H; ++h) {
      double acc = 0.0, bnd = 0.0;
      for (int j = 0; j < k; ++j) {
        int64_t z = t * k + j;
        acc += wts[t * k + j] * dn[z * H + h];
        if (bound_dn) bnd += fabs(wts[t * k + j]) * bound_dn[z * H + h];
      }
      double xr = add_residual ? (double)x_in[t * H + h] : 0.0;
      out[t * H + h] = acc + xr;
      if (bound_out) bound_out[t * H + h] = bnd + fabs(xr);
    }
  return OG_OK;
}

/* Embedding row gather (embedQ8 in qwen3_moe_ssd.js, embedQ6K in gemma4_moe_ssd.js):
 *   out[i][k] = w(ids[i], k) * scale,   k < N
 * where w(r, k) is element k of row r of the [V][N] table, dequantized by og_block_value, and
 * the product is taken in float64 and rounded once to f32 (embedQ6K multiplies by its
 * p.scale; embedQ8 has none, scale = 1).  An id outside [0, V) is an error. */
int og_embed_rows(int type, const uint8_t *table, int64_t V, int64_t N, const int32_t *ids, int64_t n,
                  float scale, float *out) {
  int qk, bb;
  if (og_block_shape(type, &qk, &bb)) return OG_EBADTYPE;
  if (N % qk || V < 0 || n < 0) return OG_EBADSHAPE;
  int64_t nb = N / qk;
  for (int64_t i = 0; i < n; ++i) {
    if (ids[i] < 0 || ids[i] >= V) return OG_EBADSHAPE;
    const uint8_t *row = table + (int64_t)ids[i] * nb * bb;
    for (int64_t k = 0; k < N; ++k) {
      double v = (double)og_block_value(type, row + (k / qk) * bb, (int)(k % qk));
      out[i * N + k] = (float)(v * (double)scale);
    }
  }
  return OG_OK;
}

/* RMSNorm (rmsnorm in qwen3_moe_ssd.js): per row t,
 *   s_t = 1 / sqrt(mean_k x[t][k]^2 + eps),   y[t][k] = x[t][k] * s_t * w[k]
 * in float64 (the page scales x first, then multiplies by w). */
int og_rmsnorm(const float *x, const float *w, int64_t T, int64_t N, double eps, double *y) {
  if (T < 0 || N <= 0) return OG_EBADSHAPE;
  for (int64_t t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int64_t k = 0; k < N; ++k) ss += (double)x[t * N + k] * (double)x[t * N + k];
    double s = 1.0 / sqrt(ss / (double)N + eps);
    for (int64_t k = 0; k < N; ++k) y[t * N + k] = ((double)x[t * N + k] * s) * (double)w[k];
  }
  return OG_OK;
}

/* argmax of each row (argmax in qwen3_moe_ssd.js, argmaxRows in qwen35_dense.js): the lowest
 * index of the largest value.  NaN never compares larger, so it is never picked; a row with
 * no value other than NaN gives 0. */
int og_argmax_rows(const double *v, int64_t T, int64_t n, int32_t *ids) {
  if (T < 0 || n <= 0) return OG_EBADSHAPE;
  for (int64_t t = 0; t < T; ++t) {
    int64_t best = -1;
    for (int64_t i = 0; i < n; ++i) {
      double a = v[t * n + i];
      if (isnan(a)) continue;
      if (best < 0 || a > v[t * n + best]) best = i;
    }
    ids[t] = (int32_t)(best < 0 ? 0 : best);
  }
  return OG_OK;
}

/* ---- MoE variants on the same path ------------------------------------------------------ */

/* GELU in the tanh form with the argument clamped to [-10, 10] (GELU / TANH preamble of
 * gemma4_moe_ssd.js): 0.5 x (1 + tanh(clamp(0.7978845608 x (1 + 0.044715 x^2), -10, 10))). */
double og_gelu_tanh(double x) {
  double a = 0.7978845608 * x * (1.0 + 0.044715 * x * x);
  if (a < -10.0) a = -10.0;
  if (a > 10.0) a = 10.0;
  return 0.5 * x * (1.0 + tanh(a));
}

/* Logistic sigmoid (SIGMOID preamble): 1 / (1 + e^-x). */
double og_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Expert activation of gate and up rows: act = SiLU(g) * u (kind 0, siluMulMoe) or
 * GELU(g) * u (kind 1, geglu). */
int og_moe_act(int kind, const double *gate, const double *up, int64_t n, double *act) {
  if (kind != 0 && kind != 1) return OG_EBADSHAPE;
  for (int64_t i = 0; i < n; ++i)
    act[i] = kind == 0 ? og_swiglu1(gate[i], up[i]) : og_gelu_tanh(gate[i]) * up[i];
  return OG_OK;
}

/* The combine with its variants, from down rows dn [T*k][H] (og_moe_down_combine's):
 *   acc = sum_j (dn[t*k + j][h] * ds[e_j]) * w[t][j]   in pick order (moeSum; ds = 1 without a
 *         per-expert down scale, e_j = ids[t*k + j])
 *   acc = acc + sh[t][h] * sigmoid(sg[t])              with a shared expert (moeAccumShared)
 *   out[t][h] = acc + (add_residual ? x[t][h] : 0)     the residual last
 * bound_out = sum_j |ds_j w_j| bound_dn + |sh sigmoid(sg)| + |x|. */
int og_moe_combine_ex(const int32_t *ids, const double *wts, const double *dn, const double *bound_dn,
                      const float *down_scale, int64_t E, const float *shared_out, const float *shared_gate,
                      const float *x_in, int64_t T, int k, int64_t H, int add_residual, double *out,
                      double *bound_out) {
  if (T < 0 || k < 1 || H < 1) return OG_EBADSHAPE;
  for (int64_t t = 0; t < T; ++t) {
    double g = shared_out ? og_sigmoid((double)shared_gate[t]) : 0.0;
    for (int64_t h = 0; h < H; ++h) {
      double acc = 0.0, bnd = 0.0;
      for (int j = 0; j < k; ++j) {
        int64_t z = t * k + j;
        double ds = 1.0;
        if (down_scale) {
          if (ids[z] < 0 || ids[z] >= E) return OG_EBADSHAPE;
          ds = (double)down_scale[ids[z]];
        }
        acc = acc + (dn[z * H + h] * ds) * wts[z];
        if (bound_dn) bnd += fabs(ds * wts[z]) * bound_dn[z * H + h];
      }
      if (shared_out) {
        double sh = (double)shared_out[t * H + h] * g;
        acc = acc + sh;
        bnd += fabs(sh);
      }
      double xr = add_residual ? (double)x_in[t * H + h] : 0.0;
      out[t * H + h] = acc + xr;
      if (bound_out) bound_out[t * H + h] = bnd + fabs(xr);
    }
  }
  return OG_OK;
}

/* RMSNorm with a factor (rmsnormK of gemma4_moe_ssd.js, the router's input with k = 1/sqrt(H)):
 *   y[t][i] = ((x[t][i] * s_t) * k) * w[i],   s_t = 1 / sqrt(mean_i x[t][i]^2 + eps). */
int og_rmsnorm_k(const float *x, const float *w, int64_t T, int64_t N, double eps, double k, double *y) {
  if (T < 0 || N <= 0) return OG_EBADSHAPE;
  for (int64_t t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int64_t i = 0; i < N; ++i) ss += (double)x[t * N + i] * (double)x[t * N + i];
    double s = 1.0 / sqrt(ss / (double)N + eps);
    for (int64_t i = 0; i < N; ++i) y[t * N + i] = (((double)x[t * N + i] * s) * k) * (double)w[i];
  }
  return OG_OK;
}
