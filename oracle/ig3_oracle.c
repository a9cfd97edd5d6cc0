/*
 * CPU oracle for the fused 3x3(x3) convolutions -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may load
 * this code.  It shares nothing with the CUDA library: every function below is
 * the plain definition of the result, written as nested loops in float64, with
 * no blocking, fusion or reordering beyond what the definition states.  The
 * only parallelism is an OpenMP loop over independent output blocks, which
 * does not change any arithmetic.
 *
 * Sources (web pages, cited by title and passage):
 *  [P47] "Kimi-K2.6__l2_p47" -- Conv3d(32->64, k=3) followed by Mish and Tanh.
 *  [P8]  "Kimi-K2.6__l2_p8"  -- Conv3d(8->16, k=3), /2, MaxPool3d(2),
 *                               AdaptiveAvgPool3d(1), +bias, sum over channels.
 *  [P86] "Kimi-K2.6__l1_p86" -- depthwise 3x3 (pad 1) then pointwise 1x1 Conv2d.
 *
 * Layouts (all dense, row-major, float32 inputs):
 *   x  [N][Cin][D][H][W]     w [Cout][Cin][3][3][3]     b [Cout] (may be NULL)
 *   y  [N][Cout][D-2][H-2][W-2]  (float64)
 *   dwsep: x [N][C][H][W], w_dw [C][1][3][3], w_pw [Cout][C][1][1], out [N][Cout][H][W]
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

typedef int64_t i64;

/* Threads the OpenMP loops use (for reporting). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/*
 * One output of the valid, stride-1, 3x3x3 cross-correlation (no kernel flip):
 *   y[n,k,od,oh,ow] = b[k] + sum_{c,kd,kh,kw} w[k,c,kd,kh,kw] * x[n,c,od+kd,oh+kh,ow+kw]
 * [P47] naive one-thread-per-output kernel and its NCDHW / [K,C,KD,KH,KW] index
 * check; output size D-3+1 etc. from the shape derivation at the page's start.
 */
double oracle_conv3d_at(const float* x, i64 N, i64 Cin, i64 D, i64 H, i64 W,
                        const float* w, i64 Cout, const float* b,
                        i64 n, i64 k, i64 od, i64 oh, i64 ow) {
  (void)N; (void)Cout;
  double acc = (b != NULL) ? (double)b[k] : 0.0;
  for (i64 c = 0; c < Cin; ++c)
    for (i64 kd = 0; kd < 3; ++kd)
      for (i64 kh = 0; kh < 3; ++kh)
        for (i64 kw = 0; kw < 3; ++kw) {
          double xv = (double)x[(((n * Cin + c) * D + (od + kd)) * H + (oh + kh)) * W + (ow + kw)];
          double wv = (double)w[(((k * Cin + c) * 3 + kd) * 3 + kh) * 3 + kw];
          acc += wv * xv;
        }
  return acc;
}

/* The whole conv output, y[N][Cout][D-2][H-2][W-2] in float64. */
void oracle_conv3d(const float* x, i64 N, i64 Cin, i64 D, i64 H, i64 W,
                   const float* w, i64 Cout, const float* b, double* y) {
  const i64 OD = D - 2, OH = H - 2, OW = W - 2;
  if (OD <= 0 || OH <= 0 || OW <= 0) return;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (i64 n = 0; n < N; ++n)
    for (i64 k = 0; k < Cout; ++k)
      for (i64 od = 0; od < OD; ++od)
        for (i64 oh = 0; oh < OH; ++oh)
          for (i64 ow = 0; ow < OW; ++ow)
            y[(((n * Cout + k) * OD + od) * OH + oh) * OW + ow] =
                oracle_conv3d_at(x, N, Cin, D, H, W, w, Cout, b, n, k, od, oh, ow);
}

/*
 * One output of the zero-padded, stride-1, 3x3x3 cross-correlation with padding P:
 *   y[n,k,od,oh,ow] = b[k] + sum_{c,kd,kh,kw} w[k,c,kd,kh,kw] * x[n,c,od+kd-P,oh+kh-P,ow+kw-P]
 * where x reads as zero outside [0,D) x [0,H) x [0,W); output size D+2P-2 etc.
 * [P47] the padding discussion: the input coordinate of an output is shifted by
 * -padding, the bounds check covers both ends and loads zero outside, and the output
 * size is (D + 2*padding - KD)/stride + 1.
 */
double oracle_conv3d_pad_at(const float* x, i64 N, i64 Cin, i64 D, i64 H, i64 W, i64 P,
                            const float* w, i64 Cout, const float* b,
                            i64 n, i64 k, i64 od, i64 oh, i64 ow) {
  (void)N; (void)Cout;
  double acc = (b != NULL) ? (double)b[k] : 0.0;
  for (i64 c = 0; c < Cin; ++c)
    for (i64 kd = 0; kd < 3; ++kd)
      for (i64 kh = 0; kh < 3; ++kh)
        for (i64 kw = 0; kw < 3; ++kw) {
          const i64 d = od + kd - P, h = oh + kh - P, ww = ow + kw - P;
          if (d < 0 || d >= D || h < 0 || h >= H || ww < 0 || ww >= W) continue;  /* zero */
          double xv = (double)x[(((n * Cin + c) * D + d) * H + h) * W + ww];
          double wv = (double)w[(((k * Cin + c) * 3 + kd) * 3 + kh) * 3 + kw];
          acc += wv * xv;
        }
  return acc;
}

/* The whole padded conv output, y[N][Cout][D+2P-2][H+2P-2][W+2P-2] in float64. */
void oracle_conv3d_pad(const float* x, i64 N, i64 Cin, i64 D, i64 H, i64 W, i64 P,
                       const float* w, i64 Cout, const float* b, double* y) {
  const i64 OD = D + 2 * P - 2, OH = H + 2 * P - 2, OW = W + 2 * P - 2;
  if (OD <= 0 || OH <= 0 || OW <= 0) return;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (i64 n = 0; n < N; ++n)
    for (i64 k = 0; k < Cout; ++k)
      for (i64 od = 0; od < OD; ++od)
        for (i64 oh = 0; oh < OH; ++oh)
          for (i64 ow = 0; ow < OW; ++ow)
            y[(((n * Cout + k) * OD + od) * OH + oh) * OW + ow] =
                oracle_conv3d_pad_at(x, N, Cin, D, H, W, P, w, Cout, b, n, k, od, oh, ow);
}

/*
 * One output of the zero-padded 3x3x3 cross-correlation with padding P and stride S:
 *   y[n,k,od,oh,ow] = b[k] + sum_{c,kd,kh,kw} w[k,c,kd,kh,kw] * x[n,c,od*S+kd-P,oh*S+kh-P,ow*S+kw-P]
 * (zero outside), output size (D + 2P - 3)/S + 1 etc. (integer division).  [P47] the
 * stride and padding discussion: the input window of output d_out starts at
 * d_out*stride - padding, and OD = (D + 2*padding - KD)/stride + 1.
 */
double oracle_conv3d_ex_at(const float* x, i64 N, i64 Cin, i64 D, i64 H, i64 W, i64 P, i64 S,
                           const float* w, i64 Cout, const float* b,
                           i64 n, i64 k, i64 od, i64 oh, i64 ow) {
  (void)N; (void)Cout;
  double acc = (b != NULL) ? (double)b[k] : 0.0;
  for (i64 c = 0; c < Cin; ++c)
    for (i64 kd = 0; kd < 3; ++kd)
      for (i64 kh = 0; kh < 3; ++kh)
        for (i64 kw = 0; kw < 3; ++kw) {
          const i64 d = od * S + kd - P, h = oh * S + kh - P, ww = ow * S + kw - P;
          if (d < 0 || d >= D || h < 0 || h >= H || ww < 0 || ww >= W) continue;  /* zero */
          double xv = (double)x[(((n * Cin + c) * D + d) * H + h) * W + ww];
          double wv = (double)w[(((k * Cin + c) * 3 + kd) * 3 + kh) * 3 + kw];
          acc += wv * xv;
        }
  return acc;
}

void oracle_conv3d_ex(const float* x, i64 N, i64 Cin, i64 D, i64 H, i64 W, i64 P, i64 S,
                      const float* w, i64 Cout, const float* b, double* y) {
  const i64 OD = (D + 2 * P - 3) / S + 1, OH = (H + 2 * P - 3) / S + 1, OW = (W + 2 * P - 3) / S + 1;
  if (D + 2 * P < 3 || H + 2 * P < 3 || W + 2 * P < 3) return;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (i64 n = 0; n < N; ++n)
    for (i64 k = 0; k < Cout; ++k)
      for (i64 od = 0; od < OD; ++od)
        for (i64 oh = 0; oh < OH; ++oh)
          for (i64 ow = 0; ow < OW; ++ow)
            y[(((n * Cout + k) * OD + od) * OH + oh) * OW + ow] =
                oracle_conv3d_ex_at(x, N, Cin, D, H, W, P, S, w, Cout, b, n, k, od, oh, ow);
}

/*
 * out = tanh(mish(y)), mish(y) = y * tanh(softplus(y)), softplus(y) = log(1 + e^y).
 * [P47] the activation description ("PyTorch computes mish first, then tanh").
 * Softplus is evaluated as log1p(exp(y)) with no threshold: for large y, exp
 * overflows to +inf, log1p(+inf) = +inf and tanh(+inf) = 1, so mish(y) = y.
 */
double oracle_tanh_mish(double y) {
  double softplus = log1p(exp(y));
  double mish = y * tanh(softplus);
  return tanh(mish);
}

void oracle_tanh_mish_array(const double* y, i64 count, double* out) {
#pragma omp parallel for schedule(static)
  for (i64 i = 0; i < count; ++i) out[i] = oracle_tanh_mish(y[i]);
}

/*
 * The reduction epilogue of [P8], step by step as the page lists it:
 *   z = y / divisor                                   (y already holds conv + bias)
 *   P[n,c,i,j,l] = max over the pool^3 block at (pool*i, pool*j, pool*l),
 *                  floor mode: i < OD/pool, j < OH/pool, l < OW/pool
 *   m[n,c] = (sum of P[n,c,...]) / (number of pooled cells)   (global average)
 *   out[n] = sum_c (m[n,c] + bias2[c])
 * y is [N][C][OD][OH][OW] float64; bias2 is [C]; out is [N].
 */
void oracle_pool_reduce(const double* y, i64 N, i64 C, i64 OD, i64 OH, i64 OW,
                        double divisor, i64 pool, const float* bias2, double* out) {
  const i64 PD = OD / pool, PH = OH / pool, PW = OW / pool;
  const i64 cells = PD * PH * PW;
  for (i64 n = 0; n < N; ++n) {
    double total = 0.0;
    for (i64 c = 0; c < C; ++c) {
      const double* yc = y + (n * C + c) * OD * OH * OW;
      double s = 0.0;
      for (i64 i = 0; i < PD; ++i)
        for (i64 j = 0; j < PH; ++j)
          for (i64 l = 0; l < PW; ++l) {
            double mx = -INFINITY;
            for (i64 a = 0; a < pool; ++a)
              for (i64 bb = 0; bb < pool; ++bb)
                for (i64 e = 0; e < pool; ++e) {
                  double z = yc[((i * pool + a) * OH + (j * pool + bb)) * OW + (l * pool + e)] / divisor;
                  if (z > mx) mx = z;
                }
            s += mx;
          }
      double mean = (cells > 0) ? s / (double)cells : 0.0;
      total += mean + (double)bias2[c];
    }
    out[n] = total;
  }
}

/*
 * Depthwise-separable conv2d of [P86], in its two stages:
 *   dw[n,c,h,w]  = sum_{kh,kw<3} w_dw[c,0,kh,kw] * x[n,c,h+kh-1,w+kw-1]   (zero outside)
 *   out[n,o,h,w] = sum_c w_pw[o,c,0,0] * dw[n,c,h,w]  (+ b[o] when b is not NULL)
 * [P86] the per-output pseudo-code (stride 1, padding 1, dilation 1) and the
 * input / depthwise / pointwise layouts listed beside it.
 * The depthwise stage is kept in float64 (scratch allocated here, per batch item).
 */
static double dw_at(const float* x, i64 C, i64 H, i64 W, const float* w_dw,
                    i64 n, i64 c, i64 h, i64 w) {
  double acc = 0.0;
  for (i64 kh = 0; kh < 3; ++kh)
    for (i64 kw = 0; kw < 3; ++kw) {
      i64 ih = h + kh - 1, iw = w + kw - 1;
      if (ih < 0 || ih >= H || iw < 0 || iw >= W) continue;
      acc += (double)w_dw[(c * 3 + kh) * 3 + kw] * (double)x[((n * C + c) * H + ih) * W + iw];
    }
  return acc;
}

int oracle_dwsep(const float* x, i64 N, i64 C, i64 H, i64 W, const float* w_dw,
                 const float* w_pw, i64 Cout, const float* b, double* out) {
  double* dw = (double*)malloc(sizeof(double) * (size_t)(C * H * W));
  if (dw == NULL) return -1;
  for (i64 n = 0; n < N; ++n) {
#pragma omp parallel for collapse(2) schedule(static)
    for (i64 c = 0; c < C; ++c)
      for (i64 h = 0; h < H; ++h)
        for (i64 w = 0; w < W; ++w)
          dw[(c * H + h) * W + w] = dw_at(x, C, H, W, w_dw, n, c, h, w);
#pragma omp parallel for collapse(2) schedule(static)
    for (i64 o = 0; o < Cout; ++o)
      for (i64 h = 0; h < H; ++h)
        for (i64 w = 0; w < W; ++w) {
          double acc = 0.0;
          for (i64 c = 0; c < C; ++c) acc += (double)w_pw[o * C + c] * dw[(c * H + h) * W + w];
          if (b != NULL) acc += (double)b[o];
          out[((n * Cout + o) * H + h) * W + w] = acc;
        }
  }
  free(dw);
  return 0;
}

/*
 * The same result as the single sum [P86] writes for one output:
 *   out[n,o,h,w] = sum_c w_pw[o,c] * sum_{kh,kw} w_dw[c,kh,kw] * x[n,c,h+kh-1,w+kw-1] (+ b[o])
 */
double oracle_dwsep_at(const float* x, i64 N, i64 C, i64 H, i64 W, const float* w_dw,
                       const float* w_pw, i64 Cout, const float* b,
                       i64 n, i64 o, i64 h, i64 w) {
  (void)N; (void)Cout;
  double acc = 0.0;
  for (i64 c = 0; c < C; ++c) {
    double dwv = 0.0;
    for (i64 kh = 0; kh < 3; ++kh)
      for (i64 kw = 0; kw < 3; ++kw) {
        i64 ih = h + kh - 1, iw = w + kw - 1;
        if (ih >= 0 && ih < H && iw >= 0 && iw < W)
          dwv += (double)x[((n * C + c) * H + ih) * W + iw] * (double)w_dw[(c * 3 + kh) * 3 + kw];
      }
    acc += dwv * (double)w_pw[o * C + c];
  }
  if (b != NULL) acc += (double)b[o];
  return acc;
}

void oracle_dwsep_single_sum(const float* x, i64 N, i64 C, i64 H, i64 W, const float* w_dw,
                             const float* w_pw, i64 Cout, const float* b, double* out) {
#pragma omp parallel for collapse(2) schedule(static)
  for (i64 n = 0; n < N; ++n)
    for (i64 o = 0; o < Cout; ++o)
      for (i64 h = 0; h < H; ++h)
        for (i64 w = 0; w < W; ++w)
          out[((n * Cout + o) * H + h) * W + w] =
              oracle_dwsep_at(x, N, C, H, W, w_dw, w_pw, Cout, b, n, o, h, w);
}

/*
 * Depthwise K x K (stride 1, dilation 1, "same" padding P = (K-1)/2, K odd) then
 * pointwise 1x1:
 *   dw[n,c,h,w]  = sum_{kh,kw<K} w_dw[c,0,kh,kw] * x[n,c,h+kh-P,w+kw-P]   (zero outside)
 *   out[n,o,h,w] = sum_c w_pw[o,c,0,0] * dw[n,c,h,w]  (+ b[o] when b is not NULL)
 * [P86] the discussion of kernel sizes other than 3 (a kernel templated on K and
 * dispatched for the common sizes 1, 3, 5, 7); K = 3 is the problem's padding 1, and
 * for the other sizes this reads the padding as the one that keeps H x W.
 * Two-stage (the depthwise stage in float64) and single-sum forms, as for K = 3.
 */
static double dwk_at(const float* x, i64 C, i64 H, i64 W, i64 K, const float* w_dw,
                     i64 n, i64 c, i64 h, i64 w) {
  const i64 P = (K - 1) / 2;
  double acc = 0.0;
  for (i64 kh = 0; kh < K; ++kh)
    for (i64 kw = 0; kw < K; ++kw) {
      i64 ih = h + kh - P, iw = w + kw - P;
      if (ih < 0 || ih >= H || iw < 0 || iw >= W) continue;
      acc += (double)w_dw[(c * K + kh) * K + kw] * (double)x[((n * C + c) * H + ih) * W + iw];
    }
  return acc;
}

int oracle_dwsep_k(const float* x, i64 N, i64 C, i64 H, i64 W, i64 K, const float* w_dw,
                   const float* w_pw, i64 Cout, const float* b, double* out) {
  double* dw = (double*)malloc(sizeof(double) * (size_t)(C * H * W));
  if (dw == NULL) return -1;
  for (i64 n = 0; n < N; ++n) {
#pragma omp parallel for collapse(2) schedule(static)
    for (i64 c = 0; c < C; ++c)
      for (i64 h = 0; h < H; ++h)
        for (i64 w = 0; w < W; ++w)
          dw[(c * H + h) * W + w] = dwk_at(x, C, H, W, K, w_dw, n, c, h, w);
#pragma omp parallel for collapse(2) schedule(static)
    for (i64 o = 0; o < Cout; ++o)
      for (i64 h = 0; h < H; ++h)
        for (i64 w = 0; w < W; ++w) {
          double acc = 0.0;
          for (i64 c = 0; c < C; ++c) acc += (double)w_pw[o * C + c] * dw[(c * H + h) * W + w];
          if (b != NULL) acc += (double)b[o];
          out[((n * Cout + o) * H + h) * W + w] = acc;
        }
  }
  free(dw);
  return 0;
}

double oracle_dwsep_k_at(const float* x, i64 N, i64 C, i64 H, i64 W, i64 K, const float* w_dw,
                         const float* w_pw, i64 Cout, const float* b, i64 n, i64 o, i64 h, i64 w) {
  (void)N; (void)Cout;
  const i64 P = (K - 1) / 2;
  double acc = 0.0;
  for (i64 c = 0; c < C; ++c) {
    double dwv = 0.0;
    for (i64 kh = 0; kh < K; ++kh)
      for (i64 kw = 0; kw < K; ++kw) {
        i64 ih = h + kh - P, iw = w + kw - P;
        if (ih >= 0 && ih < H && iw >= 0 && iw < W)
          dwv += (double)x[((n * C + c) * H + ih) * W + iw] * (double)w_dw[(c * K + kh) * K + kw];
      }
    acc += dwv * (double)w_pw[o * C + c];
  }
  if (b != NULL) acc += (double)b[o];
  return acc;
}
