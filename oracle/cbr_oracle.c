/*
 * CPU oracle for the training-mode Conv -> BatchNorm -> ReLU (CBR) operator.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's CPU
 * baseline call this file.  The CUDA library never links, loads or calls it.  It shares no
 * code, header, table or helper with the CUDA path.
 *
 * Everything is plain fp64 loops written straight from the definitions on the pages.  The
 * loops are not blocked, fused or reordered beyond what the definition states.  OpenMP
 * splits only the outermost loop over independent outputs, so every sum is taken in the
 * same order as in the serial code.
 *
 * Layouts follow the Tech-Renaissance CBR page, section 8 (constraints): NHWC activations
 * and KRSC filters.  All arrays are dense, row-major and fp64.
 *
 * Sources:
 *  [TR]  Tech-Renaissance, "CBR fused operator: Conv + BatchNorm + ReLU" (article #20).
 *        Section 2: BN folding for inference.  Section 4.1: conv_fprop + genstats.
 *        Section 4.2: bn_finalize formulas.  Section 4.3: apply + ReLU + CMP_GT mask.
 *        Section 5.1: ReLU mask before batchnorm_backward.  Section 5.2: WGrad / DGrad.
 *        Section 6: inference graph.
 *  [BN]  dpshk.com, "BatchNorm CUDA implementation walkthrough".
 *        Section 2.1: per-channel normalisation over N x H x W.  Section 2.4: running-mean
 *        update.  Section 3.1: backward formulas (s1, s2, count).  Section 4.4: inference
 *        re-parameterisation.
 *  [TL]  devpress, "TileLang Conv2D+ReLU fusion case study", basic convolution section:
 *        output pixels x (KH*KW*C) x F view of the convolution (cross-correlation, NHWC).
 *
 * Parity pins for every function live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>

/* Output extent of a convolution without dilation ([TL] basic convolution section). */
int cbr_oracle_out_dim(int in, int k, int stride, int pad) { return (in + 2 * pad - k) / stride + 1; }

/*
 * z[n,p,q,k] = sum_{r,s,c} x[n, p*stride-pad+r, q*stride-pad+s, c] * w[k,r,s,c]
 * Padding positions contribute zero.  This is the direct 7-loop cross-correlation, the
 * conv_fprop of [TR] section 4.1 and the implicit GEMM of [TL].
 */
void cbr_oracle_conv2d_fwd(int N, int H, int W, int C, int K, int R, int S, int stride, int pad,
                           const double* x, const double* w, double* z) {
  const int P = cbr_oracle_out_dim(H, R, stride, pad);
  const int Q = cbr_oracle_out_dim(W, S, stride, pad);
#pragma omp parallel for collapse(2) schedule(static)
  for (int n = 0; n < N; ++n)
    for (int p = 0; p < P; ++p)
      for (int q = 0; q < Q; ++q)
        for (int k = 0; k < K; ++k) {
          double acc = 0.0;
          for (int r = 0; r < R; ++r) {
            const int h = p * stride - pad + r;
            if (h < 0 || h >= H) continue;
            for (int s = 0; s < S; ++s) {
              const int ww = q * stride - pad + s;
              if (ww < 0 || ww >= W) continue;
              const double* xp = x + (((size_t)n * H + h) * W + ww) * C;
              const double* wp = w + (((size_t)k * R + r) * S + s) * C;
              for (int c = 0; c < C; ++c) acc += xp[c] * wp[c];
            }
          }
          z[(((size_t)n * P + p) * Q + q) * K + k] = acc;
        }
}

/* The same fprop sum, evaluated only at the listed output pixels (n,p,q triples); all K
 * channels of each listed pixel are written to z_at[i*K + k]. */
void cbr_oracle_conv2d_fwd_at(int N, int H, int W, int C, int K, int R, int S, int stride, int pad,
                              const double* x, const double* w, int npix, const int32_t* pix,
                              double* z_at) {
  (void)N;
#pragma omp parallel for schedule(static)
  for (int i = 0; i < npix; ++i) {
    const int n = pix[3 * i], p = pix[3 * i + 1], q = pix[3 * i + 2];
    for (int k = 0; k < K; ++k) {
      double acc = 0.0;
      for (int r = 0; r < R; ++r) {
        const int h = p * stride - pad + r;
        if (h < 0 || h >= H) continue;
        for (int s = 0; s < S; ++s) {
          const int ww = q * stride - pad + s;
          if (ww < 0 || ww >= W) continue;
          const double* xp = x + (((size_t)n * H + h) * W + ww) * C;
          const double* wp = w + (((size_t)k * R + r) * S + s) * C;
          for (int c = 0; c < C; ++c) acc += xp[c] * wp[c];
        }
      }
      z_at[(size_t)i * K + k] = acc;
    }
  }
}

/*
 * Input gradient of the convolution ([TR] section 5.2, DGrad):
 * dx[n,h,w,c] = sum over (k,r,s) with h = p*stride-pad+r and w = q*stride-pad+s for a
 * valid output pixel (p,q) of dz[n,p,q,k] * w[k,r,s,c].
 */
void cbr_oracle_conv2d_dgrad(int N, int H, int W, int C, int K, int R, int S, int stride, int pad,
                             const double* dz, const double* w, double* dx) {
  const int P = cbr_oracle_out_dim(H, R, stride, pad);
  const int Q = cbr_oracle_out_dim(W, S, stride, pad);
#pragma omp parallel for collapse(2) schedule(static)
  for (int n = 0; n < N; ++n)
    for (int h = 0; h < H; ++h)
      for (int ww = 0; ww < W; ++ww)
        for (int c = 0; c < C; ++c) {
          double acc = 0.0;
          for (int r = 0; r < R; ++r) {
            const int tp = h + pad - r;
            if (tp < 0 || tp % stride != 0) continue;
            const int p = tp / stride;
            if (p >= P) continue;
            for (int s = 0; s < S; ++s) {
              const int tq = ww + pad - s;
              if (tq < 0 || tq % stride != 0) continue;
              const int q = tq / stride;
              if (q >= Q) continue;
              for (int k = 0; k < K; ++k)
                acc += dz[(((size_t)n * P + p) * Q + q) * K + k] * w[(((size_t)k * R + r) * S + s) * C + c];
            }
          }
          dx[(((size_t)n * H + h) * W + ww) * C + c] = acc;
        }
}

/* The same dgrad sum, evaluated only at the listed input pixels (n,h,w triples); all C
 * channels of each listed pixel are written to dx_at[i*C + c]. */
void cbr_oracle_conv2d_dgrad_at(int N, int H, int W, int C, int K, int R, int S, int stride, int pad,
                                const double* dz, const double* w, int npix, const int32_t* pix,
                                double* dx_at) {
  const int P = cbr_oracle_out_dim(H, R, stride, pad);
  const int Q = cbr_oracle_out_dim(W, S, stride, pad);
  (void)N;
#pragma omp parallel for schedule(static)
  for (int i = 0; i < npix; ++i) {
    const int n = pix[3 * i], h = pix[3 * i + 1], ww = pix[3 * i + 2];
    for (int c = 0; c < C; ++c) {
      double acc = 0.0;
      for (int r = 0; r < R; ++r) {
        const int tp = h + pad - r;
        if (tp < 0 || tp % stride != 0) continue;
        const int p = tp / stride;
        if (p >= P) continue;
        for (int s = 0; s < S; ++s) {
          const int tq = ww + pad - s;
          if (tq < 0 || tq % stride != 0) continue;
          const int q = tq / stride;
          if (q >= Q) continue;
          for (int k = 0; k < K; ++k)
            acc += dz[(((size_t)n * P + p) * Q + q) * K + k] * w[(((size_t)k * R + r) * S + s) * C + c];
        }
      }
      dx_at[(size_t)i * C + c] = acc;
    }
  }
}

/*
 * Weight gradient of the convolution ([TR] section 5.2, WGrad):
 * dw[k,r,s,c] = sum_{n,p,q} dz[n,p,q,k] * x[n, p*stride-pad+r, q*stride-pad+s, c]
 * Each (k,r,s) task walks the pixels in (n,p,q) order and keeps one running sum per c, so
 * every dw entry is summed in the same order as the plain 7-loop form.
 */
void cbr_oracle_conv2d_wgrad(int N, int H, int W, int C, int K, int R, int S, int stride, int pad,
                             const double* dz, const double* x, double* dw) {
  const int P = cbr_oracle_out_dim(H, R, stride, pad);
  const int Q = cbr_oracle_out_dim(W, S, stride, pad);
#pragma omp parallel for collapse(3) schedule(dynamic, 1)
  for (int k = 0; k < K; ++k)
    for (int r = 0; r < R; ++r)
      for (int s = 0; s < S; ++s) {
        double* out = dw + (((size_t)k * R + r) * S + s) * C;
        for (int c = 0; c < C; ++c) out[c] = 0.0;
        for (int n = 0; n < N; ++n)
          for (int p = 0; p < P; ++p) {
            const int h = p * stride - pad + r;
            if (h < 0 || h >= H) continue;
            for (int q = 0; q < Q; ++q) {
              const int ww = q * stride - pad + s;
              if (ww < 0 || ww >= W) continue;
              const double g = dz[(((size_t)n * P + p) * Q + q) * K + k];
              const double* xp = x + (((size_t)n * H + h) * W + ww) * C;
              for (int c = 0; c < C; ++c) out[c] += g * xp[c];
            }
          }
      }
}

/* The same wgrad sum for the listed filter taps only ((k,r,s) triples): all C channels of
 * each listed tap are written to dw_at[i*C + c], summed in the (n,p,q) order of the full
 * form. */
void cbr_oracle_conv2d_wgrad_at(int N, int H, int W, int C, int K, int R, int S, int stride, int pad,
                                const double* dz, const double* x, int ntap, const int32_t* tap,
                                double* dw_at) {
  const int P = cbr_oracle_out_dim(H, R, stride, pad);
  const int Q = cbr_oracle_out_dim(W, S, stride, pad);
#pragma omp parallel for schedule(dynamic, 1)
  for (int i = 0; i < ntap; ++i) {
    const int k = tap[3 * i], r = tap[3 * i + 1], s = tap[3 * i + 2];
    double* out = dw_at + (size_t)i * C;
    for (int c = 0; c < C; ++c) out[c] = 0.0;
    for (int n = 0; n < N; ++n)
      for (int p = 0; p < P; ++p) {
        const int h = p * stride - pad + r;
        if (h < 0 || h >= H) continue;
        for (int q = 0; q < Q; ++q) {
          const int ww = q * stride - pad + s;
          if (ww < 0 || ww >= W) continue;
          const double g = dz[(((size_t)n * P + p) * Q + q) * K + k];
          const double* xp = x + (((size_t)n * H + h) * W + ww) * C;
          for (int c = 0; c < C; ++c) out[c] += g * xp[c];
        }
      }
  }
}

/*
 * Per-channel batch statistics over the M = N*P*Q rows of z ([TR] section 4.2, N_ac;
 * [BN] section 2.1).  Two passes: mean = sum(z)/M, then the biased variance
 * var = sum((z - mean)^2)/M.
 */
void cbr_oracle_bn_batch_stats(int64_t M, int C, const double* z, double* mean, double* var) {
#pragma omp parallel for schedule(static)
  for (int c = 0; c < C; ++c) {
    double s = 0.0;
    for (int64_t m = 0; m < M; ++m) s += z[m * C + c];
    const double mu = s / (double)M;
    double v = 0.0;
    for (int64_t m = 0; m < M; ++m) {
      const double d = z[m * C + c] - mu;
      v += d * d;
    }
    mean[c] = mu;
    var[c] = v / (double)M;
  }
}

/*
 * Training-mode normalise, affine and ReLU ([TR] sections 4.2-4.3; [BN] section 2.1):
 *   xhat = (z - mean) / sqrt(var + eps),  pre = gamma*xhat + beta,
 *   y = max(0, pre),  mask = (pre > 0)  (the CMP_GT comparison: pre == 0 gives mask 0).
 * Any of xhat, pre, y, mask may be NULL.
 */
void cbr_oracle_bn_relu_fwd(int64_t M, int C, const double* z, const double* mean,
                            const double* var, const double* gamma, const double* beta, double eps,
                            double* xhat, double* pre, double* y, uint8_t* mask) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int c = 0; c < C; ++c) {
      const size_t i = (size_t)m * C + c;
      const double xh = (z[i] - mean[c]) / sqrt(var[c] + eps);
      const double pr = gamma[c] * xh + beta[c];
      if (xhat) xhat[i] = xh;
      if (pre) pre[i] = pr;
      if (y) y[i] = pr > 0.0 ? pr : 0.0;
      if (mask) mask[i] = pr > 0.0 ? 1 : 0;
    }
}

/*
 * Running-statistic update ([TR] section 4.2, momentum is the weight of the new batch;
 * [BN] section 2.4):
 *   rm <- (1 - momentum)*rm + momentum*mean
 *   rv <- (1 - momentum)*rv + momentum*var*M/(M-1)   (unbiased batch variance)
 * Also returns inv_std = 1/sqrt(var + eps), the saved_inv_var of [TR] section 4.2.
 */
void cbr_oracle_bn_finalize(int C, int64_t M, const double* mean, const double* var, double eps,
                            double momentum, double* running_mean, double* running_var,
                            double* inv_std) {
  for (int c = 0; c < C; ++c) {
    const double unbiased = var[c] * (double)M / (double)(M - 1);
    running_mean[c] = (1.0 - momentum) * running_mean[c] + momentum * mean[c];
    running_var[c] = (1.0 - momentum) * running_var[c] + momentum * unbiased;
    inv_std[c] = 1.0 / sqrt(var[c] + eps);
  }
}

/*
 * BN + ReLU backward ([TR] section 5.1: dY*mask first, then batchnorm_backward;
 * [BN] section 3.1):
 *   g = dy*mask,  dbeta = s1 = sum g,  dgamma = s2 = sum g*xhat,
 *   dz = gamma/sqrt(var+eps) * (g - s1/M - xhat*s2/M)
 * dz may be NULL (only the reductions are then produced).
 */
void cbr_oracle_bn_relu_bwd(int64_t M, int C, const double* dy, const uint8_t* mask,
                            const double* xhat, const double* var, const double* gamma, double eps,
                            double* dz, double* dgamma, double* dbeta) {
#pragma omp parallel for schedule(static)
  for (int c = 0; c < C; ++c) {
    double s1 = 0.0, s2 = 0.0;
    for (int64_t m = 0; m < M; ++m) {
      const size_t i = (size_t)m * C + c;
      const double g = mask[i] ? dy[i] : 0.0;
      s1 += g;
      s2 += g * xhat[i];
    }
    dbeta[c] = s1;
    dgamma[c] = s2;
    if (dz) {
      const double a = gamma[c] / sqrt(var[c] + eps);
      for (int64_t m = 0; m < M; ++m) {
        const size_t i = (size_t)m * C + c;
        const double g = mask[i] ? dy[i] : 0.0;
        dz[i] = a * (g - s1 / (double)M - xhat[i] * s2 / (double)M);
      }
    }
  }
}

/*
 * Inference-mode BN with running statistics, unfused ([BN] section 2.4):
 *   pre = gamma*(z - running_mean)/sqrt(running_var + eps) + beta
 */
void cbr_oracle_bn_infer(int64_t M, int C, const double* z, const double* running_mean,
                         const double* running_var, const double* gamma, const double* beta,
                         double eps, double* pre) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int c = 0; c < C; ++c) {
      const size_t i = (size_t)m * C + c;
      pre[i] = gamma[c] * (z[i] - running_mean[c]) / sqrt(running_var[c] + eps) + beta[c];
    }
}

/*
 * BN folding for inference ([TR] section 2; [BN] section 4.4):
 *   w_fold[k,...] = w[k,...] * gamma[k]/sqrt(var[k]+eps)
 *   b_fold[k]     = (b[k] - mean[k]) * gamma[k]/sqrt(var[k]+eps) + beta[k]
 * with the running statistics as mean/var.  conv_bias may be NULL (b = 0).
 */
void cbr_oracle_fold(int K, int RSC, const double* w, const double* conv_bias, const double* gamma,
                     const double* beta, const double* running_mean, const double* running_var,
                     double eps, double* w_fold, double* b_fold) {
  for (int k = 0; k < K; ++k) {
    const double scale = gamma[k] / sqrt(running_var[k] + eps);
    for (int j = 0; j < RSC; ++j) w_fold[(size_t)k * RSC + j] = w[(size_t)k * RSC + j] * scale;
    const double b = conv_bias ? conv_bias[k] : 0.0;
    b_fold[k] = (b - running_mean[k]) * scale + beta[k];
  }
}

/* out = max(0, z + bias[c]) : the conv + bias + ReLU of the folded inference form
 * ([TR] section 2, out = relu(conv(x, W_fold, b_fold))). */
void cbr_oracle_bias_relu(int64_t M, int C, const double* z, const double* bias, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t m = 0; m < M; ++m)
    for (int c = 0; c < C; ++c) {
      const double v = z[(size_t)m * C + c] + bias[c];
      out[(size_t)m * C + c] = v > 0.0 ? v : 0.0;
    }
}

/* Number of OpenMP threads the oracle uses (reported beside CPU timings). */
int cbr_oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
