// K3: BN apply + ReLU + bit-packed mask (Tech-Renaissance CBR page, section 4.3:
//     relu(conv_out*eq_scale + eq_bias) with a CMP_GT mask stored as one bit per element).
// B1: BN + ReLU backward reduction (CBR page, section 5.1: dY*mask before batchnorm_backward;
//     BatchNorm CUDA page, section 3.1: dbeta = sum g, dgamma = sum g*xhat).  It also emits the
//     per-channel coefficients of dz = gamma*inv_std*(g - dbeta/M - xhat*dgamma/M), written as
//     dz = a*g - d*z + e.
// dz pass: evaluates that expression once and stores dz for both backward convolutions.
//
// All three are HBM-bound streams over NHWC tensors: 128-bit loads of 8 channels, several
// independent vectors in flight per thread, grid sized to the SM count.
#include <algorithm>
#include <map>
#include <mutex>
#include <type_traits>
#include <utility>

#include "cbr_internal.h"
#include "common.cuh"
#include "stats.cuh"

namespace cbr {
namespace {

constexpr int kApplyThreads = 256;
constexpr int kApplyUnroll = 4;
constexpr int kRedThreads = 512;
constexpr int kRedUnroll = 8;

// Sweeps the tensor last element first: the convolution before it wrote z first to last, so
// the end of z is what the L2 still holds.  The grid stride and the vector count are multiples
// of the c/8 vectors of a pixel (checked by the launcher), so every vector a thread visits has
// the same channel group and its eq_scale / eq_bias live in registers.
template <bool BF16, bool MASK>
__global__ void __launch_bounds__(kApplyThreads)
    bn_apply_relu_kernel(const ApplyArgs a) {
  const long long nvec = a.total / 8;
  const int cvec = a.c / 8;
  const long long stride = (long long)gridDim.x * kApplyThreads;
  const long long vfirst = (long long)blockIdx.x * kApplyThreads + threadIdx.x;
  if (vfirst >= nvec) return;
  const int c0 = (int)((nvec - 1 - vfirst) % cvec) * 8;
  float sc[8], bi[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    sc[e] = __ldg(a.eq + c0 + e);
    bi[e] = __ldg(a.eq + a.c + c0 + e);
  }
  const uint8_t* zb = static_cast<const uint8_t*>(a.z);
  uint8_t* yb = static_cast<uint8_t*>(a.y);
  for (long long v0 = vfirst; v0 < nvec; v0 += stride * kApplyUnroll) {
    uint4 in[kApplyUnroll];
#pragma unroll
    for (int k = 0; k < kApplyUnroll; ++k) {
      const long long v = nvec - 1 - (v0 + k * stride);
      if (v >= 0) in[k] = ld_global_nc_v4(zb + v * 16);
    }
#pragma unroll
    for (int k = 0; k < kApplyUnroll; ++k) {
      const long long v = nvec - 1 - (v0 + k * stride);
      if (v >= 0) {
        const uint32_t w[4] = {in[k].x, in[k].y, in[k].z, in[k].w};
        uint32_t o[4];
        uint32_t bits = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 zz = unpack2<BF16>(w[j]);
          const float p0 = fmaf(zz.x, sc[2 * j], bi[2 * j]);
          const float p1 = fmaf(zz.y, sc[2 * j + 1], bi[2 * j + 1]);
          bits |= (p0 > 0.f ? 1u : 0u) << (2 * j);
          bits |= (p1 > 0.f ? 1u : 0u) << (2 * j + 1);
          o[j] = pack2<BF16>(fmaxf(p0, 0.f), fmaxf(p1, 0.f));
        }
        st_global_v4(yb + v * 16, make_uint4(o[0], o[1], o[2], o[3]));
        if (MASK) a.mask[v] = (uint8_t)bits;
      }
    }
  }
}

// K2 + K3 for a training forward whose convolution left only its per-CTA partial moments
// (FpropArgs::defer): the finalize runs in this pass's prologue instead of on the last CTA of
// the convolution, where it was a serial tail of the forward.  Every block stages all partials
// in shared memory with one bulk copy, issues its first z loads, merges the partials with the
// same st::merge_partials the convolution's last CTA runs (so the statistics and y are the
// same bits either way) and keeps eq_scale / eq_bias in shared memory; block 0 also writes the
// saved and the running statistics.  The sweep is bn_apply_relu_kernel's, with one block of
// kMergeThreads per SM.
constexpr int kMergeThreads = 1024;

template <int C>
__host__ __device__ constexpr uint32_t merge_smem_bytes(int nparts) {
  return (uint32_t)nparts * st::partial_floats(C) * 4u + st::merge_scratch_floats<C>() * 4u + 2u * C * 4u + 16u;
}

template <bool BF16, bool MASK, int C>
__global__ void __launch_bounds__(kMergeThreads, 1)
    bn_apply_merge_kernel(const ApplyArgs a) {
  constexpr int kPF = st::partial_floats(C);
  constexpr int kCvec = C / 8;
  static_assert(kMergeThreads % kCvec == 0, "the grid stride must keep each thread's channel group");
  extern __shared__ __align__(16) uint8_t smem_apply[];
  float* parts = reinterpret_cast<float*>(smem_apply);   // [nparts][kPF]
  float* scratch = parts + (size_t)a.nparts * kPF;       // the merge's working set
  float* eqs = scratch + st::merge_scratch_floats<C>();  // eq_scale [C], eq_bias [C]
  const uint32_t bar = smem_u32(eqs + 2 * C);
  const uint32_t bytes = (uint32_t)a.nparts * kPF * 4u;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(bar, bytes);
    bulk_load_1d(smem_u32(parts), a.part, bytes, bar);
  }
  // the first z vectors of this thread, in flight while the partials are merged
  const long long nvec = a.total / 8;
  const long long stride = (long long)gridDim.x * kMergeThreads;
  const long long vfirst = (long long)blockIdx.x * kMergeThreads + threadIdx.x;
  const uint8_t* zb = static_cast<const uint8_t*>(a.z);
  uint8_t* yb = static_cast<uint8_t*>(a.y);
  uint4 in[kApplyUnroll];
#pragma unroll
  for (int k = 0; k < kApplyUnroll; ++k) {
    const long long v = nvec - 1 - (vfirst + k * stride);
    if (v >= 0) in[k] = ld_global_nc_v4(zb + v * 16);
  }
  float gm = 0.f, bt = 0.f, rm = 0.f, rv = 0.f;
  if (threadIdx.x < C) {
    gm = __ldg(a.gamma + threadIdx.x);
    bt = __ldg(a.beta + threadIdx.x);
    if (blockIdx.x == 0) {
      rm = a.running_mean[threadIdx.x];
      rv = a.running_var[threadIdx.x];
    }
  }
  bool staged = true;
  if (threadIdx.x < st::merge_threads<C>()) {
    staged = mbar_wait(bar, 0);
    if (!staged) report_error(a.err, kErrWaitOperand);
  }
  st::merge_partials<C, kMergeThreads, 2>(a.nparts, scratch, [&](int b, int c4, float4& m, float4& q, float& n) {
    const float* pb = parts + b * kPF;
    m = reinterpret_cast<const float4*>(pb)[c4];
    q = reinterpret_cast<const float4*>(pb + C)[c4];
    n = pb[2 * C];
  });
  if (threadIdx.x < C) {
    const int c = threadIdx.x;
    const float mean = scratch[c];
    const st::BnFinal f = st::bn_finalize(mean, scratch[C + c], gm, bt, rm, rv, a.inv_m, a.eps, a.momentum, a.unbias);
    eqs[c] = f.scale;
    eqs[C + c] = f.bias;
    if (blockIdx.x == 0) {
      a.saved_mean[c] = mean;
      a.saved_inv_var[c] = f.inv;
      a.running_mean[c] = f.run_mean;
      a.running_var[c] = f.run_var;
    }
  }
  __syncthreads();
  // a copy that never completed (reported above) is given one more bounded wait before the
  // block's shared memory is released
  if (!staged && threadIdx.x == 0) mbar_wait(bar, 0);
  if (vfirst >= nvec) return;
  const int c0 = (int)((nvec - 1 - vfirst) % kCvec) * 8;
  float sc[8], bi[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    sc[e] = eqs[c0 + e];
    bi[e] = eqs[C + c0 + e];
  }
  for (long long v0 = vfirst; v0 < nvec; v0 += stride * kApplyUnroll) {
    if (v0 != vfirst) {
#pragma unroll
      for (int k = 0; k < kApplyUnroll; ++k) {
        const long long v = nvec - 1 - (v0 + k * stride);
        if (v >= 0) in[k] = ld_global_nc_v4(zb + v * 16);
      }
    }
#pragma unroll
    for (int k = 0; k < kApplyUnroll; ++k) {
      const long long v = nvec - 1 - (v0 + k * stride);
      if (v >= 0) {
        const uint32_t w[4] = {in[k].x, in[k].y, in[k].z, in[k].w};
        uint32_t o[4];
        uint32_t bits = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 zz = unpack2<BF16>(w[j]);
          const float p0 = fmaf(zz.x, sc[2 * j], bi[2 * j]);
          const float p1 = fmaf(zz.y, sc[2 * j + 1], bi[2 * j + 1]);
          bits |= (p0 > 0.f ? 1u : 0u) << (2 * j);
          bits |= (p1 > 0.f ? 1u : 0u) << (2 * j + 1);
          o[j] = pack2<BF16>(fmaxf(p0, 0.f), fmaxf(p1, 0.f));
        }
        st_global_v4(yb + v * 16, make_uint4(o[0], o[1], o[2], o[3]));
        if (MASK) a.mask[v] = (uint8_t)bits;
      }
    }
  }
}

__device__ __forceinline__ void bwd_coef(double g, double gx, float gamma, float mean, float inv_std, double inv_m,
                                         int c, int ch, float* dgamma, float* dbeta, float* coef);

template <bool BF16, bool MASKBITS>
__global__ void __launch_bounds__(kRedThreads)
    bn_bwd_reduce_kernel(const BwdReduceArgs a) {
  // vectors in flight per thread (the y-derived mask needs a third operand)
  constexpr int kU = MASKBITS ? kRedUnroll : kRedUnroll / 2;
  __shared__ __align__(16) float red[kRedThreads * 16];  // the warps' sums; the grid sums at the end
  __shared__ uint32_t ticket;
  const int c = a.c;
  const int cvec = c / 8;
  const long long nvec = a.m_count * cvec;
  const long long stride = (long long)gridDim.x * kRedThreads;  // multiple of cvec
  const long long gtid = (long long)blockIdx.x * kRedThreads + threadIdx.x;
  const int c0 = (int)(gtid % cvec) * 8;
  float mean[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) mean[e] = a.mean[c0 + e];
  // the per-channel inputs of the finalize, loaded up front (see below)
  float f_inv = 0.f, f_gamma = 0.f, f_mean = 0.f;
  if (threadIdx.x < c && !a.sums_out) {
    f_inv = a.inv_std[threadIdx.x];
    f_gamma = a.gamma[threadIdx.x];
    f_mean = a.mean[threadIdx.x];
  }
  float sg[8], sgx[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) sg[e] = sgx[e] = 0.f;
  const uint8_t* dyb = static_cast<const uint8_t*>(a.dy);
  const uint8_t* zb = static_cast<const uint8_t*>(a.z);
  const uint8_t* yb = static_cast<const uint8_t*>(a.y);
  for (long long v0 = gtid; v0 < nvec; v0 += stride * kU) {
    uint4 dyv[kU], zv[kU], yv[kU];
    uint32_t mb[kU];
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      const long long v = v0 + k * stride;
      if (v < nvec) {
        dyv[k] = ld_global_nc_v4(dyb + v * 16);
        zv[k] = ld_global_nc_v4(zb + v * 16);
        if (MASKBITS) mb[k] = a.mask[v];
        else yv[k] = ld_global_nc_v4(yb + v * 16);
      }
    }
#pragma unroll
    for (int k = 0; k < kU; ++k) {
      const long long v = v0 + k * stride;
      if (v < nvec) {
        const uint32_t dw[4] = {dyv[k].x, dyv[k].y, dyv[k].z, dyv[k].w};
        const uint32_t zw[4] = {zv[k].x, zv[k].y, zv[k].z, zv[k].w};
        uint32_t bits;
        if (MASKBITS) {
          bits = mb[k];
        } else {
          const uint32_t yw[4] = {yv[k].x, yv[k].y, yv[k].z, yv[k].w};
          bits = 0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 yy = unpack2<BF16>(yw[j]);
            bits |= (yy.x > 0.f ? 1u : 0u) << (2 * j);
            bits |= (yy.y > 0.f ? 1u : 0u) << (2 * j + 1);
          }
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 d = unpack2<BF16>(dw[j]);
          const float2 z = unpack2<BF16>(zw[j]);
          const float g0 = (bits >> (2 * j)) & 1u ? d.x : 0.f;
          const float g1 = (bits >> (2 * j + 1)) & 1u ? d.y : 0.f;
          sg[2 * j] += g0;
          sg[2 * j + 1] += g1;
          sgx[2 * j] = fmaf(g0, z.x - mean[2 * j], sgx[2 * j]);
          sgx[2 * j + 1] = fmaf(g1, z.y - mean[2 * j + 1], sgx[2 * j + 1]);
        }
      }
    }
  }
  // block partial, in a fixed order: the lanes of a warp that share a channel group (lane mod
  // cvec) are combined by a butterfly, then the warps' sums by one thread per value
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll 1
  for (int o = cvec; o < 32; o <<= 1) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      sg[e] += __shfl_xor_sync(0xffffffffu, sg[e], o);
      sgx[e] += __shfl_xor_sync(0xffffffffu, sgx[e], o);
    }
  }
  // (cvec <= 32, checked by the launcher: lane l < cvec of every warp holds channel group l)
  constexpr int kWarps = kRedThreads / 32;
  if (lane < cvec) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      red[(warp * cvec + lane) * 16 + e] = sg[e];
      red[(warp * cvec + lane) * 16 + 8 + e] = sgx[e];
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < 2 * c; i += kRedThreads) {
    const int st = i / c, ch = i - st * c;
    const int grp = ch >> 3, e = ch & 7;
    float acc = 0.f;
    for (int w = 0; w < kWarps; ++w) acc += red[(w * cvec + grp) * 16 + st * 8 + e];
    a.part[(size_t)blockIdx.x * 2 * c + i] = acc;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) ticket = atomicInc(a.ticket, gridDim.x - 1);
  __syncthreads();
  if (ticket != gridDim.x - 1) return;
  // ------------------------------------------------------------ last block: finalize
  __threadfence();
  // One SM runs this after all the others, so it is kept short: every block partial is loaded
  // in one batch (thread t sums float4 column t / rgs of blocks t % rgs, + rgs, ..., in fp32 and
  // a fixed order), the row groups, rgs consecutive lanes of one warp, are combined by a fixed
  // pairwise butterfly (FP64 is slow on this part), and the coefficient math multiplies by the
  // host's 1/M instead of dividing.
  constexpr int kLd = 16;
  const int nv4 = (2 * c) / 4;                    // float4 columns of one partial (<= 128)
  const int rgs = min(kRedThreads / nv4, 32);     // row groups (a power of two)
  float* fred = red;                              // [2c]
  if (threadIdx.x < rgs * nv4) {
    const int rg = threadIdx.x % rgs, c4 = threadIdx.x / rgs;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int b0 = rg; b0 < (int)gridDim.x; b0 += kLd * rgs) {
      float4 v[kLd];
#pragma unroll
      for (int k = 0; k < kLd; ++k) {
        const int b = b0 + k * rgs;
        v[k] = b < (int)gridDim.x ? __ldcg(reinterpret_cast<const float4*>(a.part + (size_t)b * 2 * c) + c4)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < kLd; ++k) {
        acc.x += v[k].x;
        acc.y += v[k].y;
        acc.z += v[k].z;
        acc.w += v[k].w;
      }
    }
    // step w: lane r (r % 2w == 0) adds in lane r + w
    for (int w = 1; w < rgs; w *= 2) {
      const float bx = __shfl_down_sync(0xffffffffu, acc.x, w, rgs);
      const float by = __shfl_down_sync(0xffffffffu, acc.y, w, rgs);
      const float bz = __shfl_down_sync(0xffffffffu, acc.z, w, rgs);
      const float bw = __shfl_down_sync(0xffffffffu, acc.w, w, rgs);
      if ((rg & (2 * w - 1)) == 0) {
        acc.x += bx;
        acc.y += by;
        acc.z += bz;
        acc.w += bw;
      }
    }
    if (rg == 0) reinterpret_cast<float4*>(fred)[c4] = acc;
  }
  __syncthreads();
  const float* fin = fred;
  if (threadIdx.x < c) {
    const int ch = threadIdx.x;
    if (a.sums_out) {
      // split backward: the raw sums go to the caller, who adds other ranks' before the
      // coefficients are formed
      a.sums_out[ch] = fin[ch];
      a.sums_out[c + ch] = fin[c + ch];
    } else {
      bwd_coef(fin[ch], fin[c + ch], f_gamma, f_mean, f_inv, a.inv_m, c, ch, a.dgamma, a.dbeta, a.coef);
    }
  }
}

// dgamma, dbeta and the coefficients of dz = a*g - d*z + e for channel ch of c, from the sums
// g = sum of dy*mask and gx = sum of dy*mask*(z - mean) over the M rows (inv_m = 1/M):
// dgamma = gx*inv_std, dbeta = g, a = gamma*inv_std, d = a*dgamma*inv_std/M,
// e = -a*dbeta/M + d*mean (BatchNorm CUDA page, section 3.1).
__device__ __forceinline__ void bwd_coef(double g, double gx, float gamma, float mean, float inv_std, double inv_m,
                                         int c, int ch, float* dgamma, float* dbeta, float* coef) {
  const double inv = inv_std;
  const double dg = gx * inv;  // sum g * xhat
  const double db = g;
  const double ac = (double)gamma * inv;
  const double dc = ac * dg * inv * inv_m;
  const double ec = -ac * db * inv_m + dc * (double)mean;
  dgamma[ch] = (float)dg;
  dbeta[ch] = (float)db;
  coef[ch] = (float)ac;
  coef[c + ch] = (float)dc;
  coef[2 * c + ch] = (float)ec;
}

// Split backward, second half: one thread per channel, from the sums reduced over all ranks.
__global__ void bn_bwd_coef_kernel(const float* __restrict__ sums, int c, double inv_m, const float* gamma,
                                   const float* mean, const float* inv_std, float* dgamma, float* dbeta,
                                   float* coef) {
  const int ch = blockIdx.x * blockDim.x + threadIdx.x;
  if (ch < c) bwd_coef(sums[ch], sums[c + ch], gamma[ch], mean[ch], inv_std[ch], inv_m, c, ch, dgamma, dbeta, coef);
}

// Split forward, second half: merges `world` moment sets [mean c][M2 c][count] in order
// (Chan, in fp64: a few hundred values) and finalizes as the forward's last CTA does.
__global__ void bn_merge_finalize_kernel(const float* __restrict__ moments, int world, int c, const float* gamma,
                                         const float* beta, float* running_mean, float* running_var, float momentum,
                                         float eps, float* saved_mean, float* saved_inv_var, float* eq) {
  const int ch = blockIdx.x * blockDim.x + threadIdx.x;
  if (ch >= c) return;
  const int stride = 2 * c + 1;
  double n = 0.0, m = 0.0, q = 0.0;
  for (int r = 0; r < world; ++r) {
    const double nb = moments[(size_t)r * stride + 2 * c];
    const double mb = moments[(size_t)r * stride + ch], qb = moments[(size_t)r * stride + c + ch];
    const double nn = n + nb;
    if (nb > 0.0) {
      const double d = mb - m, fb = nb / nn;
      m += d * fb;
      q += qb + d * d * n * fb;
    }
    n = nn;
  }
  const float meanf = (float)m;
  const float var = n > 0.0 ? (float)(q / n) : 0.f;  // biased, for normalising
  const float inv = rsqrtf(var + eps);
  const float gm = gamma[ch];
  saved_mean[ch] = meanf;
  saved_inv_var[ch] = inv;
  eq[ch] = gm * inv;
  eq[c + ch] = beta[ch] - gm * meanf * inv;
  const float unbias = n > 1.0 ? (float)(n / (n - 1.0)) : 1.f;
  running_mean[ch] = (1.f - momentum) * running_mean[ch] + momentum * meanf;
  running_var[ch] = (1.f - momentum) * running_var[ch] + momentum * var * unbias;
}

__device__ __forceinline__ uint32_t fastdiv(uint32_t n, const FastDiv& f) {
  const uint32_t t = __umulhi(f.m, n);
  return (t + ((n - t) >> f.s1)) >> f.s2;
}

// dz = a*g - d*z + e with g = dy*mask, written to HBM once for both backward convolutions.
// Sweeps last element first: the reduction before it read dy and z first to last, so their
// ends are what the L2 still holds.  PAD: dz rows are stored with a pitch of a.pitch pixels
// (the padded-linear row space of the halo convolutions) and the thread holding an image
// row's last pixel also zeroes the row's pitch - q trailing pixels of its channel vector.
template <bool BF16, bool MASKBITS, bool PAD>
__global__ void __launch_bounds__(kApplyThreads)
    dz_kernel(const DzArgs a) {
  const long long nvec = a.total / 8;
  const int cvec = a.c / 8;
  const long long stride = (long long)gridDim.x * kApplyThreads;
  // as in the apply pass, a thread's channel group is fixed: its coefficients live in registers
  const long long vfirst = (long long)blockIdx.x * kApplyThreads + threadIdx.x;
  if (vfirst >= nvec) return;
  const uint32_t cv = (uint32_t)((nvec - 1 - vfirst) % cvec);
  const int c0 = (int)cv * 8;
  float ca[8], cd[8], ce[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    ca[e] = __ldg(a.coef + c0 + e);
    cd[e] = __ldg(a.coef + a.c + c0 + e);
    ce[e] = __ldg(a.coef + 2 * a.c + c0 + e);
  }
  const uint8_t* dyb = static_cast<const uint8_t*>(a.dy);
  const uint8_t* zb = static_cast<const uint8_t*>(a.z);
  const uint8_t* yb = static_cast<const uint8_t*>(a.y);
  uint8_t* ob = static_cast<uint8_t*>(a.dz);
  for (long long v0 = (long long)blockIdx.x * kApplyThreads + threadIdx.x; v0 < nvec;
       v0 += stride * kApplyUnroll) {
    uint4 dv[kApplyUnroll], zv[kApplyUnroll], yv[kApplyUnroll];
    uint32_t mb[kApplyUnroll];
#pragma unroll
    for (int k = 0; k < kApplyUnroll; ++k) {
      const long long v = nvec - 1 - (v0 + k * stride);
      if (v >= 0) {
        dv[k] = ld_global_nc_v4(dyb + v * 16);
        zv[k] = ld_global_nc_v4(zb + v * 16);
        if (MASKBITS) mb[k] = a.mask[v];
        else yv[k] = ld_global_nc_v4(yb + v * 16);
      }
    }
#pragma unroll
    for (int k = 0; k < kApplyUnroll; ++k) {
      const long long v = nvec - 1 - (v0 + k * stride);
      if (v >= 0) {
        // PAD: v < 2^31 (checked by the launcher), so the index math runs in 32 bits
        const uint32_t pix = PAD ? fastdiv((uint32_t)v, a.fd_cvec) : 0u;
        uint32_t bits;
        if (MASKBITS) {
          bits = mb[k];
        } else {
          const uint32_t yw[4] = {yv[k].x, yv[k].y, yv[k].z, yv[k].w};
          bits = 0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 yy = unpack2<BF16>(yw[j]);
            bits |= (yy.x > 0.f ? 1u : 0u) << (2 * j);
            bits |= (yy.y > 0.f ? 1u : 0u) << (2 * j + 1);
          }
        }
        const uint32_t dw[4] = {dv[k].x, dv[k].y, dv[k].z, dv[k].w};
        const uint32_t zw[4] = {zv[k].x, zv[k].y, zv[k].z, zv[k].w};
        uint32_t o[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 d = unpack2<BF16>(dw[j]);
          const float2 z = unpack2<BF16>(zw[j]);
          const float g0 = (bits >> (2 * j)) & 1u ? d.x : 0.f;
          const float g1 = (bits >> (2 * j + 1)) & 1u ? d.y : 0.f;
          const float r0 = fmaf(ca[2 * j], g0, fmaf(-cd[2 * j], z.x, ce[2 * j]));
          const float r1 = fmaf(ca[2 * j + 1], g1, fmaf(-cd[2 * j + 1], z.y, ce[2 * j + 1]));
          o[j] = pack2<BF16>(r0, r1);
        }
        if (PAD) {
          const uint32_t row = fastdiv(pix, a.fd_q);
          const uint32_t qq = pix - row * a.fd_q.d;
          const uint32_t dv32 = (row * (uint32_t)a.pitch + qq) * a.fd_cvec.d + cv;
          st_global_v4(ob + (size_t)dv32 * 16, make_uint4(o[0], o[1], o[2], o[3]));
          if (qq == a.fd_q.d - 1)
            for (uint32_t t = 1; t <= (uint32_t)(a.pitch - a.q); ++t)
              st_global_v4(ob + (size_t)(dv32 + t * a.fd_cvec.d) * 16, make_uint4(0u, 0u, 0u, 0u));
        } else {
          st_global_v4(ob + v * 16, make_uint4(o[0], o[1], o[2], o[3]));
        }
      }
    }
  }
}

}  // namespace

// Blocks of `kern` resident per SM, queried once per (kernel, device).
template <typename K>
int resident_blocks(K kern, int threads) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, int> cache;
  int dev = 0;
  cudaGetDevice(&dev);
  const auto key = std::make_pair(reinterpret_cast<const void*>(kern), dev);
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second;
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, threads, 0) != cudaSuccess || nb < 1) nb = 1;
  cache[key] = nb;
  return nb;
}

// Streaming grid: every block resident at once (one wave), grid-stride loops inside.
template <typename K>
int stream_grid(K kern, int threads, long long work_items, int num_sms) {
  const long long want = std::max<long long>(1, (work_items + threads - 1) / threads);
  return (int)std::min<long long>(want, (long long)num_sms * resident_blocks(kern, threads));
}

int launch_dz(const DzArgs& a_in, bool bf16, int num_sms, cudaStream_t st) {
  DzArgs a = a_in;
  // kApplyThreads (and so the grid stride) must be a multiple of the c/8 vectors of a pixel
  if (a.c % 8 != 0 || a.c > 256 || kApplyThreads % (a.c / 8) != 0 || a.q < 1 || a.pitch < a.q) return 3;
  const long long nvec = a.total / 8;
  const bool bits = a.mask != nullptr;
  const bool pad = a.pitch != a.q;
  // padded stores index in 32 bits: every vector of the padded tensor must fit
  if (pad && nvec / a.q * a.pitch >= (1ll << 31)) return 3;
  a.fd_cvec = make_fastdiv((uint32_t)(a.c / 8));
  a.fd_q = make_fastdiv((uint32_t)a.q);
  auto go = [&](auto kern) {
    kern<<<stream_grid(kern, kApplyThreads, nvec / kApplyUnroll, num_sms), kApplyThreads, 0, st>>>(a);
  };
  const int sel = (bf16 ? 4 : 0) + (bits ? 2 : 0) + (pad ? 1 : 0);
  switch (sel) {
    case 0: go(dz_kernel<false, false, false>); break;
    case 1: go(dz_kernel<false, false, true>); break;
    case 2: go(dz_kernel<false, true, false>); break;
    case 3: go(dz_kernel<false, true, true>); break;
    case 4: go(dz_kernel<true, false, false>); break;
    case 5: go(dz_kernel<true, false, true>); break;
    case 6: go(dz_kernel<true, true, false>); break;
    default: go(dz_kernel<true, true, true>); break;
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 6;
}

bool apply_merge_supported(int c, int max_parts) {
  uint32_t bytes = 0;
  switch (c) {
    case 16: bytes = merge_smem_bytes<16>(max_parts); break;
    case 32: bytes = merge_smem_bytes<32>(max_parts); break;
    case 64: bytes = merge_smem_bytes<64>(max_parts); break;
    case 128: bytes = merge_smem_bytes<128>(max_parts); break;
    default: return false;
  }
  return max_parts >= 1 && bytes <= 200u * 1024u;
}

int launch_apply(const ApplyArgs& a, bool bf16, int num_sms, cudaStream_t st) {
  // kApplyThreads (and so the grid stride) must be a multiple of the c/8 vectors of a pixel
  if (a.c % 8 != 0 || a.c > 256 || kApplyThreads % (a.c / 8) != 0) return 3;
  const long long nvec = a.total / 8;
  const bool mask = a.mask != nullptr;
  if (a.part) {
    // the statistics merge in the prologue: one block of kMergeThreads per SM
    if (!apply_merge_supported(a.c, a.nparts) || (reinterpret_cast<uintptr_t>(a.part) & 15) != 0) return 3;
    const long long want = (nvec + (long long)kApplyUnroll * kMergeThreads - 1) / ((long long)kApplyUnroll * kMergeThreads);
    const int grid = (int)std::max<long long>(1, std::min<long long>(want, num_sms));
    auto go = [&](auto kern, uint32_t smem) {
      // the attribute is set once per kernel: to the largest size any launch may ask for
      if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), 227 * 1024)) return 6;
      kern<<<grid, kMergeThreads, smem, st>>>(a);
      return cudaGetLastError() == cudaSuccess ? 0 : 6;
    };
    auto by_c = [&](auto bf16_c, auto mask_c) {
      constexpr bool B = decltype(bf16_c)::value, M = decltype(mask_c)::value;
      switch (a.c) {
        case 16: return go(bn_apply_merge_kernel<B, M, 16>, merge_smem_bytes<16>(a.nparts));
        case 32: return go(bn_apply_merge_kernel<B, M, 32>, merge_smem_bytes<32>(a.nparts));
        case 64: return go(bn_apply_merge_kernel<B, M, 64>, merge_smem_bytes<64>(a.nparts));
        default: return go(bn_apply_merge_kernel<B, M, 128>, merge_smem_bytes<128>(a.nparts));
      }
    };
    using T = std::true_type;
    using F = std::false_type;
    if (bf16) return mask ? by_c(T{}, T{}) : by_c(T{}, F{});
    return mask ? by_c(F{}, T{}) : by_c(F{}, F{});
  }
  auto go = [&](auto kern) {
    kern<<<stream_grid(kern, kApplyThreads, nvec / kApplyUnroll, num_sms), kApplyThreads, 0, st>>>(a);
  };
  if (bf16) {
    if (mask) go(bn_apply_relu_kernel<true, true>);
    else go(bn_apply_relu_kernel<true, false>);
  } else {
    if (mask) go(bn_apply_relu_kernel<false, true>);
    else go(bn_apply_relu_kernel<false, false>);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 6;
}

size_t bwd_reduce_partial_floats(int num_sms, int c) { return (size_t)num_sms * 2 * 2 * c; }

int launch_merge_finalize(const float* moments, int world, int c, const float* gamma, const float* beta,
                          float* running_mean, float* running_var, float momentum, float eps,
                          float* saved_mean, float* saved_inv_var, float* eq, cudaStream_t st) {
  bn_merge_finalize_kernel<<<(c + 127) / 128, 128, 0, st>>>(moments, world, c, gamma, beta, running_mean, running_var,
                                                            momentum, eps, saved_mean, saved_inv_var, eq);
  return cudaGetLastError() == cudaSuccess ? 0 : 6;
}

int launch_bwd_coef(const float* sums, int c, long long m_count, const float* gamma, const float* mean,
                    const float* inv_std, float* dgamma, float* dbeta, float* coef, cudaStream_t st) {
  bn_bwd_coef_kernel<<<(c + 127) / 128, 128, 0, st>>>(sums, c, 1.0 / (double)m_count, gamma, mean, inv_std, dgamma,
                                                      dbeta, coef);
  return cudaGetLastError() == cudaSuccess ? 0 : 6;
}

int launch_bwd_reduce(const BwdReduceArgs& a, bool bf16, int num_sms, cudaStream_t st) {
  // c <= 256: at most 32 channel groups, one per lane of a warp (the block partial relies on it)
  if (a.c % 8 != 0 || a.c > 256 || (kRedThreads % (a.c / 8)) != 0) return 3;
  const long long nvec = a.m_count * (a.c / 8);
  const bool bits = a.mask != nullptr;
  // the grid is at most the resident blocks (one wave) and the number of partials it leaves
  // is bounded by the workspace (bwd_reduce_partial_floats: two blocks per SM)
  BwdReduceArgs b = a;
  b.inv_m = 1.0 / (double)a.m_count;
  auto go = [&](auto kern) {
    const int grid = std::min(stream_grid(kern, kRedThreads, nvec / kRedUnroll, num_sms), 2 * num_sms);
    kern<<<grid, kRedThreads, 0, st>>>(b);
  };
  if (bf16) {
    if (bits) go(bn_bwd_reduce_kernel<true, true>);
    else go(bn_bwd_reduce_kernel<true, false>);
  } else {
    if (bits) go(bn_bwd_reduce_kernel<false, true>);
    else go(bn_bwd_reduce_kernel<false, false>);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 6;
}

}  // namespace cbr
