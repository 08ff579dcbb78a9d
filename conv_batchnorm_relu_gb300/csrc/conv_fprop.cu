// K1 + K2: implicit-GEMM convolution forward on tcgen05 tensor cores with the BatchNorm
// statistics generated in the epilogue ("conv_fprop + genstats", Tech-Renaissance CBR page,
// section 4.1), and the BN finalize ("bn_finalize", same page, section 4.2) run by the last
// CTA to finish.  The same kernel also serves the z recompute for backward and the folded
// inference form relu(conv(x, W_fold) + b_fold) (CBR page, sections 2 and 6).
//
// GEMM view (TileLang Conv2D page, basic convolution section): M = output pixels,
// N = Cout, K = R*S*Cin.  Design for sm_103a:
//   * persistent grid, one CTA per SM, 7 warps:
//       warp 0  TMA producer for the input halo (4D tiled load, zero fill = conv padding)
//       warp 1  TMEM owner + single-thread tcgen05.mma issuer
//       warp 2  TMA producer for the filter slabs (resident for the whole kernel when they fit)
//       warps 3-6  epilogue: TMEM -> registers -> fp16/bf16 staging -> stats + coalesced store
//   * the input halo of a unit of U*128 padded-linear output rows is loaded ONCE; the R*S
//     taps are row-shifted smem descriptors into it (see HaloGeom), so the activation is not
//     re-read per tap;
//   * fp32 accumulators live in TMEM, double-buffered so the epilogue of one unit overlaps
//     the MMAs of the next;
//   * per-channel sum / sum of squares are reduced from the staged tile per CTA, then across
//     CTAs in a fixed order in fp64 by the last CTA (deterministic).
#include <algorithm>

#include "cbr_internal.h"
#include "common.cuh"

namespace cbr {
namespace {

constexpr int kThreads = 224;
constexpr int kEpiThreads = 128;
constexpr int kStreamStages = 2;  // weight ring depth when the filter is not resident

constexpr int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

template <int NCH, int COUT, int U, bool WRES>
struct FpropCfg {
  static constexpr int kPitch = COUT * 2;            // bytes per staged output row
  static constexpr int kChunks = kPitch / 16;        // 16-byte chunks per output row
  static constexpr int kWSlab = COUT * 128;          // one (channel chunk, tap) filter slab
  static constexpr int kTmemCols = pow2_at_least(2 * U * COUT);
  static constexpr int kPairs = COUT / 2;
};

struct SmemLayout {
  uint32_t halo_stride, off_w, off_stage, off_bar, total;
  int nsw;
};

__host__ __device__ inline SmemLayout fprop_layout(const HaloGeom& g, int nch, int cout, bool wres) {
  SmemLayout L;
  const uint32_t halo = (uint32_t)g.hr * g.wp * 128;
  L.halo_stride = (halo + 1023u) & ~1023u;
  L.nsw = wres ? nch * g.r * g.s : kStreamStages;
  L.off_w = 2 * L.halo_stride;
  L.off_stage = L.off_w + (uint32_t)L.nsw * cout * 128;
  const uint32_t stage = 128u * cout * 2;
  L.off_bar = (L.off_stage + stage + 15u) & ~15u;
  const uint32_t nbar = 8 + 2 * L.nsw + 1;
  L.total = L.off_bar + nbar * 8 + 16;
  return L;
}

__device__ __forceinline__ bool is_aborted(volatile int* flag) { return *flag != 0; }

__device__ __forceinline__ void set_abort(volatile int* flag, uint32_t* err, uint32_t bits) {
  *flag = 1;
  report_error(err, bits);
}

template <int NCH, int COUT, int U, bool WRES, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    conv_fprop_genstats_kernel(const __grid_constant__ CUtensorMap map_x,
                               const __grid_constant__ CUtensorMap map_w, const FpropArgs a) {
  using Cfg = FpropCfg<NCH, COUT, U, WRES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const HaloGeom& g = a.g;
  const SmemLayout L = fprop_layout(g, NCH, COUT, WRES);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t halo_addr = sbase;
  const uint32_t w_addr = sbase + L.off_w;
  const uint32_t stage_addr = sbase + L.off_stage;
  const uint32_t bar0 = sbase + L.off_bar;
  // barrier map (8 bytes each)
  const uint32_t bar_halo_full = bar0;              // [2]
  const uint32_t bar_halo_empty = bar0 + 16;        // [2]
  const uint32_t bar_acc_full = bar0 + 32;          // [2]
  const uint32_t bar_acc_empty = bar0 + 48;         // [2]
  const uint32_t bar_w_full = bar0 + 64;            // [nsw]
  const uint32_t bar_w_empty = bar_w_full + 8 * L.nsw;  // [nsw]
  const uint32_t bar_drain = bar_w_empty + 8 * L.nsw;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.off_bar + (8 + 2 * L.nsw + 1) * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile uint32_t* ticket_slot = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rs = g.r * g.s;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_halo_full + 8 * i, 1);
      mbar_init(bar_halo_empty + 8 * i, 1);
      mbar_init(bar_acc_full + 8 * i, 1);
      mbar_init(bar_acc_empty + 8 * i, kEpiThreads);
    }
    for (int i = 0; i < L.nsw; ++i) {
      mbar_init(bar_w_full + 8 * i, 1);
      mbar_init(bar_w_empty + 8 * i, 1);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ halo producer
    if (lane == 0) {
      prefetch_tensormap(&map_x);
      const uint32_t tx = (uint32_t)g.hr * g.wp * 128;
      uint32_t it = 0;
      for (int u = blockIdx.x; u < g.total_units && !is_aborted(abort_flag); u += gridDim.x) {
        const int n = u / g.upi;
        const int m0 = (u - n * g.upi) * g.um;
        const int h_lo = m0 / g.wp - g.pad;
        for (int ch = 0; ch < NCH; ++ch, ++it) {
          const uint32_t s = it & 1, ph = (it >> 1) & 1;
          if (!mbar_wait(bar_halo_empty + 8 * s, ph ^ 1)) {
            set_abort(abort_flag, a.err, kErrWaitHalo);
            break;
          }
          mbar_arrive_expect_tx(bar_halo_full + 8 * s, tx);
          tma_load_4d(halo_addr + s * L.halo_stride, &map_x, ch * 64, -g.pad, h_lo, n,
                      bar_halo_full + 8 * s);
        }
      }
      // never leave the CTA with a copy in flight
      for (uint32_t k = (it > 2 ? it - 2 : 0); k < it; ++k)
        mbar_wait(bar_halo_full + 8 * (k & 1), (k >> 1) & 1);
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ filter producer
    if (lane == 0) {
      prefetch_tensormap(&map_w);
      if (WRES) {
        for (int i = 0; i < NCH * rs; ++i) {
          const int ch = i / rs, tap = i - ch * rs;
          mbar_arrive_expect_tx(bar_w_full + 8 * i, Cfg::kWSlab);
          tma_load_3d(w_addr + i * Cfg::kWSlab, &map_w, ch * 64, tap, 0, bar_w_full + 8 * i);
        }
        for (int i = 0; i < NCH * rs; ++i) mbar_wait(bar_w_full + 8 * i, 0);
      } else {
        uint32_t it = 0;
        for (int u = blockIdx.x; u < g.total_units && !is_aborted(abort_flag); u += gridDim.x) {
          for (int ch = 0; ch < NCH; ++ch)
            for (int tap = 0; tap < rs; ++tap, ++it) {
              const uint32_t s = it % kStreamStages, ph = (it / kStreamStages) & 1;
              if (!mbar_wait(bar_w_empty + 8 * s, ph ^ 1)) {
                set_abort(abort_flag, a.err, kErrWaitWeights);
                ch = NCH;
                break;
              }
              mbar_arrive_expect_tx(bar_w_full + 8 * s, Cfg::kWSlab);
              tma_load_3d(w_addr + s * Cfg::kWSlab, &map_w, ch * 64, tap, 0, bar_w_full + 8 * s);
            }
        }
        for (uint32_t k = (it > kStreamStages ? it - kStreamStages : 0); k < it; ++k)
          mbar_wait(bar_w_full + 8 * (k % kStreamStages), (k / kStreamStages) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = make_idesc_f16(128, COUT, BF16, false, false);
      uint32_t hit = 0, wit = 0, ait = 0;
      bool first = true;
      const int rows_img = g.p * g.wp;
      for (int u = blockIdx.x; u < g.total_units && !is_aborted(abort_flag); u += gridDim.x) {
        const int n = u / g.upi;
        const int m0 = (u - n * g.upi) * g.um;
        const int off = m0 - (m0 / g.wp) * g.wp;
        const int ntiles = min(U, (rows_img - m0 + 127) / 128);
        const uint32_t as = ait & 1, aph = (ait >> 1) & 1;
        if (!mbar_wait(bar_acc_empty + 8 * as, aph ^ 1)) {
          set_abort(abort_flag, a.err, kErrWaitAccum);
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem_base + as * (U * COUT);
        bool bad = false;
        for (int ch = 0; ch < NCH && !bad; ++ch, ++hit) {
          const uint32_t hs = hit & 1, hph = (hit >> 1) & 1;
          if (!mbar_wait(bar_halo_full + 8 * hs, hph)) {
            set_abort(abort_flag, a.err, kErrWaitHalo);
            bad = true;
            break;
          }
          tc_fence_after();
          const uint32_t hbase = halo_addr + hs * L.halo_stride;
          for (int tap = 0; tap < rs; ++tap) {
            const int r = tap / g.s, sx = tap - r * g.s;
            uint32_t wslab, ws = 0;
            if (WRES) {
              const int i = ch * rs + tap;
              if (first && !mbar_wait(bar_w_full + 8 * i, 0)) {
                set_abort(abort_flag, a.err, kErrWaitWeights);
                bad = true;
                break;
              }
              wslab = w_addr + i * Cfg::kWSlab;
            } else {
              ws = wit % kStreamStages;
              if (!mbar_wait(bar_w_full + 8 * ws, (wit / kStreamStages) & 1)) {
                set_abort(abort_flag, a.err, kErrWaitWeights);
                bad = true;
                break;
              }
              wslab = w_addr + ws * Cfg::kWSlab;
            }
            tc_fence_after();
            const uint32_t a_row0 = hbase + (uint32_t)(off + r * g.wp + sx) * 128u;
            for (int t = 0; t < ntiles; ++t) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t ad = make_sw128_desc(a_row0 + t * 128 * 128 + kk * 32, 16, 1024, 0);
                const uint64_t bd = make_sw128_desc(wslab + kk * 32, 16, 1024, 0);
                mma_f16_ss(d0 + t * COUT, ad, bd, idesc, (ch | tap | kk) != 0);
              }
            }
            if (!WRES) {
              mma_commit(bar_w_empty + 8 * ws);
              ++wit;
            }
          }
          mma_commit(bar_halo_empty + 8 * hs);
        }
        if (bad) break;
        mma_commit(bar_acc_full + 8 * as);
        ++ait;
        first = false;
      }
      // drain: every MMA this thread issued has completed before TMEM is released
      mma_commit(bar_drain);
      mbar_wait(bar_drain, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 3..6)
    const int quad = warp & 3;             // TMEM lanes 32*quad .. 32*quad+31
    const int e = quad * 32 + lane;        // row of the M tile this thread owns
    const int et = threadIdx.x - 96;       // 0..127, rank among epilogue threads
    constexpr int kPL = (Cfg::kPairs + 31) / 32;  // channel pairs per lane for the stats
    float s1[2 * kPL], s2[2 * kPL];
#pragma unroll
    for (int i = 0; i < 2 * kPL; ++i) s1[i] = s2[i] = 0.f;
    const int rows_img = g.p * g.wp;
    const bool stats = a.mode == kFpropStats;
    const bool bias_relu = a.mode == kFpropBiasRelu;
    uint32_t ait = 0;
    for (int u = blockIdx.x; u < g.total_units && !is_aborted(abort_flag); u += gridDim.x) {
      const int n = u / g.upi;
      const int m0 = (u - n * g.upi) * g.um;
      const int ntiles = min(U, (rows_img - m0 + 127) / 128);
      const uint32_t as = ait & 1, aph = (ait >> 1) & 1;
      bool ok = mbar_wait(bar_acc_full + 8 * as, aph);
      if (!ok) set_abort(abort_flag, a.err, kErrWaitMma);
      // uniform decision across the 128 epilogue threads (they share named barriers below)
      if (!named_bar_and(2, kEpiThreads, ok && !is_aborted(abort_flag))) break;
      tc_fence_after();
      uint32_t pk[U][COUT / 2];
#pragma unroll
      for (int t = 0; t < U; ++t) {
        if (t < ntiles) {
#pragma unroll
          for (int c16 = 0; c16 < COUT / 16; ++c16) {
            uint32_t r[16];
            tmem_ld16(tmem_base + ((uint32_t)(quad * 32) << 16) + as * (U * COUT) + t * COUT + c16 * 16, r);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              float lo = __uint_as_float(r[2 * i]), hi = __uint_as_float(r[2 * i + 1]);
              if (bias_relu) {
                lo = fmaxf(lo + __ldg(a.bias + c16 * 16 + 2 * i), 0.f);
                hi = fmaxf(hi + __ldg(a.bias + c16 * 16 + 2 * i + 1), 0.f);
              }
              pk[t][c16 * 8 + i] = pack2<BF16>(lo, hi);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(bar_acc_empty + 8 * as);
#pragma unroll
      for (int t = 0; t < U; ++t) {
        if (t >= ntiles) break;
        const int mt = m0 + t * 128;
        {
          const int m = mt + e;
          const int p = m / g.wp, q = m - p * g.wp;
          const bool valid = (p < g.p) && (q < g.q);
#pragma unroll
          for (int c = 0; c < Cfg::kChunks; ++c) {
            uint4 v = valid ? make_uint4(pk[t][4 * c], pk[t][4 * c + 1], pk[t][4 * c + 2], pk[t][4 * c + 3])
                            : make_uint4(0, 0, 0, 0);
            const uint32_t o = (Cfg::kPitch >= 128) ? swz_off(e, c, Cfg::kPitch) : (uint32_t)(e * Cfg::kPitch + c * 16);
            st_shared_v4(stage_addr + o, v);
          }
        }
        named_bar_sync(1, kEpiThreads);
        if (stats) {
          for (int row = quad * 32; row < quad * 32 + 32; ++row) {
#pragma unroll
            for (int k = 0; k < kPL; ++k) {
              const int j = lane + 32 * k;  // channel pair index
              if (j < Cfg::kPairs) {
                const int c = 2 * j;
                const uint32_t o = ((Cfg::kPitch >= 128) ? swz_off(row, c >> 3, Cfg::kPitch)
                                                         : (uint32_t)(row * Cfg::kPitch + (c >> 3) * 16)) +
                                   (c & 7) * 2;
                const float2 v = unpack2<BF16>(ld_shared_b32(stage_addr + o));
                s1[2 * k] += v.x;
                s1[2 * k + 1] += v.y;
                s2[2 * k] = fmaf(v.x, v.x, s2[2 * k]);
                s2[2 * k + 1] = fmaf(v.y, v.y, s2[2 * k + 1]);
              }
            }
          }
        }
        // coalesced copy-out of the valid rows
        uint8_t* zbase = static_cast<uint8_t*>(a.z);
        for (int i = et; i < 128 * Cfg::kChunks; i += kEpiThreads) {
          const int row = i / Cfg::kChunks, c = i - row * Cfg::kChunks;
          const int m = mt + row;
          const int p = m / g.wp, q = m - p * g.wp;
          if (p < g.p && q < g.q) {
            const uint32_t o = (Cfg::kPitch >= 128) ? swz_off(row, c, Cfg::kPitch) : (uint32_t)(row * Cfg::kPitch + c * 16);
            const size_t gi = ((size_t)n * g.p + p) * g.q + q;
            st_global_v4(zbase + gi * Cfg::kPitch + c * 16, ld_shared_v4(stage_addr + o));
          }
        }
        named_bar_sync(1, kEpiThreads);
      }
      ++ait;
    }
    if (stats) {
      // per-warp partials -> smem (fixed order combine below)
      float* red = reinterpret_cast<float*>(smem + L.off_stage);
      // stage buffer is free: all copy-outs finished behind the last named barrier
#pragma unroll
      for (int k = 0; k < kPL; ++k) {
        const int j = lane + 32 * k;
        if (j < Cfg::kPairs) {
          red[(quad * 2 + 0) * COUT + 2 * j] = s1[2 * k];
          red[(quad * 2 + 0) * COUT + 2 * j + 1] = s1[2 * k + 1];
          red[(quad * 2 + 1) * COUT + 2 * j] = s2[2 * k];
          red[(quad * 2 + 1) * COUT + 2 * j + 1] = s2[2 * k + 1];
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();

  if (a.mode == kFpropStats) {
    const float* red = reinterpret_cast<const float*>(smem + L.off_stage);
    for (int i = threadIdx.x; i < 2 * COUT; i += kThreads) {
      const int st = i / COUT, c = i - st * COUT;
      float v = red[(0 * 2 + st) * COUT + c];
      v += red[(1 * 2 + st) * COUT + c];
      v += red[(2 * 2 + st) * COUT + c];
      v += red[(3 * 2 + st) * COUT + c];
      a.part[(size_t)blockIdx.x * 2 * COUT + i] = v;
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) *ticket_slot = atomicInc(a.ticket, gridDim.x - 1);
    __syncthreads();
    if (*ticket_slot == gridDim.x - 1 && !is_aborted(abort_flag)) {
      // ---------------------------------------------------- K2: bn_finalize (last CTA)
      __threadfence();
      double* dred = reinterpret_cast<double*>(smem + L.off_stage);  // [7][2*COUT]
      double* fin = dred + 7 * 2 * COUT;                              // [2*COUT]
      constexpr int kV4 = (2 * COUT) / 4;
      for (int c4 = lane; c4 < kV4; c4 += 32) {
        double acc0 = 0, acc1 = 0, acc2 = 0, acc3 = 0;
        for (int b = warp; b < (int)gridDim.x; b += kThreads / 32) {
          const float4 v = __ldcg(reinterpret_cast<const float4*>(a.part + (size_t)b * 2 * COUT) + c4);
          acc0 += v.x;
          acc1 += v.y;
          acc2 += v.z;
          acc3 += v.w;
        }
        dred[warp * 2 * COUT + 4 * c4 + 0] = acc0;
        dred[warp * 2 * COUT + 4 * c4 + 1] = acc1;
        dred[warp * 2 * COUT + 4 * c4 + 2] = acc2;
        dred[warp * 2 * COUT + 4 * c4 + 3] = acc3;
      }
      __syncthreads();
      for (int i = threadIdx.x; i < 2 * COUT; i += kThreads) {
        double t = 0;
        for (int w = 0; w < kThreads / 32; ++w) t += dred[w * 2 * COUT + i];
        fin[i] = t;
      }
      __syncthreads();
      for (int c = threadIdx.x; c < COUT; c += kThreads) {
        const double M = (double)a.m_count;
        const double mean = fin[c] / M;
        double var = fin[COUT + c] / M - mean * mean;
        var = var > 0.0 ? var : 0.0;
        const double inv = 1.0 / sqrt(var + (double)a.eps);
        const double gm = a.gamma[c];
        a.saved_mean[c] = (float)mean;
        a.saved_inv_var[c] = (float)inv;
        a.eq[c] = (float)(gm * inv);
        a.eq[COUT + c] = (float)((double)a.beta[c] - gm * mean * inv);
        const double mom = a.momentum;
        a.running_mean[c] = (float)((1.0 - mom) * a.running_mean[c] + mom * mean);
        a.running_var[c] = (float)((1.0 - mom) * a.running_var[c] + mom * var * M / (M - 1.0));
      }
    }
  }

  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

template <int NCH, int COUT, int U, bool WRES, bool BF16>
int launch_inst(const FpropArgs& a, const CUtensorMap& mx, const CUtensorMap& mw, int grid,
                cudaStream_t st) {
  auto kern = conv_fprop_genstats_kernel<NCH, COUT, U, WRES, BF16>;
  const SmemLayout L = fprop_layout(a.g, NCH, COUT, WRES);
  const uint32_t smem = L.total + 1024;
  if (smem > 227 * 1024) return 3;  // CBR_ERR_UNSUPPORTED
  static int configured = 0;
  if (configured < (int)smem) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) != cudaSuccess)
      return 6;
    configured = 227 * 1024;
  }
  kern<<<grid, kThreads, smem, st>>>(mx, mw, a);
  return cudaGetLastError() == cudaSuccess ? 0 : 6;
}

}  // namespace

size_t fprop_partial_floats(int num_sms, int c_out) { return (size_t)num_sms * 2 * c_out; }

int launch_fprop(const FpropArgs& a_in, int c_in, int c_out, bool bf16, const void* x,
                 const void* w, int num_sms, cudaStream_t st) {
  FpropArgs a = a_in;
  HaloGeom& g = a.g;
  const int nch = c_in <= 64 ? 1 : (c_in <= 128 ? 2 : 0);
  if (nch == 0) return 3;
  int U = c_out <= 64 ? 2 : 1;
  g.um = U * 128;
  g.wp = g.w + 2 * g.pad;
  g.p = g.h + 2 * g.pad - g.r + 1;
  g.q = g.w + 2 * g.pad - g.s + 1;
  if (g.p <= 0 || g.q <= 0 || g.wp > 256) return 3;
  g.hr = (g.wp - 1 + g.um - 1 + (g.r - 1) * g.wp + g.s - 1) / g.wp + 1;
  if (g.hr > 256) return 3;
  g.upi = (g.p * g.wp + g.um - 1) / g.um;
  g.total_units = g.n_img * g.upi;
  const bool wres_fits = fprop_layout(g, nch, c_out, true).total + 1024 <= 227 * 1024;

  const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap mx, mw;
  {
    const uint64_t dims[4] = {(uint64_t)c_in, (uint64_t)g.w, (uint64_t)g.h, (uint64_t)g.n_img};
    const uint64_t strides[3] = {(uint64_t)c_in * 2, (uint64_t)g.w * c_in * 2, (uint64_t)g.h * g.w * c_in * 2};
    const uint32_t box[4] = {64, (uint32_t)g.wp, (uint32_t)g.hr, 1};
    if (!encode_tiled(&mx, dt, 4, x, dims, strides, box)) return 6;
  }
  {
    const uint64_t dims[3] = {(uint64_t)c_in, (uint64_t)(g.r * g.s), (uint64_t)c_out};
    const uint64_t strides[2] = {(uint64_t)c_in * 2, (uint64_t)g.r * g.s * c_in * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)c_out};
    if (!encode_tiled(&mw, dt, 3, w, dims, strides, box)) return 6;
  }
  const int grid = std::min(g.total_units, num_sms);

#define CBR_FPROP_CASE(NCH_, COUT_, U_, WRES_)                                          \
  if (nch == NCH_ && c_out == COUT_ && U == U_ && (WRES_ == wres_fits)) {                \
    return bf16 ? launch_inst<NCH_, COUT_, U_, WRES_, true>(a, mx, mw, grid, st)         \
                : launch_inst<NCH_, COUT_, U_, WRES_, false>(a, mx, mw, grid, st);       \
  }
  CBR_FPROP_CASE(1, 16, 2, true)
  CBR_FPROP_CASE(1, 32, 2, true)
  CBR_FPROP_CASE(1, 64, 2, true)
  CBR_FPROP_CASE(1, 64, 2, false)
  CBR_FPROP_CASE(1, 128, 1, false)
  CBR_FPROP_CASE(1, 128, 1, true)
  CBR_FPROP_CASE(2, 128, 1, false)
  CBR_FPROP_CASE(2, 64, 2, false)
#undef CBR_FPROP_CASE
  return 3;
}

}  // namespace cbr
