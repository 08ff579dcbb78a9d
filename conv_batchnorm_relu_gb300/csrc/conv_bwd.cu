// B3: weight gradient (WGrad) of the convolution (Tech-Renaissance CBR page, section 5.2) over
// dz = gamma*inv_std*(g - dbeta/M - xhat*dgamma/M), g = dy*mask (section 5.1; BatchNorm CUDA
// page, section 3.1), for the layers the fused backward kernel (conv_bwd_fused.cu) does not
// take: dz is materialised once by the dz pass (bn_kernels.cu) in the padded-linear row layout
// and loaded here by TMA.
//
// DGrad (B2, conv_dgrad.cu) is the stride-1 convolution of dz with the tap-flipped filter and
// padding R-1-pad on the shared halo-conv template, with the filter read MN-major.
//
// WGrad: dW[k][r][s][c] = sum over pixels of dz[pixel][k] * x[pixel shifted by (r,s)][c].  The
// reduction dimension is the pixel, so both operands are MN-major pixel-row tiles: A is the
// TMA-loaded input halo, in which each tap is a row-shifted view; B is the dz tile of the unit.
// Two taps share one M = 128 MMA (two 64-channel atoms at different row shifts, addressed by
// the descriptor's leading-dimension offset).  Each CTA accumulates its pixels in TMEM for
// the whole kernel, writes one fp32 partial, and a second kernel sums the partials in a fixed
// order (deterministic).
#include <algorithm>
#include <type_traits>

#include "halo_conv.cuh"

namespace cbr {
namespace {

constexpr int kWgThreads = 192;  // warp 0: x and dz TMA; warp 1: MMA; warps 2-5: epilogue

struct WgKArgs {
  HaloGeom g;
  WgPlan plan;
  float* part;
  uint32_t* err;
};

}  // namespace

// Tap pairs (0,1), (2,3), ...; an odd last tap is paired with itself (its second half is
// discarded).  Groups are split into contiguous subsets so that one CTA's accumulators
// (groups x NOUT fp32 columns) fit the 512 TMEM columns; every 64-channel input chunk is a
// separate split as well.
bool make_wg_plan(WgPlan& P, int taps, int c_in, int nout) {
  P = WgPlan{};
  const int ngroups = (taps + 1) / 2;
  if (ngroups > kWgMaxGroups) return false;
  for (int gi = 0; gi < ngroups; ++gi) {
    P.ta[gi] = 2 * gi;
    P.tb[gi] = std::min(2 * gi + 1, taps - 1);
  }
  const int gcap = std::min(512 / nout, 16);  // TMEM columns; at most 16 groups per CTA
  const int nsub = (ngroups + gcap - 1) / gcap;
  const int nchunk = (c_in + 63) / 64;
  if (nsub * nchunk > kWgMaxSplits) return false;
  P.ngroups = ngroups;
  P.nsplit = nsub * nchunk;
  P.gmax = 0;
  for (int ch = 0; ch < nchunk; ++ch)
    for (int sb = 0; sb < nsub; ++sb) {
      const int s = ch * nsub + sb;
      const int g0 = ngroups * sb / nsub, g1 = ngroups * (sb + 1) / nsub;
      P.split_chunk[s] = ch;
      P.split_g0[s] = g0;
      P.split_ng[s] = g1 - g0;
      P.gmax = std::max(P.gmax, g1 - g0);
    }
  return true;
}

namespace {

struct WgLayout {
  uint32_t halo_stride, dz_sub, dz_stride, off_dz, off_bar, total;
};

// The dz tile of a unit is its um padded-linear rows, 64 channels per sub-tile, loaded by TMA
// from a dz materialised in the same padded-linear row layout (the rows past the last image
// row read as zero).
__host__ __device__ inline WgLayout wg_layout(const HaloGeom& g, int nout) {
  WgLayout L;
  L.halo_stride = (((uint32_t)g.hr * g.wp * 128) + 1023u) & ~1023u;
  const int nkc = nout > 64 ? nout / 64 : 1;
  L.dz_sub = (uint32_t)g.um * 128;
  L.dz_stride = (uint32_t)nkc * L.dz_sub;
  L.off_dz = 2 * L.halo_stride;
  L.off_bar = L.off_dz + 2 * L.dz_stride;
  L.total = L.off_bar + 12 * 8 + 16;
  return L;
}

// Warp 0 loads both operands (the x halo and the dz tile) by TMA; warp 1 issues the MMAs;
// warps 2-5 write the per-CTA partial at the end.
template <int NOUT, bool BF16>
__global__ void __launch_bounds__(kWgThreads, 1)
    wgrad_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_dz,
                 const WgKArgs a) {
  constexpr int kNkc = NOUT > 64 ? NOUT / 64 : 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const HaloGeom& g = a.g;
  const WgPlan& P = a.plan;
  const WgLayout L = wg_layout(g, NOUT);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t x_addr = sbase, dz_addr = sbase + L.off_dz;
  const uint32_t bar0 = sbase + L.off_bar;
  const uint32_t bar_x_full = bar0, bar_x_empty = bar0 + 16;
  const uint32_t bar_acc_full = bar0 + 64, bar_drain = bar0 + 72;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.off_bar + 12 * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int split = blockIdx.x % P.nsplit;
  const int ustart = blockIdx.x / P.nsplit;
  const int ustride = gridDim.x / P.nsplit;
  const int chunk = P.split_chunk[split];
  const int g0 = P.split_g0[split], ng = P.split_ng[split];
  const int tmem_cols = hc::pow2_at_least(P.gmax * NOUT);

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_x_full + 8 * i, 1);
      mbar_init(bar_x_empty + 8 * i, 1);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tensormap(&map_x);
      prefetch_tensormap(&map_dz);
      const uint32_t tx = (uint32_t)g.hr * g.wp * 128 + (uint32_t)kNkc * L.dz_sub;
      uint32_t it = 0;
      for (int u = ustart; u < g.total_units && !hc::is_aborted(abort_flag); u += ustride, ++it) {
        const int n = u / g.upi;
        const int m0 = (u - n * g.upi) * g.um;
        const uint32_t s = it & 1, ph = (it >> 1) & 1;
        if (!mbar_wait_backoff(bar_x_empty + 8 * s, ph ^ 1, 128)) {
          hc::set_abort(abort_flag, a.err, kErrWaitHalo);
          break;
        }
        // the x and dz stages are released together by the same MMA commit
        mbar_arrive_expect_tx(bar_x_full + 8 * s, tx);
        for (int r0 = 0; r0 < g.hr; r0 += g.box_rows)
          tma_load_4d(x_addr + s * L.halo_stride + (uint32_t)r0 * g.wp * 128, &map_x, chunk * 64, -g.pad,
                      m0 / g.wp - g.pad + r0, n, bar_x_full + 8 * s);
        for (int kc = 0; kc < kNkc; ++kc)
            tma_load_3d(dz_addr + s * L.dz_stride + kc * L.dz_sub, &map_dz, kc * 64, m0, n,
                        bar_x_full + 8 * s);
      }
      for (uint32_t k = (it > 2 ? it - 2 : 0); k < it; ++k)
        mbar_wait(bar_x_full + 8 * (k & 1), (k >> 1) & 1);
    }
  } else if (warp == 1) {
    // The whole warp runs the issue loop (warp-uniform descriptor arithmetic) and one elected
    // lane issues each MMA and commit; control-flow decisions are voted across the warp.
    {
      const uint32_t idesc = make_idesc_f16(128, NOUT, BF16, true, true);
      // per-group A descriptor with a zero start address: LBO = the two taps' row distance.
      // Kept in registers (fully unrolled over the compile-time maximum group count).
      constexpr int kG = (512 / NOUT) < 16 ? (512 / NOUT) : 16;
      uint64_t a_grp[kG];
#pragma unroll
      for (int gl = 0; gl < kG; ++gl) {
        a_grp[gl] = 0;
        if (gl < ng) {
          const int ta = P.ta[g0 + gl], tb = P.tb[g0 + gl];
          const int sha = (ta / g.s) * g.wp + ta % g.s;
          const int shb = (tb / g.s) * g.wp + tb % g.s;
          a_grp[gl] = make_sw128_desc((uint32_t)sha * 128u, (uint32_t)(shb - sha) * 128u, 1024, 0);
        }
      }
      uint32_t it = 0;
      bool first = true;
      for (int u = ustart; u < g.total_units && !__any_sync(0xffffffffu, hc::is_aborted(abort_flag));
           u += ustride, ++it) {
        const int n = u / g.upi;
        const int m0 = (u - n * g.upi) * g.um;
        const int off = m0 - (m0 / g.wp) * g.wp;
        const uint32_t s = it & 1, ph = (it >> 1) & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(bar_x_full + 8 * s, ph))) {
          hc::set_abort(abort_flag, a.err, kErrWaitOperand);
          break;
        }
        tc_fence_after();
        const uint32_t xh = x_addr + s * L.halo_stride;
        const uint32_t dzs = dz_addr + s * L.dz_stride;
        const uint64_t a_unit = (uint64_t)((xh + (uint32_t)off * 128u) >> 4);
        uint64_t bd = make_sw128_desc(dzs, L.dz_sub, 1024, 0);
        // The group count is fixed per CTA: dispatch once per unit to a loop with a
        // compile-time trip count (a runtime guard around each MMA slows issue ~2x).
        auto issue = [&](auto ng_c) {
          constexpr int NG = decltype(ng_c)::value;
          if constexpr (NG <= kG) {
            uint32_t acc = first ? 0u : 1u;
            // 16-pixel K steps of a unit (um = U * 128 rows, U fixed by NOUT): a compile-time
            // trip count, like the group count
            constexpr int KK = (NOUT <= 64 ? 2 : 1) * 8;
#pragma unroll 4
            for (int kk = 0; kk < KK; ++kk) {
              const uint64_t ak = a_unit + (uint64_t)kk * 128;  // 16 pixel rows further
#pragma unroll
              for (int gl = 0; gl < NG; ++gl) mma_f16_ss_warp(tmem_base + gl * NOUT, a_grp[gl] + ak, bd, idesc, acc);
              bd += 128;
              acc = 1u;
            }
          }
        };
        switch (ng) {
#define CBR_WG_NG(k) case k: issue(std::integral_constant<int, k>{}); break;
          CBR_WG_NG(1) CBR_WG_NG(2) CBR_WG_NG(3) CBR_WG_NG(4) CBR_WG_NG(5) CBR_WG_NG(6)
          CBR_WG_NG(7) CBR_WG_NG(8) CBR_WG_NG(9) CBR_WG_NG(10) CBR_WG_NG(11) CBR_WG_NG(12)
          CBR_WG_NG(13) CBR_WG_NG(14) CBR_WG_NG(15) CBR_WG_NG(16)
#undef CBR_WG_NG
          default: break;
        }
        mma_commit_warp(bar_x_empty + 8 * s);
        first = false;
      }
      mma_commit_warp(bar_acc_full);
      mma_commit_warp(bar_drain);
      mbar_wait(bar_drain, 0);
    }
  } else {
    // warps 2..5: the epilogue
    const bool ok = mbar_wait_backoff(bar_acc_full, 0, 1024);
    if (!ok) hc::set_abort(abort_flag, a.err, kErrWaitMma);
    tc_fence_after();
    if (ok) {
      const int quad = warp & 3;
      const int e = quad * 32 + lane;  // accumulator row = (tap half, channel)
      for (int gl = 0; gl < ng; ++gl) {
#pragma unroll
        for (int c16 = 0; c16 < NOUT / 16; ++c16) {
          uint32_t r[16];
          tmem_ld16(tmem_base + ((uint32_t)(quad * 32) << 16) + gl * NOUT + c16 * 16, r);
          tmem_ld_wait();
          // partial layout [cta][group][c16][v][row][4]: a warp's store is 512 contiguous bytes
          float4* dst = reinterpret_cast<float4*>(a.part) +
                        (((size_t)blockIdx.x * P.gmax + gl) * (NOUT / 16) + c16) * 512 + e;
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v * 128] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                       __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

// dW = sum over the CTAs of each split of their partials, in a fixed order.  A block owns 16
// consecutive float4 of the per-CTA partial (the same span in every CTA, so the loads are
// coalesced) and 16 slices of the split's CTA list: slice sl sums CTAs sl, sl+16, ... in fp32
// with all of its (at most 16) loads in flight, and the slices are combined by a fixed pairwise
// tree in shared memory.  Each summed element is then written to its dW[k][tap][c] position.
// 256-thread blocks keep the grid within one wave of resident blocks at 128 channels (a
// 512-thread shape ran a tail wave: 20.5 against 16.4 us there, the same at 64 channels).
constexpr int kRedSpan = 16;                         // float4 columns per block
constexpr int kRedSlices = 16;                       // CTA slices per column
constexpr int kRedThreads = kRedSpan * kRedSlices;   // 256
constexpr int kRedLd = 16;                           // CTAs per slice in flight (grids up to 256)
static_assert(kRedSlices * kRedLd >= kMaxCtas, "one round of loads covers every CTA's partial");

template <int NOUT>
__global__ void __launch_bounds__(kRedThreads)
    wgrad_reduce_kernel(const float* __restrict__ part, float* __restrict__ dw, const WgPlan P,
                        int grid, int cin, int taps) {
  __shared__ float4 red[kRedSlices][kRedSpan];
  constexpr int kC16 = NOUT / 16;
  const size_t per_cta = (size_t)P.gmax * kC16 * 512;  // float4 per CTA partial
  const int blocks_per_split = (int)((per_cta + kRedSpan - 1) / kRedSpan);
  const int split = blockIdx.x / blocks_per_split;
  const int col = threadIdx.x % kRedSpan;
  const size_t f4 = (size_t)(blockIdx.x % blocks_per_split) * kRedSpan + col;
  const int sl = threadIdx.x / kRedSpan;
  const int nb = (grid - split + P.nsplit - 1) / P.nsplit;  // CTAs of this split
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (f4 < per_cta) {
    const float4* base = reinterpret_cast<const float4*>(part) + f4;
    for (int t0 = sl; t0 < nb; t0 += kRedLd * kRedSlices) {
      float4 v[kRedLd];
#pragma unroll
      for (int u = 0; u < kRedLd; ++u) {
        const int t = t0 + u * kRedSlices;
        v[u] = t < nb ? __ldg(base + (size_t)(split + t * P.nsplit) * per_cta) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kRedLd; ++u) {
        acc.x += v[u].x;
        acc.y += v[u].y;
        acc.z += v[u].z;
        acc.w += v[u].w;
      }
    }
  }
  red[sl][col] = acc;
#pragma unroll
  for (int w = kRedSlices / 2; w >= 1; w >>= 1) {
    __syncthreads();
    if (sl < w) {
      const float4 b = red[sl + w][col];
      float4& a = red[sl][col];
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
  }
  if (sl != 0 || f4 >= per_cta) return;
  const float4 v = red[0][col];
  const float t4[4] = {v.x, v.y, v.z, v.w};
  // f4 -> (group, c16, v, row): see the partial layout in wgrad_kernel
  const int row = (int)(f4 % 128);
  const int vq = (int)((f4 / 128) % 4);
  const int c16 = (int)((f4 / 512) % kC16);
  const int gl = (int)(f4 / (512 * (size_t)kC16));
  if (gl >= P.split_ng[split]) return;
  const int grp = P.split_g0[split] + gl;
  const int tap = row < 64 ? P.ta[grp] : P.tb[grp];
  if (row >= 64 && P.tb[grp] == P.ta[grp]) return;  // discarded half of a self-paired tap
  const int c = P.split_chunk[split] * 64 + (row & 63);
  if (c >= cin) return;
  for (int j = 0; j < 4; ++j) {
    const int k = c16 * 16 + vq * 4 + j;
    dw[((size_t)k * taps + tap) * cin + c] = t4[j];
  }
}

}  // namespace

size_t wgrad_partial_floats(int num_sms, int c_in, int c_out, int taps) {
  WgPlan P;
  const int nout = nout_for(c_out);
  if (!make_wg_plan(P, taps, c_in, nout)) return 0;
  return (size_t)num_sms * P.gmax * 128 * nout;
}

bool wgrad_dz_tma_fits(const HaloGeom& g_in, int c_out) {
  HaloGeom g = g_in;
  const int nout = nout_for(c_out);
  if (nout != c_out || !hc::finish_geom(g, nout <= 64 ? 2 : 1)) return false;
  return wg_layout(g, nout).total + 1024 <= 227 * 1024;
}

int launch_wgrad_reduce(const float* part, float* dw, const WgPlan& plan, int grid, int c_in, int taps,
                        int nout, cudaStream_t st) {
  const size_t per_cta = (size_t)plan.gmax * (nout / 16) * 512;
  const int rgrid = (int)((per_cta + kRedSpan - 1) / kRedSpan) * plan.nsplit;
  switch (nout) {
    case 16: wgrad_reduce_kernel<16><<<rgrid, kRedThreads, 0, st>>>(part, dw, plan, grid, c_in, taps); break;
    case 32: wgrad_reduce_kernel<32><<<rgrid, kRedThreads, 0, st>>>(part, dw, plan, grid, c_in, taps); break;
    case 64: wgrad_reduce_kernel<64><<<rgrid, kRedThreads, 0, st>>>(part, dw, plan, grid, c_in, taps); break;
    case 128: wgrad_reduce_kernel<128><<<rgrid, kRedThreads, 0, st>>>(part, dw, plan, grid, c_in, taps); break;
    default: return 3;
  }
  return cudaGetLastError() == cudaSuccess ? 0 : 6;
}

int launch_wgrad(const WgradArgs& w, int c_in, int c_out, bool bf16, const void* x, int num_sms,
                 cudaStream_t st, void (*between)(void*), void* ctx) {
  WgKArgs a{};
  a.g = w.g;
  a.part = w.part;
  a.err = w.err;
  const int nout = nout_for(c_out);
  if (c_in > 128 || nout != c_out || w.dz_full == nullptr) return 3;
  const int U = nout <= 64 ? 2 : 1;
  if (!hc::finish_geom(a.g, U)) return 3;
  const int taps = a.g.r * a.g.s;
  if (!make_wg_plan(a.plan, taps, c_in, nout)) return 3;
  const WgLayout L = wg_layout(a.g, nout);
  const uint32_t smem = L.total + 1024;
  if (smem > 227 * 1024) return 3;
  const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap mx, mdz;
  const HaloGeom& g = a.g;
  {
    const uint64_t dims[4] = {(uint64_t)c_in, (uint64_t)g.w, (uint64_t)g.h, (uint64_t)g.n_img};
    const uint64_t strides[3] = {(uint64_t)c_in * 2, (uint64_t)g.w * c_in * 2, (uint64_t)g.h * g.w * c_in * 2};
    const uint32_t box[4] = {64, (uint32_t)g.wp, (uint32_t)g.box_rows, 1};
    if (!encode_tiled(&mx, dt, 4, x, dims, strides, box)) return 6;
  }
  {
    // [n][p*wp][cout]: the unit's um padded-linear rows are one box
    const uint64_t rows = (uint64_t)g.p * g.wp;
    const uint64_t dims[3] = {(uint64_t)c_out, rows, (uint64_t)g.n_img};
    const uint64_t strides[2] = {(uint64_t)c_out * 2, rows * c_out * 2};
    const uint32_t box[3] = {64, (uint32_t)g.um, 1};
    if (!encode_tiled(&mdz, dt, 3, w.dz_full, dims, strides, box)) return 6;
  }
  // every CTA gets at least one unit, so every partial it writes is initialised
  const int per_split = std::max(1, std::min(num_sms / a.plan.nsplit, g.total_units));
  const int grid = per_split * a.plan.nsplit;
  auto launch = [&](auto kern) -> int {
    if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), 227 * 1024)) return 6;
    kern<<<grid, kWgThreads, smem, st>>>(mx, mdz, a);
    return cudaGetLastError() == cudaSuccess ? 0 : 6;
  };
  int rc;
  switch (nout * 2 + (bf16 ? 1 : 0)) {
#define CBR_WG_CASE(N_)                                            \
    case N_ * 2 + 0: rc = launch(wgrad_kernel<N_, false>); break; \
    case N_ * 2 + 1: rc = launch(wgrad_kernel<N_, true>); break;
    CBR_WG_CASE(16)
    CBR_WG_CASE(32)
    CBR_WG_CASE(64)
    CBR_WG_CASE(128)
#undef CBR_WG_CASE
    default: return 3;
  }
  if (rc) return rc;
  if (between) between(ctx);
  return launch_wgrad_reduce(a.part, w.dw, a.plan, grid, c_in, taps, nout, st);
}

}  // namespace cbr
