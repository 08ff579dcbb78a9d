// B2 + B3 in one kernel: the data gradient (DGrad) and the weight gradient (WGrad) of the
// convolution (Tech-Renaissance CBR page, section 5.2) over one on-chip tile of
//   dz = gamma*inv_std*(g - dbeta/M - xhat*dgamma/M),  g = dy*mask
// (section 5.1; BatchNorm CUDA page, section 3.1), evaluated as dz = a*g - d*z + e with the
// per-channel coefficients of the backward reduction pass.  dz never reaches HBM: producer
// warps read dy, z and the mask (or y) once per tile, evaluate dz in fp32, round it to the
// storage dtype and write it into a 128-byte-swizzled shared-memory tile that both tcgen05
// contractions read:
//   DGrad: dx[m] = sum over taps (r,s) of dz[m + (r-pad)*wp + (s-pad)] . W[flipped tap], with the
//          dz tile as the K-major A operand (one row-shifted descriptor per tap) and the filter
//          (resident in shared memory) as the MN-major B operand;
//   WGrad: dW[tap pair] += x_halo[rows shifted by the tap]^T . dz, with the TMA-loaded input halo
//          as the MN-major A operand (two taps per M = 128 MMA) and the same dz tile, read
//          MN-major, as B.
// The convolution must be stride 1 with 'same' padding (R = S in {1, 3}, pad = (R-1)/2), so the
// forward and data-gradient convolutions share one padded-linear row space of width
// wp = W + 2*pad (see HaloGeom): dz row L = p*wp + q (q >= Q, or p outside [0, P), is zero),
// and the tile of a unit of output rows [m0, m0 + 256) holds dz rows [m0 - D, m0 + 256 + D),
// D = pad*wp + pad, which covers the data gradient's halo and, at offset D, the weight
// gradient's rows.
//
// Warps: 0 TMA (filter once, input halo per unit); 1 tcgen05.mma issuer and TMEM owner;
// 2-5 data-gradient epilogue (TMEM -> registers -> dx); 6-11 dz producers.  At the end warps
// 2-9 write the CTA's weight-gradient partial, which wgrad_reduce_kernel (conv_bwd.cu) sums
// over CTAs in a fixed order.  Pipelines: 2 dz stages, 1 input-halo stage (its next load runs
// under the next unit's data-gradient MMAs), 1 data-gradient accumulator stage (drained under
// the same unit's weight-gradient MMAs).  TMEM: weight-gradient accumulators in columns
// [0, groups*Cout) for the whole kernel, the data-gradient accumulator in [384, 512).
#include <algorithm>
#include <type_traits>

#include "halo_conv.cuh"

namespace cbr {
namespace {

// 12 warps: the register file is split over the SM's four sub-partitions, so with 12 warps
// (three per sub-partition) every thread can hold up to 168 registers.
constexpr int kEpiWarps = 4;
constexpr int kProdWarps = 6;
constexpr int kEpiWarp0 = 2;
constexpr int kProdWarp0 = kEpiWarp0 + kEpiWarps;
constexpr int kThreads = (kProdWarp0 + kProdWarps) * 32;  // 384
constexpr int kProdThreads = kProdWarps * 32;
constexpr int kRowStep = kProdThreads / 8;                // tile rows per producer sweep (24)
constexpr int kU = 2;                 // M tiles of 128 rows per unit
constexpr int kND = 64;               // data-gradient MMA N (input channels, zero-padded)
constexpr int kDcol = 384;            // TMEM column of the data-gradient accumulator
constexpr int kMaxGroups = 5;         // tap pairs of a 3x3 filter
constexpr int kWslab = 64 * 128;      // one flipped filter tap: 64 x 64 in the storage dtype
constexpr int kPU = 6;                // dz vectors in flight per producer thread (bit mask)
constexpr int kPUY = 5;               // the same when the mask is re-derived from y (3 loads each)

struct FusedKArgs {
  HaloGeom g;               // forward geometry, finished for U = 2 (um = 256)
  const void* x;            // the forward input (for L2 prefetches; the halo itself is read by TMA)
  const void* dy;
  const void* z;
  const void* y;
  const uint8_t* mask;
  const float* coef;
  void* dx;
  float* part;
  uint32_t* err;
  int cin, cout;
  int D;                    // pad*wp + pad
  int nb;                   // dz tile rows: um + 2*D
  int ngroups;
  int has_dx;
  int ta[kMaxGroups], tb[kMaxGroups];
};

struct FusedLayout {
  uint32_t x_bytes, dz_stride, off_dz, off_w, off_bar, total;
};

enum : int { kBarXFull = 0, kBarXEmpty, kBarDzFull, kBarDzFull1, kBarDzEmpty, kBarDzEmpty1, kBarAccFull,
             kBarAccEmpty, kBarWFull, kBarDrain, kNumBars };

__host__ __device__ inline FusedLayout fused_layout(const HaloGeom& g, int nb, int taps) {
  FusedLayout L;
  L.x_bytes = ((uint32_t)g.hr * g.wp * 128 + 1023u) & ~1023u;
  L.dz_stride = ((uint32_t)nb * 128 + 1023u) & ~1023u;
  L.off_dz = L.x_bytes;
  L.off_w = L.off_dz + 2 * L.dz_stride;
  L.off_bar = L.off_w + (uint32_t)taps * kWslab;
  L.total = L.off_bar + kNumBars * 8 + 16;
  return L;
}

// floor(v / d) for d > 0 and any sign of v
__device__ __forceinline__ int floor_div(int v, int d) { return v >= 0 ? v / d : -((-v + d - 1) / d); }

template <int NW, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    dgrad_wgrad_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                       const FusedKArgs a) {
  static_assert(kMaxGroups * NW <= kDcol, "TMEM columns");
  static_assert(kProdWarps >= 4, "the weight-gradient drain uses warps 2-9");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const HaloGeom& g = a.g;
  const int rs = g.r * g.s;
  const FusedLayout L = fused_layout(g, a.nb, rs);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t x_addr = sbase, dz_addr = sbase + L.off_dz, w_addr = sbase + L.off_w;
  const uint32_t bar0 = sbase + L.off_bar;
  auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.off_bar + kNumBars * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int T = g.total_units;
  const int rows_img = g.p * g.wp;
  const bool has_dx = a.has_dx != 0;
  // units of this CTA: a contiguous run of the T units (balanced to within one), walked from
  // its last unit to its first, so that consecutive units of one image share 2*D dz tile rows
  const int per = T / (int)gridDim.x, rem = T % (int)gridDim.x;
  const int first = (int)blockIdx.x * per + min((int)blockIdx.x, rem);
  const int nunits = per + ((int)blockIdx.x < rem ? 1 : 0);
  auto unit_of = [&](int jj) { return first + nunits - 1 - jj; };

  if (threadIdx.x == 0) {
    mbar_init(bar(kBarXFull), 1);
    mbar_init(bar(kBarXEmpty), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kBarDzFull + i), kProdWarps);
      mbar_init(bar(kBarDzEmpty + i), 1);
    }
    mbar_init(bar(kBarAccFull), 1);
    mbar_init(bar(kBarAccEmpty), kEpiWarps);
    mbar_init(bar(kBarWFull), 1);
    mbar_init(bar(kBarDrain), 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA: filter, input halos
    if (lane == 0) {
      prefetch_tensormap(&map_x);
      if (has_dx) {
        prefetch_tensormap(&map_w);
        mbar_arrive_expect_tx(bar(kBarWFull), (uint32_t)rs * kWslab);
        // slab t holds flipped tap rs-1-t: [k][c] with c contiguous (read MN-major)
        for (int t = 0; t < rs; ++t) tma_load_3d(w_addr + (uint32_t)t * kWslab, &map_w, 0, rs - 1 - t, 0, bar(kBarWFull));
      }
      const uint32_t tx = (uint32_t)g.hr * g.wp * 128;
      // L2 prefetch of what a unit's producers and halo load will read: the dy, z and mask (or
      // y) pixels of its dz tile rows, and its input halo rows.  Issued two units ahead for the
      // producers and one ahead for the halo, so their loads hit L2 instead of waiting on HBM.
      const size_t img_px = (size_t)g.p * g.q;
      auto prefetch_dz_inputs = [&](int u) {
        const int n = u / g.upi;
        const int m0 = (u - n * g.upi) * g.um;
        const int l0 = max(m0 - a.D, 0), l1 = min(m0 + g.um + a.D, rows_img) - 1;
        if (l1 < l0) return;
        const int p0 = l0 / g.wp, p1 = l1 / g.wp;
        const size_t px0 = (size_t)n * img_px + (size_t)p0 * g.q + min(l0 - p0 * g.wp, g.q);
        const size_t px1 = (size_t)n * img_px + (size_t)p1 * g.q + min(l1 - p1 * g.wp, g.q - 1) + 1;
        if (px1 <= px0) return;
        const size_t row_b = (size_t)a.cout * 2;
        const uint32_t bytes = (uint32_t)((px1 - px0) * row_b);
        bulk_prefetch_l2(static_cast<const uint8_t*>(a.dy) + px0 * row_b, bytes);
        bulk_prefetch_l2(static_cast<const uint8_t*>(a.z) + px0 * row_b, bytes);
        if (a.mask) {
          // whole 16-byte blocks inside the mask (one bit per element, n*P*Q*cout/8 bytes)
          const size_t mask_end = ((size_t)g.n_img * img_px * a.cout / 8) & ~(size_t)15;
          const size_t b0 = (px0 * a.cout / 8) & ~(size_t)15;
          const size_t b1 = min((px1 * a.cout / 8 + 15) & ~(size_t)15, mask_end);
          if (b1 > b0) bulk_prefetch_l2(a.mask + b0, (uint32_t)(b1 - b0));
        } else {
          bulk_prefetch_l2(static_cast<const uint8_t*>(a.y) + px0 * row_b, bytes);
        }
      };
      const size_t xrow_b = (size_t)g.w * a.cin * 2;
      auto prefetch_halo = [&](int u) {
        const int n = u / g.upi;
        const int m0 = (u - n * g.upi) * g.um;
        const int h0 = max(m0 / g.wp - g.pad, 0), h1 = min(m0 / g.wp - g.pad + g.hr, g.h);
        if (h1 > h0)
          bulk_prefetch_l2(static_cast<const uint8_t*>(a.x) + ((size_t)n * g.h + h0) * xrow_b,
                           (uint32_t)((size_t)(h1 - h0) * xrow_b));
      };
      int issued = 0;
      for (int jj = 0; jj < nunits && !hc::is_aborted(abort_flag); ++jj) {
        const int u = unit_of(jj);
        const int n = u / g.upi;
        const int m0 = (u - n * g.upi) * g.um;
        if (jj + 2 < nunits) prefetch_dz_inputs(unit_of(jj + 2));
        if (jj + 1 < nunits) prefetch_halo(unit_of(jj + 1));
        if (!mbar_wait_backoff(bar(kBarXEmpty), (uint32_t)(jj & 1) ^ 1u, 64)) {
          hc::set_abort(abort_flag, a.err, kErrWaitHalo);
          break;
        }
        mbar_arrive_expect_tx(bar(kBarXFull), tx);
        for (int r0 = 0; r0 < g.hr; r0 += g.box_rows)
          tma_load_4d(x_addr + (uint32_t)r0 * g.wp * 128, &map_x, 0, -g.pad, m0 / g.wp - g.pad + r0, n,
                      bar(kBarXFull));
        issued = jj + 1;
      }
      // never leave the CTA with a copy in flight
      if (issued) mbar_wait(bar(kBarXFull), (uint32_t)((issued - 1) & 1));
      if (has_dx) mbar_wait(bar(kBarWFull), 0);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop in converged control flow (warp-uniform descriptor
    // arithmetic) and one elected lane issues each MMA and commit; every decision that changes
    // control flow is voted across the warp.
    const uint32_t idesc_d = make_idesc_f16(128, kND, BF16, false, true);
    const uint32_t idesc_w = make_idesc_f16(128, NW, BF16, true, true);
    const uint64_t b_w = make_sw128_desc(w_addr, 8192, 1024, 0);
    const uint64_t a_row_skip = (uint64_t)((g.wp - g.s) * 128 / 16);  // end of a filter row
    // weight-gradient A descriptors with a zero start address: LBO = the two taps' row distance
    uint64_t a_grp[kMaxGroups];
#pragma unroll
    for (int gl = 0; gl < kMaxGroups; ++gl) {
      a_grp[gl] = 0;
      if (gl < a.ngroups) {
        const int ta = a.ta[gl], tb = a.tb[gl];
        const int sha = (ta / g.s) * g.wp + ta % g.s;
        const int shb = (tb / g.s) * g.wp + tb % g.s;
        a_grp[gl] = make_sw128_desc((uint32_t)sha * 128u, (uint32_t)(shb - sha) * 128u, 1024, 0);
      }
    }
    bool bad = false;
    if (has_dx && !__all_sync(0xffffffffu, mbar_wait(bar(kBarWFull), 0))) {
      hc::set_abort(abort_flag, a.err, kErrWaitWeights);
      bad = true;
    }
    tc_fence_after();
    uint32_t wacc = 0;  // 0 until the first weight-gradient MMA of the CTA
    for (int jj = 0; jj < nunits && !bad; ++jj) {
      if ((jj & 7) == 7 && __any_sync(0xffffffffu, hc::is_aborted(abort_flag))) break;
      const int u = unit_of(jj);
      const int n = u / g.upi;
      const int m0 = (u - n * g.upi) * g.um;
      const int off = m0 - (m0 / g.wp) * g.wp;
      const int ntiles = min(kU, (rows_img - m0 + 127) / 128);
      const uint32_t s = jj & 1, ph = (jj >> 1) & 1;
      const uint32_t dzb = dz_addr + s * L.dz_stride;
      // the dz tile and the data-gradient accumulator are tested back to back (their latencies
      // overlap); only when one is not complete yet are they waited for one by one
      const bool ready = __all_sync(0xffffffffu, mbar_test(bar(kBarDzFull + s), ph) &
                                                     (!has_dx || mbar_test(bar(kBarAccEmpty), (uint32_t)(jj & 1) ^ 1u)));
      if (!ready) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarDzFull + s), ph))) {
          hc::set_abort(abort_flag, a.err, kErrWaitOperand);
          break;
        }
        if (has_dx && !__all_sync(0xffffffffu, mbar_wait(bar(kBarAccEmpty), (uint32_t)(jj & 1) ^ 1u))) {
          hc::set_abort(abort_flag, a.err, kErrWaitAccum);
          break;
        }
      }
      tc_fence_after();
      if (has_dx) {
        // ---- data gradient: tap (r, s) of the flipped filter reads tile rows t*128 + r*wp + s
        const uint32_t dcol = tmem_base + kDcol;
        auto run_taps = [&](auto nt_c, auto rs_c) {
          constexpr int NT = decltype(nt_c)::value, RS = decltype(rs_c)::value;
          uint64_t a_tap = make_sw128_desc(dzb, 16, 1024, 0);
          uint64_t b_tap = b_w;
          int sx = 0;
          // not unrolled: one tap's 8 MMAs are the loop body, which keeps the issue loop in the
          // instruction cache (unrolled over the taps, the issue ran about 6% slower)
#pragma unroll 1
          for (int tap = 0; tap < RS; ++tap) {
            // opaque to the compiler, so the 8 descriptors of a tap are formed just before their
            // MMAs instead of all 72 of a unit being precomputed into registers
            asm volatile("" : "+l"(a_tap), "+l"(b_tap));
            const uint32_t acc0 = tap != 0 ? 1u : 0u;
#pragma unroll
            for (int t = 0; t < NT; ++t)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_f16_ss_warp(dcol + t * kND, a_tap + (uint64_t)((t * 128 * 128 + kk * 32) >> 4),
                                b_tap + (uint64_t)((kk * 2048) >> 4), idesc_d, kk ? 1u : acc0);
            const bool wrap = sx + 1 == g.s;
            sx = wrap ? 0 : sx + 1;
            a_tap += wrap ? 8 + a_row_skip : 8;
            b_tap += kWslab >> 4;
          }
        };
        if (rs == 9) {
          if (ntiles == kU) run_taps(std::integral_constant<int, kU>{}, std::integral_constant<int, 9>{});
          else run_taps(std::integral_constant<int, 1>{}, std::integral_constant<int, 9>{});
        } else {
          if (ntiles == kU) run_taps(std::integral_constant<int, kU>{}, std::integral_constant<int, 1>{});
          else run_taps(std::integral_constant<int, 1>{}, std::integral_constant<int, 1>{});
        }
        mma_commit_warp(bar(kBarAccFull));
      }
      // ---- weight gradient over the unit's 256 rows: A = input halo, B = dz rows [D, D + 256)
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kBarXFull), (uint32_t)(jj & 1)))) {
        hc::set_abort(abort_flag, a.err, kErrWaitHalo);
        break;
      }
      tc_fence_after();
      const uint64_t a_unit = (uint64_t)((x_addr + (uint32_t)off * 128u) >> 4);
      uint64_t bd = make_sw128_desc(dzb + (uint32_t)a.D * 128u, (uint32_t)a.nb * 128u, 1024, 0);
      auto issue = [&](auto ng_c) {
        constexpr int NG = decltype(ng_c)::value;
#pragma unroll 4
        for (int kk = 0; kk < kU * 8; ++kk) {
          const uint64_t ak = a_unit + (uint64_t)kk * 128;  // 16 pixel rows further
#pragma unroll
          for (int gl = 0; gl < NG; ++gl) mma_f16_ss_warp(tmem_base + gl * NW, a_grp[gl] + ak, bd, idesc_w, wacc);
          bd += 128;
          wacc = 1u;
        }
      };
      if (a.ngroups == 5) issue(std::integral_constant<int, 5>{});
      else issue(std::integral_constant<int, 1>{});
      // the input halo and the dz stage are free once these MMAs complete
      mma_commit_warp(bar(kBarXEmpty));
      mma_commit_warp(bar(kBarDzEmpty + s));
    }
    mma_commit_warp(bar(kBarDrain));
    mbar_wait(bar(kBarDrain), 0);
  } else if (warp < kProdWarp0) {
    // ------------------------------------------------------------ data-gradient epilogue
    const int quad = warp & 3;
    const int e = quad * 32 + lane;  // accumulator row (TMEM lane) owned by this thread
    const int cin = a.cin;
    const size_t opitch = (size_t)cin * 2;
    const bool v8 = (cin % 16) == 0 && (reinterpret_cast<uintptr_t>(a.dx) & 31) == 0;
    uint8_t* obase = static_cast<uint8_t*>(a.dx);
    for (int jj = 0; has_dx && jj < nunits && !hc::is_aborted(abort_flag); ++jj) {
      const int u = unit_of(jj);
      const int n = u / g.upi;
      const int m0 = (u - n * g.upi) * g.um;
      const int ntiles = min(kU, (rows_img - m0 + 127) / 128);
      if (!mbar_wait_backoff(bar(kBarAccFull), (uint32_t)(jj & 1), 128)) {
        hc::set_abort(abort_flag, a.err, kErrWaitMma);
        break;
      }
      tc_fence_after();
      for (int t = 0; t < ntiles; ++t) {
        const int m = m0 + t * 128 + e;
        const int h = m / g.wp, w = m - h * g.wp;
        const bool valid = h < g.h && w < g.w;
        uint8_t* orow = obase + (size_t)(((long long)n * g.h + h) * g.w + w) * opitch;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t r[32];
          const uint32_t ta = tmem_base + ((uint32_t)(quad * 32) << 16) + kDcol + t * kND + half * 32;
          tmem_ld16(ta, *reinterpret_cast<uint32_t(*)[16]>(r));
          tmem_ld16(ta + 16, *reinterpret_cast<uint32_t(*)[16]>(r + 16));
          tmem_ld_wait();
          if (half == 1 && t == ntiles - 1) {
            // the warp's last read of the accumulator: order it before the arrival
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarAccEmpty));
          }
          if (valid) {
            uint4 pk[4];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc)
              pk[cc] = make_uint4(pack2<BF16>(__uint_as_float(r[8 * cc + 0]), __uint_as_float(r[8 * cc + 1])),
                                  pack2<BF16>(__uint_as_float(r[8 * cc + 2]), __uint_as_float(r[8 * cc + 3])),
                                  pack2<BF16>(__uint_as_float(r[8 * cc + 4]), __uint_as_float(r[8 * cc + 5])),
                                  pack2<BF16>(__uint_as_float(r[8 * cc + 6]), __uint_as_float(r[8 * cc + 7])));
            const int c0 = half * 32;
            if (v8) {
#pragma unroll
              for (int cc = 0; cc < 2; ++cc)
                if (c0 + 16 * cc < cin) st_global_v8(orow + (c0 + 16 * cc) * 2, pk[2 * cc], pk[2 * cc + 1]);
            } else {
#pragma unroll
              for (int cc = 0; cc < 4; ++cc)
                if (c0 + 8 * cc < cin) st_global_v4(orow + (c0 + 8 * cc) * 2, pk[cc]);
            }
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ dz producers
    // Thread tid always handles 16-byte chunk c8 (8 channels) of tile rows rsub, rsub + 24, ...,
    // so its coefficients stay in registers; a warp covers 4 rows x 128 bytes (coalesced).
    const int tid = threadIdx.x - kProdWarp0 * 32;
    const int c8 = tid & 7, rsub = tid >> 3;
    const int ch0 = c8 * 8;
    const int cout = a.cout;
    const bool ch_ok = ch0 < cout;
    float ca[8], cd[8], ce[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      ca[j] = ch_ok ? __ldg(a.coef + ch0 + j) : 0.f;
      cd[j] = ch_ok ? __ldg(a.coef + cout + ch0 + j) : 0.f;
      ce[j] = ch_ok ? __ldg(a.coef + 2 * cout + ch0 + j) : 0.f;
    }
    const uint8_t* dyb = static_cast<const uint8_t*>(a.dy);
    const uint8_t* zb = static_cast<const uint8_t*>(a.z);
    const uint8_t* yb = static_cast<const uint8_t*>(a.y);
    const int P = g.p, Q = g.q, wp = g.wp;
    const int ov = 2 * a.D;  // tile rows shared by consecutive units of one image
    // Evaluate tile rows [0, nrows) of one unit: rows L = m0 - D + rsub + 24k of image n, in
    // batches of NP items whose loads are all issued before the first is used.  MB: the mask is
    // the bit-packed forward mask, else it is re-derived as y > 0.
    auto fill = [&](auto maskbits_c, uint32_t dst, int n, int m0, int nrows) {
      constexpr bool MB = decltype(maskbits_c)::value;
      constexpr int NP = MB ? kPU : kPUY;
      const int nit = (nrows - rsub + kRowStep - 1) / kRowStep;  // tile rows of this thread
      const int L0 = m0 - a.D + rsub;
      int p = floor_div(L0, wp);
      int q = L0 - p * wp;
      for (int k0 = 0; k0 < nit; k0 += NP) {
        uint4 dv[NP], zv[NP], yv[MB ? 1 : NP];
        uint32_t mb[MB ? NP : 1];
        uint32_t okm = 0;  // bit j: item j is inside the image (loaded)
#pragma unroll
        for (int j = 0; j < NP; ++j) {
          if (k0 + j < nit && ch_ok && p >= 0 && p < P && q < Q) {
            okm |= 1u << j;
            const size_t v = (((size_t)n * P + p) * Q + q) * cout + ch0;  // element index
            dv[j] = ld_global_nc_v4(dyb + v * 2);
            zv[j] = ld_global_nc_v4(zb + v * 2);
            if constexpr (MB) mb[j] = a.mask[v >> 3];
            else yv[j] = ld_global_nc_v4(yb + v * 2);
          }
          q += kRowStep;
          while (q >= wp) {
            q -= wp;
            ++p;
          }
        }
#pragma unroll
        for (int j = 0; j < NP; ++j) {
          if (k0 + j >= nit) break;
          uint4 o = make_uint4(0u, 0u, 0u, 0u);
          if (okm & (1u << j)) {
            uint32_t bits;
            if constexpr (MB) {
              bits = mb[j];
            } else {
              const uint32_t yw[4] = {yv[j].x, yv[j].y, yv[j].z, yv[j].w};
              bits = 0;
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 yy = unpack2<BF16>(yw[e]);
                bits |= (yy.x > 0.f ? 1u : 0u) << (2 * e);
                bits |= (yy.y > 0.f ? 1u : 0u) << (2 * e + 1);
              }
            }
            const uint32_t dw[4] = {dv[j].x, dv[j].y, dv[j].z, dv[j].w};
            const uint32_t zw[4] = {zv[j].x, zv[j].y, zv[j].z, zv[j].w};
            uint32_t ow[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 d = unpack2<BF16>(dw[e]);
              const float2 zz = unpack2<BF16>(zw[e]);
              const float g0 = (bits >> (2 * e)) & 1u ? d.x : 0.f;
              const float g1 = (bits >> (2 * e + 1)) & 1u ? d.y : 0.f;
              const float r0 = fmaf(ca[2 * e], g0, fmaf(-cd[2 * e], zz.x, ce[2 * e]));
              const float r1 = fmaf(ca[2 * e + 1], g1, fmaf(-cd[2 * e + 1], zz.y, ce[2 * e + 1]));
              ow[e] = pack2<BF16>(r0, r1);
            }
            o = make_uint4(ow[0], ow[1], ow[2], ow[3]);
          }
          st_shared_v4(dst + swz_off((uint32_t)(rsub + kRowStep * (k0 + j)), (uint32_t)c8, 128), o);
        }
      }
    };
    int prev_u = -1;
    for (int jj = 0; jj < nunits; ++jj) {
      const int u = unit_of(jj);
      const int n = u / g.upi;
      const int m0 = (u - n * g.upi) * g.um;
      const uint32_t s = jj & 1, ph = (jj >> 1) & 1;
      const bool live = !hc::is_aborted(abort_flag);
      const bool waited = live && mbar_wait_backoff(bar(kBarDzEmpty + s), ph ^ 1u, 64);
      if (live && !waited) hc::set_abort(abort_flag, a.err, kErrWaitOperand);
      // Every producer thread votes here once per unit, so they all leave the loop together (a
      // named barrier has no time limit).  Passing it also means every producer has finished
      // writing the previous unit's tile, whose rows are copied below.
      if (!named_bar_and(1, kProdThreads, waited)) break;
      const uint32_t dst = dz_addr + s * L.dz_stride;
      // The previous unit (u + 1, same image) begins um rows later: its tile rows [0, 2D) are
      // this tile's rows [um, um + 2D).  um is a multiple of 8, so both have the same swizzle
      // phase and the 128-byte rows are copied verbatim.
      const bool reuse = prev_u == u + 1 && prev_u / g.upi == n && ov > 0;
      if (reuse) {
        const uint32_t src = dz_addr + (s ^ 1u) * L.dz_stride;
        for (int i = tid; i < ov * 8; i += kProdThreads)
          st_shared_v4(dst + (uint32_t)g.um * 128u + (uint32_t)i * 16u, ld_shared_v4(src + (uint32_t)i * 16u));
      }
      const int nrows = reuse ? g.um : a.nb;
      if (a.mask) fill(std::true_type{}, dst, n, m0, nrows);
      else fill(std::false_type{}, dst, n, m0, nrows);
      // generic-proxy writes -> visible to the tensor cores; one arrival per warp
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarDzFull + s));
      prev_u = u;
    }
  }

  // ------------------------------------------------------------ weight-gradient partial
  if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 8) {
    const bool ok = mbar_wait_backoff(bar(kBarDrain), 0, 256);
    if (!ok) hc::set_abort(abort_flag, a.err, kErrWaitMma);
    tc_fence_after();
    if (ok) {
      // 8 warps, two per TMEM lane quadrant: warp jq of a quadrant takes column blocks
      // jq, jq + 2, ... of the groups x (Cout / 16) blocks
      constexpr int kC16 = NW / 16;
      const int quad = warp & 3, jq = (warp - kEpiWarp0) >> 2;
      const int e = quad * 32 + lane;  // accumulator row = (tap half, input channel)
      const int nblk = a.ngroups * kC16;
      for (int blk = jq; blk < nblk; blk += 2) {
        const int gl = blk / kC16, c16 = blk - gl * kC16;
        uint32_t r[16];
        tmem_ld16(tmem_base + ((uint32_t)(quad * 32) << 16) + gl * NW + c16 * 16, r);
        tmem_ld_wait();
        // partial layout [cta][group][c16][v][row][4] (wgrad_reduce_kernel): a warp's store is
        // 512 contiguous bytes
        float4* dst = reinterpret_cast<float4*>(a.part) +
                      (((size_t)blockIdx.x * a.ngroups + gl) * kC16 + c16) * 512 + e;
#pragma unroll
        for (int v = 0; v < 4; ++v)
          dst[v * 128] = make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                     __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// Geometry of the fused kernel for a layer, or false if it does not take the layer.
bool fused_geom(HaloGeom& g, int c_in, int c_out, int stride, int* D, int* nb) {
  if (stride != 1 || g.r != g.s || !(g.r == 1 || g.r == 3) || g.pad != (g.r - 1) / 2) return false;
  if (c_in % 8 != 0 || c_in > 64 || !(c_out == 16 || c_out == 32 || c_out == 64)) return false;
  if (!hc::finish_geom(g, kU)) return false;
  *D = g.pad * g.wp + g.pad;
  *nb = g.um + 2 * *D;
  return fused_layout(g, *nb, g.r * g.s).total + 1024 <= 227 * 1024;
}

}  // namespace

bool bwd_fused_supported(int n, int h, int w, int c_in, int c_out, int r, int s, int stride, int pad) {
  HaloGeom g{};
  g.n_img = n;
  g.h = h;
  g.w = w;
  g.r = r;
  g.s = s;
  g.pad = pad;
  int D = 0, nb = 0;
  return fused_geom(g, c_in, c_out, stride, &D, &nb);
}

int launch_bwd_fused(const BwdFusedArgs& f, int c_in, int c_out, bool bf16, const void* x, const void* w,
                     int num_sms, cudaStream_t st, void (*between)(void*), void* ctx) {
  FusedKArgs a{};
  a.g = f.g;
  if (!fused_geom(a.g, c_in, c_out, 1, &a.D, &a.nb)) return 3;
  const HaloGeom& g = a.g;
  const int taps = g.r * g.s;
  WgPlan plan;
  if (!make_wg_plan(plan, taps, c_in, c_out) || plan.nsplit != 1 || plan.ngroups > kMaxGroups) return 3;
  a.ngroups = plan.ngroups;
  for (int i = 0; i < plan.ngroups; ++i) {
    a.ta[i] = plan.ta[i];
    a.tb[i] = plan.tb[i];
  }
  a.x = x;
  a.dy = f.dy;
  a.z = f.z;
  a.y = f.y;
  a.mask = f.mask;
  a.coef = f.coef;
  a.dx = f.dx;
  a.has_dx = f.dx != nullptr;
  a.part = f.part;
  a.err = f.err;
  a.cin = c_in;
  a.cout = c_out;
  const FusedLayout L = fused_layout(g, a.nb, taps);
  const uint32_t smem = L.total + 1024;
  const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap mx, mw;
  {
    const uint64_t dims[4] = {(uint64_t)c_in, (uint64_t)g.w, (uint64_t)g.h, (uint64_t)g.n_img};
    const uint64_t strides[3] = {(uint64_t)c_in * 2, (uint64_t)g.w * c_in * 2, (uint64_t)g.h * g.w * c_in * 2};
    const uint32_t box[4] = {64, (uint32_t)g.wp, (uint32_t)g.box_rows, 1};
    if (!encode_tiled(&mx, dt, 4, x, dims, strides, box)) return 6;
  }
  {
    // [cout][taps][cin]: one box is one tap, 64 output channels (K) x 64 input channels (N)
    const uint64_t dims[3] = {(uint64_t)c_in, (uint64_t)taps, (uint64_t)c_out};
    const uint64_t strides[2] = {(uint64_t)c_in * 2, (uint64_t)taps * c_in * 2};
    const uint32_t box[3] = {64, 1, 64};
    if (!encode_tiled(&mw, dt, 3, w, dims, strides, box)) return 6;
  }
  // every CTA gets at least one unit, so every partial it writes is initialised
  const int grid = std::min(g.total_units, num_sms);
  auto launch = [&](auto kern) -> int {
    if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), 227 * 1024)) return 6;
    kern<<<grid, kThreads, smem, st>>>(mx, mw, a);
    return cudaGetLastError() == cudaSuccess ? 0 : 6;
  };
  int rc;
  switch (c_out * 2 + (bf16 ? 1 : 0)) {
    case 16 * 2 + 0: rc = launch(dgrad_wgrad_kernel<16, false>); break;
    case 16 * 2 + 1: rc = launch(dgrad_wgrad_kernel<16, true>); break;
    case 32 * 2 + 0: rc = launch(dgrad_wgrad_kernel<32, false>); break;
    case 32 * 2 + 1: rc = launch(dgrad_wgrad_kernel<32, true>); break;
    case 64 * 2 + 0: rc = launch(dgrad_wgrad_kernel<64, false>); break;
    case 64 * 2 + 1: rc = launch(dgrad_wgrad_kernel<64, true>); break;
    default: return 3;
  }
  if (rc) return rc;
  if (between) between(ctx);
  return launch_wgrad_reduce(f.part, f.dw, plan, grid, c_in, taps, c_out, st);
}

}  // namespace cbr
