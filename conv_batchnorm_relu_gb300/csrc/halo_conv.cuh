// Generic stride-1 implicit-GEMM convolution over a halo tile, on tcgen05 tensor cores.
//
// Used for the forward convolution (A = input activations, loaded by TMA) and for the data
// gradient of the layers the fused backward kernel does not take (A = dz, loaded by TMA from
// the materialised dz; the filter is the forward filter read MN-major with flipped taps).  See
// HaloGeom for the padded-linear row space in which every filter tap is a row-shifted view of
// one halo tile.
//
// Warp roles:
//   warp 0             TMA producer of the A halo (one halo stage per (unit, 64-channel chunk))
//   warp 1             TMEM owner and tcgen05.mma issuer
//   warp 2             TMA producer for the filter slabs (resident when they fit in smem)
//   warps 3 .. 10      epilogue, two warps per TMEM lane quadrant (each takes half of the
//                      columns): TMEM -> registers -> stats / store
// Pipelines: 2 halo stages, 2 TMEM accumulator stages (U*NOUT fp32 columns each), and a
// 3-deep filter ring when the filter is streamed.  All waits are bounded (ptx.cuh).
#pragma once
#include <type_traits>
#include "cbr_internal.h"
#include "common.cuh"
#include "stats.cuh"

namespace cbr {

// Fprop: A = input halo by TMA.  DgradTma: A = a materialised dz halo by TMA, the filter read
// MN-major with flipped taps, plain epilogue.  FpropBn: the forward convolution whose epilogue
// applies inference BatchNorm and ReLU to the fp32 accumulator, relu(acc*scale + shift), with
// the per-channel scale and shift computed by each CTA into shared memory at its start.
// FpropApply: the whole training forward in one persistent, cooperative launch for batches
// whose accumulators all fit in TMEM at once (at most 4 units per CTA): convolution, z and
// statistics, the finalize by the last CTA, a grid-wide wait for its scale and bias, then
// y = relu(acc*scale + bias) and the bit mask from the accumulators still in TMEM.
enum ConvKind : int { kKindFprop = 0, kKindDgradTma = 2, kKindFpropBn = 3, kKindFpropApply = 4 };

__host__ __device__ constexpr bool is_forward_kind(int kind) {
  return kind == kKindFprop || kind == kKindFpropBn || kind == kKindFpropApply;
}
constexpr int kPersistMaxUnits = 4;  // FpropApply: units per CTA (U*NOUT TMEM columns each, 512 in all)

struct ConvArgs {
  HaloGeom g;
  void* out;                // [n][p][q][out_c] storage dtype: z, y (inference) or dx
  int out_c;                // channels stored per output pixel (<= NOUT)
  int mode;                 // FpropMode (fprop only)
  // forward statistics / finalize
  float* part;
  uint32_t* ticket;
  const float* gamma;
  const float* beta;
  float* running_mean;
  float* running_var;
  float* saved_mean;
  float* saved_inv_var;
  float* eq;
  float* moments;           // split forward: merged moments out instead of the finalize
  int defer;                // write the CTA partials only: the apply pass merges and finalizes
  // FpropApply: y, the bit mask (may be null) and the grid-wide word the last CTA bumps once
  // eq is written (each CTA reads it at its start, then waits for a different value)
  void* y;
  uint32_t* mask;
  uint32_t* ready;
  const float* bias;
  // epilogue-only inference (kKindFpropBn): scale = gamma/sqrt(rv + eps),
  // shift = beta + (conv_bias - rm)*scale (conv_bias may be null)
  const float* bn_gamma;
  const float* bn_beta;
  const float* bn_mean;
  const float* bn_var;
  const float* conv_bias;
  float momentum;
  float eps;
  long long m_count;
  double inv_m;             // 1 / m_count
  float unbias;             // m_count / (m_count - 1)
  uint32_t* err;
};

namespace hc {

constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kStreamStages = 3;

constexpr int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

template <int KIND>
struct Roles {
  static constexpr int kAWarps = 1;
  static constexpr int kMmaWarp = kAWarps;
  static constexpr int kWWarp = kAWarps + 1;
  static constexpr int kEpiWarp0 = kAWarps + 2;
  static constexpr int kThreads = (kAWarps + 2 + kEpiWarps) * 32;
};

// Bytes of one filter slab (one 64-channel K chunk x one tap).
__host__ __device__ constexpr int wslab_bytes(int kind, int nout) {
  return is_forward_kind(kind) ? nout * 128 : (nout > 64 ? nout : 64) * 128;
}

struct Layout {
  uint32_t halo_stride, off_w, off_stage, off_bar, total, wslab, off_bn;
  int nsw;
};

__host__ __device__ inline Layout layout(const HaloGeom& g, int kind, int nch, int nout, bool wres) {
  Layout L;
  const uint32_t halo = (uint32_t)g.hr * g.wp * 128;
  L.halo_stride = (halo + 1023u) & ~1023u;
  L.wslab = (uint32_t)wslab_bytes(kind, nout);
  L.nsw = wres ? nch * g.r * g.s : kStreamStages;
  L.off_w = 2 * L.halo_stride;
  const uint32_t stage = 128u * nout * 2;
  // off_stage: scratch for the end-of-kernel statistics reduction (and the finalize).  It is
  // used only after the epilogue has drained the last accumulator, when every MMA of the CTA
  // has completed and with it every halo load they read, so it shares the halo stages.
  const bool alias = 2 * L.halo_stride >= stage;
  L.off_stage = alias ? 0u : L.off_w + (uint32_t)L.nsw * L.wslab;
  L.off_bar = ((alias ? L.off_w + (uint32_t)L.nsw * L.wslab : L.off_stage + stage) + 15u) & ~15u;
  const uint32_t nbar = 8 + 2 * L.nsw + 1;
  L.total = L.off_bar + nbar * 8 + 16;
  if (kind == kKindFpropBn) {
    // the per-channel inference scale and shift
    L.off_bn = (L.total + 15u) & ~15u;
    L.total = L.off_bn + 2u * (uint32_t)nout * 4u;
  }
  return L;
}

__device__ __forceinline__ bool is_aborted(volatile int* flag) { return *flag != 0; }

__device__ __forceinline__ void set_abort(volatile int* flag, uint32_t* err, uint32_t bits) {
  *flag = 1;
  report_error(err, bits);
}

// Forward statistics, after the main loop: `red` holds the moments of each TMEM lane quadrant
// of this CTA, [4][2][COUT] (mean, M2) followed by the 4 row counts (written by the epilogue,
// visible after a __syncthreads).  Every thread calls this: the quadrants are merged in fixed
// order into the CTA's partial.  With a.defer set that is all (the apply pass merges the grid's
// partials in its prologue); otherwise a wrap-around ticket elects the last CTA, which merges
// the grid's partials (st::merge_partials) and runs bn_finalize.  `scratch` (SCRATCH bytes, may
// alias `red`) holds the merge's working set.
template <int COUT, int kThreads, int SCRATCH>
__device__ void stats_partial_finalize(const ConvArgs& a, const float* red, uint8_t* scratch,
                                       volatile uint32_t* ticket_slot, volatile int* abort_flag) {
  static_assert(kThreads >= COUT, "one thread per channel in the finalize");
  static_assert(st::merge_scratch_floats<COUT>() * 4 <= SCRATCH, "finalize scratch");
  constexpr int kPF = st::partial_floats(COUT);
  // the per-channel inputs of the finalize, loaded before the ticket by every CTA (cheap) so
  // the last one does not wait for them after its merges
  float gm = 0.f, bt = 0.f, rm = 0.f, rv = 0.f;
  if (threadIdx.x < COUT && !a.moments && !a.defer) {
    gm = a.gamma[threadIdx.x];
    bt = a.beta[threadIdx.x];
    rm = a.running_mean[threadIdx.x];
    rv = a.running_var[threadIdx.x];
  }
  float* mypart = a.part + (size_t)blockIdx.x * kPF;
  if (threadIdx.x < COUT) {
    const int c = threadIdx.x;
    const float* cnt = red + 8 * COUT;
    float n = cnt[0], m = red[0 * COUT + c], q = red[1 * COUT + c];
#pragma unroll
    for (int k = 1; k < 4; ++k) st::chan_merge(n, m, q, cnt[k], red[(2 * k) * COUT + c], red[(2 * k + 1) * COUT + c]);
    mypart[c] = m;
    mypart[COUT + c] = q;
    if (c == 0) mypart[2 * COUT] = n;
  }
  if (a.defer) return;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) *ticket_slot = atomicInc(a.ticket, gridDim.x - 1);
  __syncthreads();
  if (*ticket_slot == gridDim.x - 1 && !is_aborted(abort_flag)) {
    // ---------------------------------------------------- bn_finalize (last CTA)
    __threadfence();
    float* fg = reinterpret_cast<float*>(scratch);
    // the other CTAs' partials were written during this launch: read them from L2, ten a
    // thread in flight (four in kernels of more than 512 threads, whose register budget is less)
    constexpr int kLdF = kThreads > 512 ? 4 : 10;
    const float tot_n = st::merge_partials<COUT, kThreads, kLdF>(
        (int)gridDim.x, fg, [&](int b, int c4, float4& m, float4& q, float& n) {
          const float* pb = a.part + (size_t)b * kPF;
          m = __ldcg(reinterpret_cast<const float4*>(pb) + c4);
          q = __ldcg(reinterpret_cast<const float4*>(pb + COUT) + c4);
          n = __ldcg(pb + 2 * COUT);
        });
    if (threadIdx.x < COUT) {
      const int c = threadIdx.x;
      const float tot_m = fg[c], tot_q = fg[COUT + c];
      if (a.moments) {
        // split forward: this call's moments go to the caller, who merges them with other
        // ranks' and finalizes later
        a.moments[c] = tot_m;
        a.moments[COUT + c] = tot_q;
        if (c == 0) a.moments[2 * COUT] = tot_n;
        return;
      }
      const st::BnFinal f = st::bn_finalize(tot_m, tot_q, gm, bt, rm, rv, (float)a.inv_m, a.eps, a.momentum, a.unbias);
      a.saved_mean[c] = tot_m;
      a.saved_inv_var[c] = f.inv;
      a.eq[c] = f.scale;
      a.eq[COUT + c] = f.bias;
      a.running_mean[c] = f.run_mean;
      a.running_var[c] = f.run_var;
    }
  }
}

template <int KIND, int NCH, int NOUT, int U, bool WRES, bool BF16>
__global__ void __launch_bounds__(Roles<KIND>::kThreads, 1)
    halo_conv_kernel(const __grid_constant__ CUtensorMap map_x,
                     const __grid_constant__ CUtensorMap map_w, const ConvArgs a) {
  using R = Roles<KIND>;
  constexpr int kThreads = R::kThreads;
  constexpr bool kPersist = KIND == kKindFpropApply;
  static_assert(!kPersist || kPersistMaxUnits * U * NOUT <= 512, "persistent accumulators");
  constexpr int kTmemCols = kPersist ? 512 : pow2_at_least(2 * U * NOUT);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const HaloGeom& g = a.g;
  const Layout L = layout(g, KIND, NCH, NOUT, WRES);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t halo_addr = sbase;
  const uint32_t w_addr = sbase + L.off_w;
  const uint32_t bar0 = sbase + L.off_bar;
  const uint32_t bar_halo_full = bar0;
  const uint32_t bar_halo_empty = bar0 + 16;
  const uint32_t bar_acc_full = bar0 + 32;
  const uint32_t bar_acc_empty = bar0 + 48;
  const uint32_t bar_w_full = bar0 + 64;
  const uint32_t bar_w_empty = bar_w_full + 8 * L.nsw;
  const uint32_t bar_drain = bar_w_empty + 8 * L.nsw;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.off_bar + (8 + 2 * L.nsw + 1) * 8);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile uint32_t* ticket_slot = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rs = g.r * g.s;
  const int rows_img = g.p * g.wp;
  // FpropApply: the ready word as this launch found it (the last CTA changes it only after
  // every CTA has taken its finalize ticket, so after every CTA has read it here)
  const uint32_t gen0 = kPersist && threadIdx.x == 0 ? ld_acquire_gpu(a.ready) : 0u;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_halo_full + 8 * i, 1);
      mbar_init(bar_halo_empty + 8 * i, 1);
      mbar_init(bar_acc_full + 8 * i, 1);
      // (FpropApply: acc_full and acc_empty are four one-shot unit barriers, bar_acc_full + 8k)
      mbar_init(bar_acc_empty + 8 * i, kPersist ? 1 : kEpiWarps);  // one arrival per epilogue warp
    }
    for (int i = 0; i < L.nsw; ++i) {
      mbar_init(bar_w_full + 8 * i, 1);
      mbar_init(bar_w_empty + 8 * i, 1);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if constexpr (KIND == kKindFpropBn) {
    // inference BatchNorm folded into the epilogue: one thread per output channel
    float* st = reinterpret_cast<float*>(smem + L.off_bn);
    for (int c = threadIdx.x; c < NOUT; c += kThreads) {
      const bool ok = c < a.out_c;
      const float sc = ok ? a.bn_gamma[c] * rsqrtf(a.bn_var[c] + a.eps) : 0.f;
      const float b = ok && a.conv_bias ? a.conv_bias[c] : 0.f;
      st[c] = sc;
      st[NOUT + c] = ok ? fmaf(b - a.bn_mean[c], sc, a.bn_beta[c]) : 0.f;
    }
  }
  if (warp == R::kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp < R::kAWarps) {
    // ------------------------------------------------------------ A producer
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
          if (!mbar_wait_backoff(bar_halo_empty + 8 * s, ph ^ 1, 128)) {
            set_abort(abort_flag, a.err, kErrWaitHalo);
            break;
          }
          mbar_arrive_expect_tx(bar_halo_full + 8 * s, tx);
          // several smaller boxes in flight instead of one large one (lower latency)
          for (int r0 = 0; r0 < g.hr; r0 += g.box_rows)
            tma_load_4d(halo_addr + s * L.halo_stride + (uint32_t)r0 * g.wp * 128, &map_x, ch * 64,
                        -g.pad, h_lo + r0, n, bar_halo_full + 8 * s);
        }
      }
      // never leave the CTA with a copy in flight
      for (uint32_t k = (it > 2 ? it - 2 : 0); k < it; ++k)
        mbar_wait(bar_halo_full + 8 * (k & 1), (k >> 1) & 1);
    }
  } else if (warp == R::kWWarp) {
    // ------------------------------------------------------------ filter producer
    if (lane == 0) {
      prefetch_tensormap(&map_w);
      auto load_slab = [&](uint32_t dst, int ch, int tap, uint32_t bar) {
        mbar_arrive_expect_tx(bar, L.wslab);
        if constexpr (is_forward_kind(KIND)) {
          tma_load_3d(dst, &map_w, ch * 64, tap, 0, bar);
        } else {
          const int ftap = rs - 1 - tap;  // (R-1-r, S-1-s)
#pragma unroll
          for (int at = 0; at < (NOUT > 64 ? NOUT / 64 : 1); ++at)
            tma_load_3d(dst + at * 8192, &map_w, at * 64, ftap, ch * 64, bar);
        }
      };
      if (WRES) {
        for (int i = 0; i < NCH * rs; ++i) load_slab(w_addr + i * L.wslab, i / rs, i % rs, bar_w_full + 8 * i);
        for (int i = 0; i < NCH * rs; ++i) mbar_wait(bar_w_full + 8 * i, 0);
      } else {
        uint32_t it = 0;
        bool bad = false;
        for (int u = blockIdx.x; u < g.total_units && !is_aborted(abort_flag) && !bad; u += gridDim.x) {
          for (int ch = 0; ch < NCH && !bad; ++ch)
            for (int tap = 0; tap < rs; ++tap, ++it) {
              const uint32_t s = it % kStreamStages, ph = (it / kStreamStages) & 1;
              if (!mbar_wait_backoff(bar_w_empty + 8 * s, ph ^ 1, 64)) {
                set_abort(abort_flag, a.err, kErrWaitWeights);
                bad = true;
                break;
              }
              load_slab(w_addr + s * L.wslab, ch, tap, bar_w_full + 8 * s);
            }
        }
        for (uint32_t k = (it > kStreamStages ? it - kStreamStages : 0); k < it; ++k)
          mbar_wait(bar_w_full + 8 * (k % kStreamStages), (k / kStreamStages) & 1);
      }
    }
  } else if (warp == R::kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop in converged control flow, so all descriptor
    // arithmetic is warp-uniform, and one elected lane issues each tcgen05.mma and commit.
    // (Issued from a single lane under a divergent branch, the same sequence ran 20-35%
    // slower.)  Every decision that changes control flow is voted across the warp, so the
    // lanes can never part (a full-mask elect.sync with absent lanes would not return).  The
    // sequence is also kept free of runtime conditions: a guard beside each MMA halves the
    // rate.
    {
      constexpr bool kBMn = !is_forward_kind(KIND);
      const uint32_t idesc = make_idesc_f16(128, NOUT, BF16, false, kBMn);
      const uint64_t b_base = kBMn ? make_sw128_desc(w_addr, 8192, 1024, 0) : make_sw128_desc(w_addr, 16, 1024, 0);
      const uint64_t a_row_skip = (uint64_t)((g.wp - g.s) * 128 / 16);  // end of a filter row
      bool bad = false;
      if (WRES) {
        // resident filter: every slab is waited for once, before the first unit
        for (int i = 0; i < NCH * rs && !bad; ++i)
          if (!__all_sync(0xffffffffu, mbar_wait(bar_w_full + 8 * i, 0))) {
            set_abort(abort_flag, a.err, kErrWaitWeights);
            bad = true;
          }
        tc_fence_after();
      }
      uint32_t hit = 0, wit = 0, ait = 0;
      for (int u = blockIdx.x; u < g.total_units && !bad; u += gridDim.x) {
        // another role's failed wait is noticed every 8 units (a vote per unit costs
        // issue time that the tensor pipe then waits for)
        if ((ait & 7) == 7 && __any_sync(0xffffffffu, is_aborted(abort_flag))) break;
        const int n = u / g.upi;
        const int m0 = (u - n * g.upi) * g.um;
        const int off = m0 - (m0 / g.wp) * g.wp;
        const int ntiles = min(U, (rows_img - m0 + 127) / 128);
        const uint32_t as = ait & 1, aph = (ait >> 1) & 1;
        // the accumulator stage and the first halo are tested back to back (their latencies
        // overlap); only when one is not complete yet are they waited for one by one
        // (FpropApply: every unit has its own accumulator columns, nothing to wait for)
        const bool ready = __all_sync(0xffffffffu, (kPersist || mbar_test(bar_acc_empty + 8 * as, aph ^ 1)) &
                                                       mbar_test(bar_halo_full + 8 * (hit & 1), (hit >> 1) & 1));
        if (!kPersist && !ready && !__all_sync(0xffffffffu, mbar_wait(bar_acc_empty + 8 * as, aph ^ 1))) {
          set_abort(abort_flag, a.err, kErrWaitAccum);
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem_base + (kPersist ? ait : as) * (U * NOUT);
        for (int ch = 0; ch < NCH && !bad; ++ch, ++hit) {
          const uint32_t hs = hit & 1, hph = (hit >> 1) & 1;
          if (!(ch == 0 && ready) && !__all_sync(0xffffffffu, mbar_wait(bar_halo_full + 8 * hs, hph))) {
            set_abort(abort_flag, a.err, kErrWaitHalo);
            bad = true;
            break;
          }
          tc_fence_after();
          const uint32_t hbase = halo_addr + hs * L.halo_stride;
          // taps advance the A start address incrementally (one 128-byte row per tap, plus the
          // rest of the padded row at the end of a filter row)
          // NT tiles; RS taps at compile time for 3x3 and 1x1 filters (0: the runtime r*s)
          auto run_taps = [&](auto nt_c, auto rs_c) {
            constexpr int NT = decltype(nt_c)::value, RS = decltype(rs_c)::value;
            uint64_t a_tap = make_sw128_desc(hbase + (uint32_t)off * 128u, 16, 1024, 0);
            int sx = 0;
            // With several input-channel chunks the fully unrolled issue code no longer stays in
            // the instruction cache; the forward then issues one tap per loop iteration (7-8%
            // faster there, and slightly slower for a single chunk or the data gradient).
#pragma unroll(is_forward_kind(KIND) && NCH > 1 ? 1 : 9)
            for (int tap = 0; tap < (RS ? RS : rs); ++tap) {
              uint32_t wslab_off, ws = 0;
              if (WRES) {
                wslab_off = (uint32_t)(ch * rs + tap) * L.wslab;
              } else {
                ws = wit % kStreamStages;
                if (!__all_sync(0xffffffffu, mbar_wait(bar_w_full + 8 * ws, (wit / kStreamStages) & 1))) {
                  set_abort(abort_flag, a.err, kErrWaitWeights);
                  bad = true;
                  break;
                }
                tc_fence_after();
                wslab_off = ws * L.wslab;
              }
              const uint64_t b_tap = b_base + (uint64_t)(wslab_off >> 4);
              const uint32_t acc0 = (ch | tap) != 0 ? 1u : 0u;
#pragma unroll
              for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_f16_ss_warp(d0 + t * NOUT, a_tap + (uint64_t)((t * 128 * 128 + kk * 32) >> 4),
                             b_tap + (uint64_t)((kBMn ? kk * 2048 : kk * 32) >> 4), idesc, kk ? 1u : acc0);
              const bool wrap = sx + 1 == g.s;
              sx = wrap ? 0 : sx + 1;
              a_tap += wrap ? 8 + a_row_skip : 8;
              if (!WRES) {
                mma_commit_warp(bar_w_empty + 8 * ws);
                ++wit;
              }
            }
          };
          auto run_rs = [&](auto nt_c) {
            if (rs == 9)
              run_taps(nt_c, std::integral_constant<int, 9>{});
            else if (rs == 1)
              run_taps(nt_c, std::integral_constant<int, 1>{});
            else
              run_taps(nt_c, std::integral_constant<int, 0>{});
          };
          if (ntiles == U)
            run_rs(std::integral_constant<int, U>{});
          else
            run_rs(std::integral_constant<int, 1>{});  // ragged tail of an image (U = 2 only)
          mma_commit_warp(bar_halo_empty + 8 * hs);
        }
        if (bad) break;
        mma_commit_warp(kPersist ? bar_acc_full + 8 * ait : bar_acc_full + 8 * as);
        ++ait;
      }
      mma_commit_warp(bar_drain);
      mbar_wait(bar_drain, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    constexpr int kHalves = NOUT >= 64 ? 2 : 1;
    constexpr int kCPH = NOUT / kHalves;        // channels per half
    constexpr int kSB = kCPH < 32 ? kCPH : 32;  // channels per reduce block
    constexpr int kNB = kCPH / kSB;             // reduce blocks per half
    constexpr int kSh = kSB == 32 ? 0 : 1;      // lane -> channel shift after reduce-scatter
    const int ew = warp - R::kEpiWarp0;         // 0..7
    const int quad = warp & 3;                  // TMEM lanes 32*quad .. +31
    const int half = ew >> 2;
    const int e = quad * 32 + lane;             // M-tile row owned by this thread
    float s1[kNB], s2[kNB];
#pragma unroll
    for (int b = 0; b < kNB; ++b) s1[b] = s2[b] = 0.f;
    // Statistics (moments, stats.cuh): with at most 32 channels per thread, each thread keeps
    // the running mean and M2 of its own rows in registers for the whole kernel and the warp
    // merge runs once at the end (shuffles share the shared-memory pipe with the tensor cores'
    // operand reads); otherwise every tile is merged across the warp as it is produced.
    constexpr bool kRegStats = kCPH <= 32;
    // r1, r2: running mean and M2 of this thread's rows (Welford), rn: their count
    float r1[kRegStats ? kCPH : 1], r2[kRegStats ? kCPH : 1];
    float rn = 0.f;
#pragma unroll
    for (int i = 0; i < (kRegStats ? kCPH : 1); ++i) r1[i] = r2[i] = 0.f;
    float sn = 0.f;  // rows merged into s1 / s2 (the mean and M2 of channel lane >> kSh)
    const bool stats = kPersist || (KIND == kKindFprop && a.mode == kFpropStats);
    const bool bias_relu = KIND == kKindFprop && a.mode == kFpropBiasRelu;
    const float* bn_st = reinterpret_cast<const float*>(smem + L.off_bn);  // kKindFpropBn: [scale][shift]
    const int out_c = a.out_c;
    const size_t opitch = (size_t)out_c * 2;
    // 32-byte stores when every 16-channel group of a row is whole and aligned
    const bool v8 = (out_c % 16) == 0 && (reinterpret_cast<uintptr_t>(a.out) & 31) == 0;
    uint8_t* obase = static_cast<uint8_t*>(a.out);
    uint32_t ait = 0;
    for (int u = blockIdx.x; u < g.total_units && !is_aborted(abort_flag); u += gridDim.x) {
      const int n = u / g.upi;
      const int m0 = (u - n * g.upi) * g.um;
      const int ntiles = min(U, (rows_img - m0 + 127) / 128);
      const uint32_t as = ait & 1, aph = (ait >> 1) & 1;
      if (!mbar_wait_backoff(kPersist ? bar_acc_full + 8 * ait : bar_acc_full + 8 * as, kPersist ? 0u : aph, 256)) {
        set_abort(abort_flag, a.err, kErrWaitMma);
        break;
      }
      tc_fence_after();
      const uint32_t acol = (kPersist ? ait : as) * (U * NOUT);  // the unit's accumulator columns
      // Each thread owns one accumulator row (an output pixel) and kCPH channels of it: the
      // values go from TMEM to registers to HBM without a shared-memory round trip (shared
      // memory bandwidth is what the tensor cores' operand reads need).
      for (int t = 0; t < ntiles; ++t) {
        const int m = m0 + t * 128 + e;
        const int p = m / g.wp, q = m - p * g.wp;
        const bool valid = (p < g.p) && (q < g.q);
        uint8_t* orow = obase + (size_t)(((long long)n * g.p + p) * g.q + q) * opitch;
        if (half < kHalves) {
#pragma unroll
          for (int b = 0; b < kNB; ++b) {
            const int c0 = half * kCPH + b * kSB;
            uint32_t r[kSB];
#pragma unroll
            for (int q16 = 0; q16 < kSB / 16; ++q16)
              tmem_ld16(tmem_base + ((uint32_t)(quad * 32) << 16) + acol + t * NOUT + c0 + q16 * 16,
                        *reinterpret_cast<uint32_t(*)[16]>(r + q16 * 16));
            tmem_ld_wait();
            if (!kPersist && t == ntiles - 1 && b == kNB - 1) {
              // the warp's last read of the accumulator stage (a warp-uniform branch): every
              // lane orders its TMEM reads before the warp sync, then one lane arrives
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(bar_acc_empty + 8 * as);
            }
            float v[kSB];
#pragma unroll
            for (int i = 0; i < kSB; ++i) {
              float x = __uint_as_float(r[i]);
              if (bias_relu) x = fmaxf(x + __ldg(a.bias + c0 + i), 0.f);
              if constexpr (KIND == kKindFpropBn) x = fmaxf(fmaf(x, bn_st[c0 + i], bn_st[NOUT + c0 + i]), 0.f);
              v[i] = valid ? x : 0.f;
            }
            if (valid) {
              uint4 pk[kSB / 8];
#pragma unroll
              for (int cc = 0; cc < kSB / 8; ++cc)
                pk[cc] = make_uint4(pack2<BF16>(v[8 * cc + 0], v[8 * cc + 1]), pack2<BF16>(v[8 * cc + 2], v[8 * cc + 3]),
                                    pack2<BF16>(v[8 * cc + 4], v[8 * cc + 5]), pack2<BF16>(v[8 * cc + 6], v[8 * cc + 7]));
              if (v8) {
#pragma unroll
                for (int cc = 0; cc < kSB / 16; ++cc)
                  if (c0 + 16 * cc < out_c) st_global_v8(orow + (c0 + 16 * cc) * 2, pk[2 * cc], pk[2 * cc + 1]);
              } else {
#pragma unroll
                for (int cc = 0; cc < kSB / 8; ++cc)
                  if (c0 + 8 * cc < out_c) st_global_v4(orow + (c0 + 8 * cc) * 2, pk[cc]);
              }
            }
            if (stats) {
              if constexpr (kRegStats) {
                // kNB == 1: one Welford update per valid row
                if (valid) {
                  rn += 1.f;
                  st::welford_row<kSB>(r1 + b * kSB, r2 + b * kSB, v, __fdividef(1.f, rn));
                }
              } else {
                // the tile's rows (each: count 1, mean v, M2 0) merged across the warp, then into
                // the lane's running moments of its channel
                float q0[kSB];
#pragma unroll
                for (int i = 0; i < kSB; ++i) q0[i] = 0.f;
                const float tn = st::chan_scatter<kSB>(v, q0, valid ? 1.f : 0.f, lane);
                float nn = sn;
                st::chan_merge(nn, s1[b], s2[b], tn, v[0], q0[0]);
                if (b == kNB - 1) sn = nn;
              }
            }
          }
        } else if (!kPersist && t == ntiles - 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_acc_empty + 8 * as);
        }
      }
      ++ait;
    }
    if constexpr (kRegStats) {
      if (stats && half < kHalves) {
#pragma unroll
        for (int b = 0; b < kNB; ++b) {
          float v1[kSB], v2[kSB];
#pragma unroll
          for (int i = 0; i < kSB; ++i) {
            v1[i] = r1[b * kSB + i];
            v2[i] = r2[b * kSB + i];
          }
          sn = st::chan_scatter<kSB>(v1, v2, rn, lane);
          s1[b] = v1[0];
          s2[b] = v2[0];
        }
      }
    }
    if (stats && half < kHalves && (lane & ((1 << kSh) - 1)) == 0) {
      // per-(quad) partials -> smem; the staging buffer is free behind the last named barrier
      float* red = reinterpret_cast<float*>(smem + L.off_stage);
#pragma unroll
      for (int b = 0; b < kNB; ++b) {
        const int c = half * kCPH + b * kSB + (lane >> kSh);
        red[(quad * 2 + 0) * NOUT + c] = s1[b];
        red[(quad * 2 + 1) * NOUT + c] = s2[b];
      }
      if (half == 0 && lane == 0) red[8 * NOUT + quad] = sn;  // the quadrant's row count
    }
  }

  tc_fence_before();
  __syncthreads();

  if (kPersist || (KIND == kKindFprop && a.mode == kFpropStats))
    stats_partial_finalize<NOUT, kThreads, 128 * NOUT * 2>(a, reinterpret_cast<const float*>(smem + L.off_stage),
                                                           smem + L.off_stage, ticket_slot, abort_flag);

  if constexpr (kPersist) {
    // The last CTA has written eq (scale, bias); once all its threads are past the finalize it
    // releases the ready word.  Every other CTA waits for the word to change (bounded), then
    // applies BatchNorm and ReLU to its accumulators, which are still in TMEM.
    __syncthreads();
    if (threadIdx.x == 0) {
      if (*ticket_slot == gridDim.x - 1) {
        __threadfence();
        atomicAdd(a.ready, 1u);
      } else {
        const uint64_t t0 = globaltimer_ns();
        while (ld_acquire_gpu(a.ready) == gen0) {
          if (globaltimer_ns() - t0 > kWaitLimitNs) {
            set_abort(abort_flag, a.err, kErrWaitMma);
            break;
          }
          __nanosleep(128);
        }
      }
    }
    __syncthreads();
    constexpr int kHalves = NOUT >= 64 ? 2 : 1;
    constexpr int kCPH = NOUT / kHalves;  // 32: one 32-bit mask word per row and half
    static_assert(kCPH == 32, "persistent apply: 32 channels per epilogue thread");
    if (warp >= R::kEpiWarp0 && !is_aborted(abort_flag)) {
      const int ew = warp - R::kEpiWarp0;
      const int quad = warp & 3;
      const int half = ew >> 2;
      const int e = quad * 32 + lane;
      if (half < kHalves) {
        const int c0 = half * kCPH;
        float sc[kCPH], bi[kCPH];
#pragma unroll
        for (int i = 0; i < kCPH; ++i) {
          sc[i] = __ldcg(a.eq + c0 + i);
          bi[i] = __ldcg(a.eq + NOUT + c0 + i);
        }
        const size_t opitch = (size_t)NOUT * 2;
        uint8_t* ybase = static_cast<uint8_t*>(a.y);
        uint32_t k = 0;
        for (int u = blockIdx.x; u < g.total_units; u += gridDim.x, ++k) {
          const int n = u / g.upi;
          const int m0 = (u - n * g.upi) * g.um;
          const int ntiles = min(U, (rows_img - m0 + 127) / 128);
          for (int t = 0; t < ntiles; ++t) {
            const int m = m0 + t * 128 + e;
            const int p = m / g.wp, q = m - p * g.wp;
            const bool valid = (p < g.p) && (q < g.q);
            uint32_t r[kCPH];
            tmem_ld16(tmem_base + ((uint32_t)(quad * 32) << 16) + k * (U * NOUT) + t * NOUT + c0,
                      *reinterpret_cast<uint32_t(*)[16]>(r));
            tmem_ld16(tmem_base + ((uint32_t)(quad * 32) << 16) + k * (U * NOUT) + t * NOUT + c0 + 16,
                      *reinterpret_cast<uint32_t(*)[16]>(r + 16));
            tmem_ld_wait();
            if (!valid) continue;
            // the accumulator rounded to the storage dtype, as the stored z the apply pass of
            // the two-kernel forward reads: both forms give the same y and mask
            float yv[kCPH];
            uint32_t bits = 0;
#pragma unroll
            for (int i = 0; i < kCPH; i += 2) {
              const float2 zz = unpack2<BF16>(pack2<BF16>(__uint_as_float(r[i]), __uint_as_float(r[i + 1])));
              const float p0 = fmaf(zz.x, sc[i], bi[i]);
              const float p1 = fmaf(zz.y, sc[i + 1], bi[i + 1]);
              bits |= (p0 > 0.f ? 1u : 0u) << i;  // CMP_GT: 0 at pre == 0
              bits |= (p1 > 0.f ? 1u : 0u) << (i + 1);
              yv[i] = fmaxf(p0, 0.f);
              yv[i + 1] = fmaxf(p1, 0.f);
            }
            const long long pix = ((long long)n * g.p + p) * g.q + q;
            uint8_t* yrow = ybase + (size_t)pix * opitch;
#pragma unroll
            for (int cc = 0; cc < kCPH / 16; ++cc) {
              const uint4 lo = make_uint4(pack2<BF16>(yv[16 * cc + 0], yv[16 * cc + 1]), pack2<BF16>(yv[16 * cc + 2], yv[16 * cc + 3]),
                                          pack2<BF16>(yv[16 * cc + 4], yv[16 * cc + 5]), pack2<BF16>(yv[16 * cc + 6], yv[16 * cc + 7]));
              const uint4 hi = make_uint4(pack2<BF16>(yv[16 * cc + 8], yv[16 * cc + 9]), pack2<BF16>(yv[16 * cc + 10], yv[16 * cc + 11]),
                                          pack2<BF16>(yv[16 * cc + 12], yv[16 * cc + 13]), pack2<BF16>(yv[16 * cc + 14], yv[16 * cc + 15]));
              st_global_v8(yrow + (c0 + 16 * cc) * 2, lo, hi);
            }
            if (a.mask) a.mask[(pix * NOUT + c0) >> 5] = bits;
          }
        }
      }
    }
    tc_fence_before();
    __syncthreads();
  }

  if (warp == R::kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// Host: geometry of a stride-1 halo conv (fills wp, p, q, hr, upi, total_units, um).
inline bool finish_geom(HaloGeom& g, int U) {
  g.um = U * 128;
  g.wp = g.w + 2 * g.pad;
  g.p = g.h + 2 * g.pad - g.r + 1;
  g.q = g.w + 2 * g.pad - g.s + 1;
  if (g.p <= 0 || g.q <= 0 || g.wp > 256) return false;
  g.hr = (g.wp - 1 + g.um - 1 + (g.r - 1) * g.wp + g.s - 1) / g.wp + 1;
#ifndef CBR_HALO_BOX_ROWS
#define CBR_HALO_BOX_ROWS 1
#endif
  g.box_rows = CBR_HALO_BOX_ROWS < g.hr ? CBR_HALO_BOX_ROWS : g.hr;
  g.hr = (g.hr + g.box_rows - 1) / g.box_rows * g.box_rows;
  if (g.hr > 256) return false;
  g.upi = (g.p * g.wp + g.um - 1) / g.um;
  g.total_units = g.n_img * g.upi;
  return true;
}

template <int KIND, int NCH, int NOUT, int U, bool WRES, bool BF16>
int launch_halo_conv(const ConvArgs& a, const CUtensorMap& mx, const CUtensorMap& mw, int grid,
                     cudaStream_t st) {
  auto kern = halo_conv_kernel<KIND, NCH, NOUT, U, WRES, BF16>;
  const Layout L = layout(a.g, KIND, NCH, NOUT, WRES);
  const uint32_t smem = L.total + 1024;
  if (smem > 227 * 1024) return 3;
  if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), 227 * 1024)) return 6;
  if constexpr (KIND == kKindFpropApply) {
    // every CTA waits for the last one: a cooperative launch, which the runtime refuses unless
    // the whole grid is resident at once
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(Roles<KIND>::kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, mx, mw, a) == cudaSuccess ? 0 : 6;
  }
  kern<<<grid, Roles<KIND>::kThreads, smem, st>>>(mx, mw, a);
  return cudaGetLastError() == cudaSuccess ? 0 : 6;
}

}  // namespace hc
}  // namespace cbr
