// Batch statistics of the convolution output as running moments (count n, mean, M2 = sum of
// squared deviations from the mean), so the variance M2/M never comes from the difference
// E[z^2] - mean^2, which cancels when |mean| is large against the standard deviation (BatchNorm
// CUDA page, section 4.3, numerical stability and Welford's algorithm).
//   - each epilogue thread updates the moments of its own rows one row at a time (Welford:
//     d = v - mean; mean += d/n; M2 += d*(v - mean));
//   - partial moments are combined pairwise (Chan, Golub and LeVeque's parallel formula:
//     n = na + nb, d = mean_b - mean_a, mean = mean_a + d*nb/n, M2 = M2a + M2b + d^2*na*nb/n)
//     across the lanes of a warp, the lane quadrants of a CTA and the CTAs of the grid, always in
//     the same order, so the result is deterministic.
#pragma once
#include "common.cuh"

namespace cbr {
namespace st {

// Two fp32 lanes in one 64-bit register, and the packed arithmetic of sm_100+ on them
// (one instruction for both lanes).
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t sub_x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma_x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// Welford update of N channels (N even) with one new row v; rn = 1/n after counting the row.
// Channels go in pairs through the packed fp32x2 pipe: four instructions per two channels.
template <int N>
__device__ __forceinline__ void welford_row(float* mean, float* m2, const float* v, float rn) {
  static_assert(N % 2 == 0, "channel pairs");
  const uint64_t r2 = pk2(rn, rn);
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    const uint64_t vv = pk2(v[i], v[i + 1]);
    uint64_t mv = pk2(mean[i], mean[i + 1]);
    uint64_t qv = pk2(m2[i], m2[i + 1]);
    const uint64_t d = sub_x2(vv, mv);  // v - mean
    mv = fma_x2(d, r2, mv);             // mean += d / n
    qv = fma_x2(d, sub_x2(vv, mv), qv); // M2 += d * (v - mean)
    upk2(mv, mean[i], mean[i + 1]);
    upk2(qv, m2[i], m2[i + 1]);
  }
}

// Merge weights of two sets of na and nb rows: fb = nb / (na + nb) and g = na * nb / (na + nb)
// (both 0 when the union is empty).  They depend only on the counts, which a lane, a thread
// or a CTA shares across all its channels, so they are computed once per merge step.
struct ChanW {
  float fb, g;
};
__device__ __forceinline__ ChanW chan_weights(float na, float nb) {
  // Counts are whole numbers, so the union is empty (nb = 0, fb = 0) or has n >= 1: a fast
  // division by max(n, 1) (2 ulp) never meets 0/0, whose IEEE special-case path is slow.
  const float fb = __fdividef(nb, fmaxf(na + nb, 1.f));
  return ChanW{fb, na * fb};
}

// (ma, qa) <- the mean and M2 of the union of a and b (a first), given their weights.  Empty
// moments are (0, 0) with count 0, so an empty side needs no branch: fb = 1 takes b's mean
// exactly (ma = 0), fb = 0 keeps a's, and g = 0 adds no cross term.
__device__ __forceinline__ void chan_merge_w(float& ma, float& qa, float mb, float qb, ChanW w) {
  const float d = mb - ma;
  ma = fmaf(d, w.fb, ma);
  qa = fmaf(d * d, w.g, qa + qb);
}

// (na, ma, qa) <- the moments of the union of a and b (a first).
__device__ __forceinline__ void chan_merge(float& na, float& ma, float& qa, float nb, float mb, float qb) {
  chan_merge_w(ma, qa, mb, qb, chan_weights(na, nb));
  na += nb;
}

// Warp merge-scatter, the moments counterpart of a reduce-scatter: on entry each lane holds the
// moments of L channels over its own rows (count n, the same for all its channels); on exit
// mean[0], m2[0] of every lane hold the moments over the 32 lanes of channel (lane >> s),
// s = log2(32 / L), and the return value is the merged count.  Each butterfly step merges the
// lower lane's moments with the upper lane's (a first), so both partners of the final steps
// compute the same values.
template <int L>
__device__ __forceinline__ float chan_scatter(float (&mean)[L], float (&m2)[L], float n, int lane) {
  int o = 16;
#pragma unroll
  for (int len = L; len > 1; len >>= 1, o >>= 1) {
    const bool hi = (lane & o) != 0;
    const float pn = __shfl_xor_sync(0xffffffffu, n, o);
    const ChanW w = chan_weights(hi ? pn : n, hi ? n : pn);
#pragma unroll
    for (int j = 0; j < len / 2; ++j) {
      const float send_m = hi ? mean[j] : mean[j + len / 2];
      const float send_q = hi ? m2[j] : m2[j + len / 2];
      const float keep_m = hi ? mean[j + len / 2] : mean[j];
      const float keep_q = hi ? m2[j + len / 2] : m2[j];
      const float rm = __shfl_xor_sync(0xffffffffu, send_m, o);
      const float rq = __shfl_xor_sync(0xffffffffu, send_q, o);
      // lower lane's moments first
      float am = hi ? rm : keep_m, aq = hi ? rq : keep_q;
      chan_merge_w(am, aq, hi ? keep_m : rm, hi ? keep_q : rq, w);
      mean[j] = am;
      m2[j] = aq;
    }
    n += pn;
  }
#pragma unroll
  for (; o >= 1; o >>= 1) {
    const bool hi = (lane & o) != 0;
    const float pn = __shfl_xor_sync(0xffffffffu, n, o);
    const float rm = __shfl_xor_sync(0xffffffffu, mean[0], o);
    const float rq = __shfl_xor_sync(0xffffffffu, m2[0], o);
    const ChanW w = chan_weights(hi ? pn : n, hi ? n : pn);
    float am = hi ? rm : mean[0], aq = hi ? rq : m2[0];
    chan_merge_w(am, aq, hi ? mean[0] : rm, hi ? m2[0] : rq, w);
    mean[0] = am;
    m2[0] = aq;
    n += pn;
  }
  return n;
}

// Floats of one CTA's partial statistics: means [C], M2 [C], then the row count and padding.
__host__ __device__ constexpr int partial_floats(int c) { return 2 * c + 4; }

// ------------------------------------------------------------------ grid merge and finalize
// Every kernel that merges the grid's partial moments (the convolution's last CTA, the
// persistent forward, the apply pass) runs the same merge, so the statistics and y come out
// bit-identical whichever kernel merged them.  The row-group count kRG depends on the channel
// count alone (a power of two that divides 32): thread t < kRG * C/4 takes row group t % kRG of
// float4 column t / kRG, so the kRG groups of a column are kRG consecutive lanes of one warp.
// Group r merges partials r, r + kRG, r + 2 kRG, ... in order; a fixed pairwise tree then merges
// the groups across those lanes (step w: lane r, r % 2w == 0, takes in lane r + w, r first).
template <int C>
__host__ __device__ constexpr int merge_groups() {
  return 1024 / C < 16 ? 1024 / C : 16;
}
template <int C>
__host__ __device__ constexpr int merge_threads() {
  return merge_groups<C>() * (C / 4);
}
// Working set of the merge: the merged means [C], M2s [C] and the row count.
template <int C>
__host__ __device__ constexpr int merge_scratch_floats() {
  return partial_floats(C);
}

// Merge `nparts` partial moments into scratch[0 .. 2C): means, then M2s; returns the total row
// count.  Every thread of the block calls it (it synchronises the block once); `load(b, c4, m,
// q, n)` fetches float4 column c4 of partial b's means and M2s and its row count.  kLd partials
// of a thread are loaded before the first is merged (the merge order does not depend on it).
template <int C, int kThreads, int kLd, class Load>
__device__ float merge_partials(int nparts, float* scratch, Load load) {
  constexpr int kV = C / 4;
  constexpr int kRG = merge_groups<C>();
  static_assert(kThreads >= merge_threads<C>() && kThreads >= C, "merge threads");
  static_assert(32 % kRG == 0 && merge_threads<C>() % 32 == 0, "row groups within whole warps");
  if (threadIdx.x < merge_threads<C>()) {
    const int rg = threadIdx.x % kRG, c4 = threadIdx.x / kRG;
    float n = 0.f;
    float m[4] = {0.f, 0.f, 0.f, 0.f}, q[4] = {0.f, 0.f, 0.f, 0.f};
    for (int b0 = rg; b0 < nparts; b0 += kLd * kRG) {
      float4 vm[kLd], vq[kLd];
      float vn[kLd];
#pragma unroll
      for (int k = 0; k < kLd; ++k) {
        const int b = b0 + k * kRG;
        if (b < nparts) {
          load(b, c4, vm[k], vq[k], vn[k]);
        } else {
          vm[k] = vq[k] = make_float4(0.f, 0.f, 0.f, 0.f);
          vn[k] = 0.f;
        }
      }
#pragma unroll
      for (int k = 0; k < kLd; ++k) {
        const float bm[4] = {vm[k].x, vm[k].y, vm[k].z, vm[k].w};
        const float bq[4] = {vq[k].x, vq[k].y, vq[k].z, vq[k].w};
        const ChanW w = chan_weights(n, vn[k]);  // one division for the 4 channels
#pragma unroll
        for (int j = 0; j < 4; ++j) chan_merge_w(m[j], q[j], bm[j], bq[j], w);
        n += vn[k];
      }
    }
#pragma unroll
    for (int w = 1; w < kRG; w *= 2) {
      const float pn = __shfl_down_sync(0xffffffffu, n, w, kRG);
      float pm[4], pq[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        pm[j] = __shfl_down_sync(0xffffffffu, m[j], w, kRG);
        pq[j] = __shfl_down_sync(0xffffffffu, q[j], w, kRG);
      }
      if ((rg & (2 * w - 1)) == 0) {
        const ChanW cw = chan_weights(n, pn);
#pragma unroll
        for (int j = 0; j < 4; ++j) chan_merge_w(m[j], q[j], pm[j], pq[j], cw);
        n += pn;
      }
    }
    if (rg == 0) {
      reinterpret_cast<float4*>(scratch)[c4] = make_float4(m[0], m[1], m[2], m[3]);
      reinterpret_cast<float4*>(scratch + C)[c4] = make_float4(q[0], q[1], q[2], q[3]);
      if (c4 == 0) scratch[2 * C] = n;
    }
  }
  __syncthreads();
  return scratch[2 * C];
}

// BatchNorm finalize of one channel from its batch mean and M2 over M rows (inv_m = 1/M):
// var = M2/M (biased), inv = 1/sqrt(var + eps), eq_scale = gamma*inv, eq_bias = beta -
// eq_scale*mean; the running statistics move by `momentum` towards the batch mean and the
// unbiased variance (BatchNorm CUDA page, sections 2 and 3).  Explicit roundings, so that every
// kernel computes the same bits.
struct BnFinal {
  float inv, scale, bias, run_mean, run_var;
};
__device__ __forceinline__ BnFinal bn_finalize(float mean, float m2, float gamma, float beta, float run_mean,
                                               float run_var, float inv_m, float eps, float momentum, float unbias) {
  BnFinal f;
  const float var = fmaxf(__fmul_rn(m2, inv_m), 0.f);
  f.inv = rsqrtf(__fadd_rn(var, eps));
  f.scale = __fmul_rn(gamma, f.inv);
  f.bias = __fmaf_rn(-f.scale, mean, beta);
  const float keep = __fsub_rn(1.f, momentum);
  f.run_mean = __fmaf_rn(keep, run_mean, __fmul_rn(momentum, mean));
  f.run_var = __fmaf_rn(keep, run_var, __fmul_rn(__fmul_rn(momentum, var), unbias));
  return f;
}

}  // namespace st
}  // namespace cbr
