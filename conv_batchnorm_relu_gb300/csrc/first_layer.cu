// First-layer convolution: the CBR block that takes the 3-channel image (Tech-Renaissance CBR
// page, section 5.3: the first layer's backward skips DGrad, because its input is the training
// data).  The 7x7 stride-2 padding-3 shape is the standard image stem these kernels are tuned
// for.  A 3-channel pixel is 6 bytes, so the input cannot be the innermost dimension of a TMA
// tile or an MMA operand row; two designs handle it:
//   - implicit im2col (the main path, stride 1 or 2; first_fprop_imp_kernel and
//     first_wgrad_imp_kernel): every input row is padded to 16-byte groups of 8/stride channel
//     slots per pixel, and each filter row's im2col tile is read straight out of the padded
//     row through an unswizzled descriptor whose core matrices overlap (no tile is assembled);
//   - builder warps (other strides, and the weight gradient at Cout other than 64;
//     first_fprop_kernel and first_wgrad_kernel): whole input rows are staged in shared memory
//     and four warps assemble an im2col tile with K slot r*24 + s*3 + c (each filter row a
//     24-slot segment, three 128-byte K atoms, K <= 192).
// Forward: z = im2col(x) * W^T on the tensor cores, with the epilogue of the other convolutions
// (statistics in registers, direct stores).  WGrad: dW^T = im2col(x)^T * dz, with the same
// operand read MN-major.
#include <algorithm>
#include <type_traits>

#include "halo_conv.cuh"

namespace cbr {
namespace {

constexpr int kFlAtoms = 3;                          // 192 K slots
constexpr uint32_t kFlAtomBytes = 128 * 128;         // 128 rows x 128 B
constexpr uint32_t kFlTile = kFlAtoms * kFlAtomBytes;
constexpr int kFlBuildWarps = 4;
constexpr int kFlEpiWarp0 = 6;                       // warp 0: x TMA, 1-4: builders, 5: MMA
constexpr int kFlThreads = (kFlEpiWarp0 + 8) * 32;   // 448
constexpr int kFlXStages = 4;                        // staged input rows in flight

struct FirstGeom {
  int n_img, h, w;       // x [n][h][w][3]
  int p, q;              // output rows and columns (q <= 128)
  int r, s, stride, pad; // r, s <= 8
  int units;             // n_img * p
  int rowp;              // bytes per staged row: 64-byte zero margin, the row, a zero tail
  int nk;                // MMA K steps: ceil(r*24/16)
  int tma;               // input rows staged by TMA (row pitch a multiple of 16 bytes), else by warp 0
  // implicit-im2col forward (stride 1 or 2): input rows padded to 16-byte pixel groups
  int imp;               // the geometry fits the implicit path
  int gpx;               // pixels per 16-byte group (= stride)
  int cpx;               // channel slots per pixel (8 / gpx; 3 values then zeros)
  int jm;                // groups of left margin: ceil(pad / gpx)
  int lead;              // zero-weight pixels ahead of tap 0 in a run: gpx*jm - pad
  int nmr;               // MMAs per filter row (two groups = K 16 each)
  int rowb;              // bytes per padded row: (128 + 2*nmr) groups
  int xal4;              // x is 4-byte aligned
  int rawtma;            // input rows copied whole into shared memory (row bytes and x 16-byte aligned)
  int rawb;              // bytes of one such row (w * 6)
};

__host__ __device__ inline uint32_t fl_xstage_bytes(const FirstGeom& g) {
  return ((uint32_t)g.r * g.rowp + 1023u) & ~1023u;
}

// Staged input rows: row rr of a unit (input row p*stride - pad + rr) sits at rr*rowp + 64
// bytes, contiguous over W*3 elements, with zeros before it (the margin covers the left
// padding) and after it (TMA out-of-bounds fill, or never written) and zeros throughout when
// the input row is outside the image.  With TMA the x tensor is viewed in 8-byte units, so one
// box {rowp/8 units starting 8 units before the row, R rows} stages a whole unit.  So the S*3 values of filter row rr for output pixel q
// are one contiguous run that needs no bounds check.
//
// Build the im2col tile: thread q (< Q) writes row q, one 24-slot segment per filter row (the
// run read as 12 aligned 32-bit words and realigned by a funnel shift, values past S*3 zero).
__device__ __forceinline__ void fl_build_tile(uint32_t a_stage, uint32_t xs, const FirstGeom& g, int q) {
  if (q >= g.q) return;
  const int e0 = (q * g.stride - g.pad) * 3;  // first element of the run, >= -3*pad
  const int nval = g.s * 3;
  uint32_t keep[12];                          // values past S*3 are zero
#pragma unroll
  for (int j = 0; j < 12; ++j) keep[j] = 2 * j >= nval ? 0u : (2 * j + 1 >= nval ? 0xffffu : 0xffffffffu);
  const uint32_t run0 = xs + 64 + 2 * e0;
  const uint32_t sh = (run0 & 2) ? 16u : 0u;
  uint32_t wa = run0 & ~3u;
  // Software-pipelined over filter rows: the next row's words are loaded
  // before this row's stores, so one builder warp per sub-partition keeps
  // its shared-memory loads in flight.
  uint32_t v[13];
#pragma unroll
  for (int j = 0; j < 13; ++j) asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v[j]) : "r"(wa + 4 * j));
  for (int rr = 0; rr < g.r; ++rr) {
    uint32_t o[12];
#pragma unroll
    for (int j = 0; j < 12; ++j) o[j] = __funnelshift_r(v[j], v[j + 1], sh) & keep[j];
    if (rr + 1 < g.r) {
      wa += g.rowp;
#pragma unroll
      for (int j = 0; j < 13; ++j) asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v[j]) : "r"(wa + 4 * j));
    }
#pragma unroll
    for (int cj = 0; cj < 3; ++cj) {
      const int chunk = rr * 3 + cj;
      const uint32_t addr = a_stage + (uint32_t)(chunk >> 3) * kFlAtomBytes + (uint32_t)q * 128u +
                            ((uint32_t)((chunk & 7) ^ (q & 7)) << 4);
      st_shared_v4(addr, make_uint4(o[4 * cj], o[4 * cj + 1], o[4 * cj + 2], o[4 * cj + 3]));
    }
  }
}

// Input rows without TMA (row pitch not a multiple of 16 bytes): the whole warp copies the R
// rows of each unit, zero outside the image, then lane 0 marks the stage full.  Waits are
// voted across the warp so its lanes stay together.
__device__ void fl_stage_rows_plain(const uint16_t* x, const FirstGeom& g, uint16_t* stages, uint32_t xst,
                                    uint32_t bar_x_full, uint32_t bar_x_empty, volatile int* abort_flag,
                                    uint32_t* err) {
  const int lane = threadIdx.x & 31;
  const int row = g.w * 3;
  uint32_t it = 0;
  for (int u = blockIdx.x; u < g.units && !__any_sync(0xffffffffu, hc::is_aborted(abort_flag)); u += gridDim.x, ++it) {
    const int n = u / g.p, p = u - n * g.p;
    const uint32_t s = it % kFlXStages, ph = (it / kFlXStages) & 1;
    if (!__all_sync(0xffffffffu, mbar_wait_backoff(bar_x_empty + 8 * s, ph ^ 1, 64))) {
      hc::set_abort(abort_flag, err, kErrWaitHalo);
      break;
    }
    uint8_t* dst = reinterpret_cast<uint8_t*>(stages) + s * xst;
    for (int i = lane; i < g.r * row; i += 32) {
      const int rr = i / row, e = i - rr * row;
      const int h = p * g.stride - g.pad + rr;
      *reinterpret_cast<uint16_t*>(dst + rr * g.rowp + 64 + 2 * e) =
          (h >= 0 && h < g.h) ? x[((size_t)n * g.h + h) * row + e] : (uint16_t)0;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_x_full + 8 * s);
  }
}

// ------------------------------------------------------------------------------ forward
template <int NOUT, bool BF16>
__global__ void __launch_bounds__(kFlThreads, 1)
    first_fprop_kernel(const __grid_constant__ CUtensorMap map_x, const ConvArgs a, const FirstGeom g,
                       const void* wts, const void* xin) {
  constexpr int kTmemCols = hc::pow2_at_least(2 * NOUT);
  constexpr uint32_t kBBytes = kFlAtoms * NOUT * 128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t xst = fl_xstage_bytes(g);
  const uint32_t off_a = kFlXStages * xst, off_b = off_a + 2 * kFlTile, off_bar = off_b + kBBytes;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + off_bar;
  const uint32_t bar_x_full = bar0, bar_x_empty = bar0 + 32, bar_a_full = bar0 + 64, bar_a_empty = bar0 + 80;
  const uint32_t bar_acc_full = bar0 + 96, bar_acc_empty = bar0 + 112, bar_drain = bar0 + 128;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + off_bar + 136);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile uint32_t* ticket_slot = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // zero the x stages (row margins and tails stay zero) and both A stages (rows >= Q and slots
  // never written stay zero), build the filter tile
  for (uint32_t i = threadIdx.x; i < (off_a + 2 * kFlTile) / 16; i += kFlThreads)
    st_shared_v4(sbase + i * 16, make_uint4(0, 0, 0, 0));
  {
    const uint16_t* wsrc = static_cast<const uint16_t*>(wts);
    for (int i = threadIdx.x; i < NOUT * kFlAtoms * 8; i += kFlThreads) {
      const int n = i / (kFlAtoms * 8), chunk = i - n * (kFlAtoms * 8);
      uint32_t w32[4] = {0, 0, 0, 0};
      const int rr = chunk / 3;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int slot = (chunk - rr * 3) * 8 + e;  // 0..23 within the filter row
        const int sx = slot / 3, c = slot - sx * 3;
        if (rr < g.r && sx < g.s && n < a.out_c) {
          const uint32_t v = wsrc[((n * g.r + rr) * g.s + sx) * 3 + c];
          w32[e >> 1] |= v << ((e & 1) * 16);
        }
      }
      st_shared_v4(sbase + off_b + (uint32_t)(chunk >> 3) * (NOUT * 128) + (uint32_t)n * 128u +
                       ((uint32_t)((chunk & 7) ^ (n & 7)) << 4),
                   make_uint4(w32[0], w32[1], w32[2], w32[3]));
    }
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kFlXStages; ++i) {
      mbar_init(bar_x_full + 8 * i, 1);
      mbar_init(bar_x_empty + 8 * i, kFlBuildWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_a_full + 8 * i, kFlBuildWarps);
      mbar_init(bar_a_empty + 8 * i, 1);
      mbar_init(bar_acc_full + 8 * i, 1);
      mbar_init(bar_acc_empty + 8 * i, hc::kEpiThreads);
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- input-row stager
    if (!g.tma) {
      fl_stage_rows_plain(static_cast<const uint16_t*>(xin), g, reinterpret_cast<uint16_t*>(smem), xst,
                          bar_x_full, bar_x_empty, abort_flag, a.err);
    } else if (lane == 0) {
      prefetch_tensormap(&map_x);
      const uint32_t tx = (uint32_t)g.r * g.rowp;
      uint32_t it = 0;
      for (int u = blockIdx.x; u < g.units && !hc::is_aborted(abort_flag); u += gridDim.x, ++it) {
        const int n = u / g.p, p = u - n * g.p;
        const uint32_t s = it % kFlXStages, ph = (it / kFlXStages) & 1;
        if (!mbar_wait_backoff(bar_x_empty + 8 * s, ph ^ 1, 64)) {
          hc::set_abort(abort_flag, a.err, kErrWaitHalo);
          break;
        }
        mbar_arrive_expect_tx(bar_x_full + 8 * s, tx);
        tma_load_3d(sbase + s * xst, &map_x, -8, p * g.stride - g.pad, n, bar_x_full + 8 * s);
      }
      for (uint32_t k = (it > kFlXStages ? it - kFlXStages : 0); k < it; ++k)
        mbar_wait(bar_x_full + 8 * (k % kFlXStages), (k / kFlXStages) & 1);
    }
  } else if (warp <= kFlBuildWarps) {
    // ---------------------------------------------------------------- im2col builders
    const int tid = threadIdx.x - 32;
    uint32_t it = 0;
    for (int u = blockIdx.x; u < g.units && !hc::is_aborted(abort_flag); u += gridDim.x, ++it) {
      const uint32_t s = it & 1, ph = (it >> 1) & 1;
      const uint32_t sx = it % kFlXStages, phx = (it / kFlXStages) & 1;
      if (!mbar_wait_backoff(bar_a_empty + 8 * s, ph ^ 1, 64) || !mbar_wait(bar_x_full + 8 * sx, phx)) {
        hc::set_abort(abort_flag, a.err, kErrWaitOperand);
        break;
      }
      fl_build_tile(sbase + off_a + s * kFlTile, sbase + sx * xst, g, tid);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar_x_empty + 8 * sx);
        mbar_arrive(bar_a_full + 8 * s);
      }
    }
  } else if (warp == 5) {
    // ---------------------------------------------------------------- MMA issuer (whole warp)
    const uint32_t idesc = make_idesc_f16(128, NOUT, BF16, false, false);
    const uint64_t b_base = make_sw128_desc(sbase + off_b, 16, 1024, 0);
    uint32_t it = 0;
    for (int u = blockIdx.x; u < g.units && !__any_sync(0xffffffffu, hc::is_aborted(abort_flag));
         u += gridDim.x, ++it) {
      const uint32_t s = it & 1, ph = (it >> 1) & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_acc_empty + 8 * s, ph ^ 1) && mbar_wait(bar_a_full + 8 * s, ph))) {
        hc::set_abort(abort_flag, a.err, kErrWaitAccum);
        break;
      }
      tc_fence_after();
      const uint64_t a_base = make_sw128_desc(sbase + off_a + s * kFlTile, 16, 1024, 0);
      const uint32_t d = tmem_base + s * NOUT;
      for (int kk = 0; kk < g.nk; ++kk)
        mma_f16_ss_warp(d, a_base + (uint64_t)(((kk >> 2) * kFlAtomBytes + (kk & 3) * 32) >> 4),
                        b_base + (uint64_t)(((kk >> 2) * (NOUT * 128) + (kk & 3) * 32) >> 4), idesc, kk ? 1u : 0u);
      mma_commit_warp(bar_a_empty + 8 * s);
      mma_commit_warp(bar_acc_full + 8 * s);
    }
    mma_commit_warp(bar_drain);
    mbar_wait(bar_drain, 0);
  } else {
    // ---------------------------------------------------------------- epilogue (8 warps)
    constexpr int kHalves = NOUT >= 64 ? 2 : 1;
    constexpr int kCPH = NOUT / kHalves;
    constexpr int kSB = kCPH < 32 ? kCPH : 32;
    constexpr int kNB = kCPH / kSB;
    constexpr int kSh = kSB == 32 ? 0 : 1;
    const int ew = warp - kFlEpiWarp0;
    const int quad = warp & 3;
    const int half = ew >> 2;
    const int e = quad * 32 + lane;
    float s1[kNB], s2[kNB];
#pragma unroll
    for (int b = 0; b < kNB; ++b) s1[b] = s2[b] = 0.f;
    constexpr bool kRegStats = kCPH <= 32;
    // r1, r2: running mean and M2 of this thread's rows (Welford), rn: their count
    float r1[kRegStats ? kCPH : 1], r2[kRegStats ? kCPH : 1];
    float rn = 0.f;
#pragma unroll
    for (int i = 0; i < (kRegStats ? kCPH : 1); ++i) r1[i] = r2[i] = 0.f;
    float sn = 0.f;  // rows merged into s1 / s2 (the mean and M2 of channel lane >> kSh)
    const bool stats = a.mode == kFpropStats;
    const bool bias_relu = a.mode == kFpropBiasRelu;
    const int out_c = a.out_c;
    const size_t opitch = (size_t)out_c * 2;
    const bool v8 = (out_c % 16) == 0 && (reinterpret_cast<uintptr_t>(a.out) & 31) == 0;
    uint8_t* obase = static_cast<uint8_t*>(a.out);
    const bool valid = e < g.q;
    uint32_t it = 0;
    for (int u = blockIdx.x; u < g.units && !hc::is_aborted(abort_flag); u += gridDim.x, ++it) {
      const uint32_t s = it & 1, ph = (it >> 1) & 1;
      if (!mbar_wait_backoff(bar_acc_full + 8 * s, ph, 128)) {
        hc::set_abort(abort_flag, a.err, kErrWaitMma);
        break;
      }
      tc_fence_after();
      uint8_t* orow = obase + ((size_t)u * g.q + e) * opitch;  // u = n * P + p
      if (half < kHalves) {
#pragma unroll
        for (int b = 0; b < kNB; ++b) {
          const int c0 = half * kCPH + b * kSB;
          uint32_t r[kSB];
#pragma unroll
          for (int q16 = 0; q16 < kSB / 16; ++q16)
            tmem_ld16(tmem_base + ((uint32_t)(quad * 32) << 16) + s * NOUT + c0 + q16 * 16,
                      *reinterpret_cast<uint32_t(*)[16]>(r + q16 * 16));
          tmem_ld_wait();
          if (b == kNB - 1) {
            tc_fence_before();
            mbar_arrive(bar_acc_empty + 8 * s);
          }
          float v[kSB];
#pragma unroll
          for (int i = 0; i < kSB; ++i) {
            float x = __uint_as_float(r[i]);
            if (bias_relu) x = fmaxf(x + __ldg(a.bias + c0 + i), 0.f);
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
      } else {
        tc_fence_before();
        mbar_arrive(bar_acc_empty + 8 * s);
      }
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
      float* red = reinterpret_cast<float*>(smem + off_a);  // the A stages are free now
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
  if (a.mode == kFpropStats)
    hc::stats_partial_finalize<NOUT, kFlThreads, 2 * kFlTile>(a, reinterpret_cast<const float*>(smem + off_a),
                                                               smem + off_a, ticket_slot, abort_flag);
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}


// ------------------------------------------------------------------------------ forward, implicit im2col
// Stride 1 or 2 (the 7x7 stride-2 image stem among them): pad each
// pixel to 8/stride channel slots, so `stride` adjacent pixels fill one 16-byte group and the
// run of filter row rr for output pixel q starts at group q + const of the padded input row.
// The im2col tile of a filter row is then the padded row itself read through a descriptor
// without swizzle whose 8-row core matrices step 16 bytes per M row (one output pixel) and 16
// bytes per K group: core matrices overlap, and no tile is ever assembled.  One unit (an
// output row) is R * nmr MMAs.  Each CTA takes a contiguous range of output rows, so
// consecutive units share R - stride input rows: a ring of padded rows is converted once per
// input row by four warps reading x from global memory.  The epilogue stages each warp's
// 32 x (channels) block swizzled in shared memory and writes it with one TMA store.
constexpr int kImpRing = 16;                          // padded input rows in the ring (>= 2R)
constexpr int kImpRaw = 8;                            // raw input rows in flight (bulk copies)
constexpr int kImpProdWarp = 0;                       // warp 0: bulk copies of raw input rows
constexpr int kImpConv0 = 1, kImpConvWarps = 4;       // warps 1-4 convert input rows
constexpr int kImpMmaWarp = 5;
constexpr int kImpEpiWarp0 = 6;                       // warps 6+: epilogue
// The epilogue: kHalves warps per TMEM lane quadrant, each taking kCPH of the channels of its
// 32 rows.  16 channels a warp up to 64 channels: the epilogue sets the pace of this kernel
// (a unit is only 14 MMAs), and with 32 channels a warp its per-unit chain of TMEM load, pack,
// staging, Welford update and store ran at about 0.9 us a unit; at 128 channels two warps per
// quadrant keep the registers of 64 channels a thread within the budget.
template <int NOUT>
struct ImpEpi {
  static constexpr int kHalves = NOUT == 128 ? 2 : NOUT / 16;
  static constexpr int kWarps = 4 * kHalves;
  static constexpr int kThreads = (kImpEpiWarp0 + kWarps) * 32;
  static constexpr int kCPH = NOUT / kHalves;                 // channels of one warp's block
  static constexpr uint32_t kStageBytes = 32u * kCPH * 2u;    // one warp's staged 32-row block
};
constexpr int kImpGroupsPerLane = 5;                  // ceil(max groups per row / 32)
constexpr int kImpAcc = 4;                            // accumulator stages in TMEM

__host__ __device__ inline uint32_t imp_align(uint32_t v) { return (v + 1023u) & ~1023u; }

struct ImpLayout {
  uint32_t off_raw, off_b, off_stage, off_bar, total;
};

template <int NOUT>
__host__ __device__ inline ImpLayout imp_layout(const FirstGeom& g) {
  ImpLayout L;
  L.off_raw = imp_align((uint32_t)kImpRing * g.rowb);
  L.off_b = imp_align(L.off_raw + (g.rawtma ? (uint32_t)kImpRaw * g.rawb : 0u));
  L.off_stage = L.off_b + imp_align((uint32_t)(g.r * g.nmr) * NOUT * 32);
  L.off_bar = L.off_stage + (uint32_t)ImpEpi<NOUT>::kWarps * 2u * ImpEpi<NOUT>::kStageBytes;
  L.total = L.off_bar + 512;
  return L;
}

// First filter row that unit (n, p) appends to the ring, given the unit before it in the
// CTA's range: R - stride when the two are consecutive rows of one image, else 0 (all R rows).
__device__ __forceinline__ int imp_first_new(const FirstGeom& g, int prev_n, int prev_p, int n, int p) {
  return (n == prev_n && p == prev_p + 1 && g.stride < g.r) ? g.r - g.stride : 0;
}

// Padded row of input row h of image n: group t holds pixels gpx*(t - jm) + i (i < gpx), each as
// cpx slots (the 3 channels, then zeros); zeros outside the image.  One warp, lane = group mod 32.
// Every load of the row is issued before the first is used (one memory latency per row): the
// common groups (a whole aligned pixel pair inside the image) load from a clamped, always-valid
// address and are zeroed by a select; groups at a ragged edge take a second, element-wise pass.
__device__ __forceinline__ void imp_convert_row(const uint16_t* x, const FirstGeom& g, int n, int h, uint32_t dst,
                                                int lane) {
  const int ngroups = g.rowb / 16;
  const bool row_in = h >= 0 && h < g.h;
  const size_t pix0 = ((size_t)n * g.h + (row_in ? h : 0)) * g.w;
  const uint16_t* xr = x + pix0 * 3;
  uint4 o[kImpGroupsPerLane];
  if (g.gpx == 2) {
    const bool al4 = g.xal4 && (pix0 & 1) == 0;  // then pixel pairs start 4-byte aligned
    // a 4-byte aligned base for the unconditional loads (x aligned down when it is not)
    const uint32_t* xw = al4 ? reinterpret_cast<const uint32_t*>(xr)
                             : reinterpret_cast<const uint32_t*>(reinterpret_cast<uintptr_t>(x) & ~static_cast<uintptr_t>(3));
    uint32_t w[kImpGroupsPerLane][3];
    bool edge[kImpGroupsPerLane];
#pragma unroll
    for (int k = 0; k < kImpGroupsPerLane; ++k) {
      const int t = lane + 32 * k;
      const int w0 = 2 * (t - g.jm);
      const bool in = row_in && t < ngroups && w0 + 1 >= 0 && w0 < g.w;  // some pixel inside the image
      const bool fast = in && al4 && w0 >= 0 && w0 + 1 < g.w;
      edge[k] = in && !fast;
      const uint32_t* pa = xw + (fast ? 3 * (w0 >> 1) : 0);
      w[k][0] = __ldg(pa);
      w[k][1] = __ldg(pa + 1);
      w[k][2] = __ldg(pa + 2);
      if (!fast) w[k][0] = w[k][1] = w[k][2] = 0u;
    }
#pragma unroll
    for (int k = 0; k < kImpGroupsPerLane; ++k) {
      if (edge[k]) {
        const int w0 = 2 * (lane + 32 * k - g.jm);
        uint32_t v[6];
#pragma unroll
        for (int e = 0; e < 6; ++e) {
          const int px = w0 + e / 3;
          v[e] = (px >= 0 && px < g.w) ? (uint32_t)__ldg(xr + px * 3 + e % 3) : 0u;
        }
        w[k][0] = v[0] | (v[1] << 16);
        w[k][1] = v[2] | (v[3] << 16);
        w[k][2] = v[4] | (v[5] << 16);
      }
      o[k] = make_uint4(w[k][0], w[k][1] & 0xffffu, (w[k][1] >> 16) | (w[k][2] << 16), w[k][2] >> 16);
    }
  } else {
#pragma unroll
    for (int k = 0; k < kImpGroupsPerLane; ++k) {
      const int t = lane + 32 * k;
      const int px = t - g.jm;
      const bool in = row_in && t < ngroups && px >= 0 && px < g.w;
      const uint16_t* pa = xr + (in ? px * 3 : 0);
      uint32_t v[3];
#pragma unroll
      for (int c = 0; c < 3; ++c) v[c] = in ? (uint32_t)__ldg(pa + c) : 0u;
      o[k] = make_uint4(v[0] | (v[1] << 16), v[2], 0u, 0u);
    }
  }
#pragma unroll
  for (int k = 0; k < kImpGroupsPerLane; ++k) {
    const int t = lane + 32 * k;
    if (t < ngroups) st_shared_v4(dst + 16u * t, o[k]);
  }
}

// The same padded row from a raw input row already in shared memory (w * 3 contiguous values,
// w a multiple of 8 so pixel pairs never straddle the row end).
__device__ __forceinline__ void imp_convert_row_smem(uint32_t raw, const FirstGeom& g, int h, uint32_t dst,
                                                     int lane) {
  const int ngroups = g.rowb / 16;
  const bool row_in = h >= 0 && h < g.h;
  uint4 o[kImpGroupsPerLane];
  if (g.gpx == 2) {
    uint32_t w[kImpGroupsPerLane][3];
#pragma unroll
    for (int k = 0; k < kImpGroupsPerLane; ++k) {
      const int pi = lane + 32 * k - g.jm;  // pixel pair
      const bool in = row_in && lane + 32 * k < ngroups && pi >= 0 && 2 * pi < g.w;
      const uint32_t a = raw + 12u * (uint32_t)(in ? pi : 0);
#pragma unroll
      for (int j = 0; j < 3; ++j) asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w[k][j]) : "r"(a + 4 * j));
      if (!in) w[k][0] = w[k][1] = w[k][2] = 0u;
    }
#pragma unroll
    for (int k = 0; k < kImpGroupsPerLane; ++k)
      o[k] = make_uint4(w[k][0], w[k][1] & 0xffffu, (w[k][1] >> 16) | (w[k][2] << 16), w[k][2] >> 16);
  } else {
#pragma unroll
    for (int k = 0; k < kImpGroupsPerLane; ++k) {
      const int px = lane + 32 * k - g.jm;
      const bool in = row_in && lane + 32 * k < ngroups && px >= 0 && px < g.w;
      const uint32_t a = raw + 6u * (uint32_t)(in ? px : 0);
      uint32_t v[3];
#pragma unroll
      for (int c = 0; c < 3; ++c)
        asm volatile("{ .reg .b16 t; ld.shared.b16 t, [%1]; cvt.u32.u16 %0, t; }" : "=r"(v[c]) : "r"(a + 2 * c));
      o[k] = in ? make_uint4(v[0] | (v[1] << 16), v[2], 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
#pragma unroll
  for (int k = 0; k < kImpGroupsPerLane; ++k) {
    const int t = lane + 32 * k;
    if (t < ngroups) st_shared_v4(dst + 16u * t, o[k]);
  }
}

template <int NOUT, bool BF16>
__global__ void __launch_bounds__(ImpEpi<NOUT>::kThreads, 1)
    first_fprop_imp_kernel(const __grid_constant__ CUtensorMap map_z, const ConvArgs a, const FirstGeom g,
                           const void* wts, const void* xin) {
  constexpr int kTmemCols = hc::pow2_at_least(kImpAcc * NOUT);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const ImpLayout L = imp_layout<NOUT>(g);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L.off_bar;
  const uint32_t bar_row_full = bar0, bar_row_empty = bar0 + 8 * kImpRing;
  const uint32_t bar_raw_full = bar0 + 16 * kImpRing, bar_raw_empty = bar_raw_full + 8 * kImpRaw;
  const uint32_t bar_acc_full = bar_raw_empty + 8 * kImpRaw, bar_acc_empty = bar_acc_full + 8 * kImpAcc;
  const uint32_t bar_drain = bar_acc_empty + 8 * kImpAcc;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + (bar_drain + 8 - sbase));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile uint32_t* ticket_slot = reinterpret_cast<volatile uint32_t*>(tmem_slot + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = g.r * g.nmr;
  // contiguous unit range of this CTA
  const int u_begin = (int)(((long long)blockIdx.x * g.units) / gridDim.x);
  const int u_end = (int)(((long long)(blockIdx.x + 1) * g.units) / gridDim.x);

  // filter as the B operand, K-major without swizzle: MMA t = rr*nmr + m reads groups 2m, 2m+1
  // of filter row rr; 16 bytes of (group kc, output channel o) at t*NOUT*32 + kc*NOUT*16 + o*16
  {
    const uint16_t* wsrc = static_cast<const uint16_t*>(wts);
    for (int i = threadIdx.x; i < nk * 2 * NOUT; i += ImpEpi<NOUT>::kThreads) {
      const int t = i / (2 * NOUT), rem = i - t * 2 * NOUT;
      const int kc = rem / NOUT, o = rem - kc * NOUT;
      const int rr = t / g.nmr, jj = 2 * (t - rr * g.nmr) + kc;
      uint32_t w32[4] = {0, 0, 0, 0};
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int gp = e / g.cpx, c = e - gp * g.cpx;
        const int sx = g.gpx * jj + gp - g.lead;
        if (sx >= 0 && sx < g.s && c < 3 && o < a.out_c)
          w32[e >> 1] |= (uint32_t)wsrc[((o * g.r + rr) * g.s + sx) * 3 + c] << ((e & 1) * 16);
      }
      st_shared_v4(sbase + L.off_b + (uint32_t)t * (NOUT * 32) + (uint32_t)kc * (NOUT * 16) + (uint32_t)o * 16u,
                   make_uint4(w32[0], w32[1], w32[2], w32[3]));
    }
  }
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kImpRing; ++i) {
      mbar_init(bar_row_full + 8 * i, 1);
      mbar_init(bar_row_empty + 8 * i, 1);
    }
    for (int i = 0; i < kImpRaw; ++i) {
      mbar_init(bar_raw_full + 8 * i, 1);
      mbar_init(bar_raw_empty + 8 * i, 1);
    }
    for (int i = 0; i < kImpAcc; ++i) {
      mbar_init(bar_acc_full + 8 * i, 1);
      mbar_init(bar_acc_empty + 8 * i, ImpEpi<NOUT>::kWarps);  // lane 0 of each epilogue warp
    }
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kImpMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == kImpProdWarp) {
    // ---------------------------------------------------------------- raw input rows (bulk copies)
    if (g.rawtma && lane == 0) {
      const uint8_t* xb = static_cast<const uint8_t*>(xin);
      int prev_n = -1, prev_p = -2;
      uint32_t i = 0;
      bool ok = true;
      for (int u = u_begin; u < u_end && ok && !hc::is_aborted(abort_flag); ++u) {
        const int n = u / g.p, p = u - n * g.p;
        const int f = imp_first_new(g, prev_n, prev_p, n, p);
        prev_n = n;
        prev_p = p;
        for (int rr = f; rr < g.r; ++rr, ++i) {
          const uint32_t rs = i % kImpRaw;
          if (!mbar_wait_backoff(bar_raw_empty + 8 * rs, ((i / kImpRaw) & 1) ^ 1, 32)) {
            hc::set_abort(abort_flag, a.err, kErrWaitHalo);
            ok = false;
            break;
          }
          const int h = p * g.stride - g.pad + rr;
          if (h >= 0 && h < g.h) {
            mbar_arrive_expect_tx(bar_raw_full + 8 * rs, (uint32_t)g.rawb);
            bulk_load_1d(sbase + L.off_raw + rs * g.rawb, xb + ((size_t)n * g.h + h) * g.rawb, (uint32_t)g.rawb,
                         bar_raw_full + 8 * rs);
          } else {
            mbar_arrive(bar_raw_full + 8 * rs);  // a zero row: nothing to copy
          }
        }
      }
    }
  } else if (warp < kImpConv0 + kImpConvWarps) {
    // ---------------------------------------------------------------- input-row converters
    // Rows go round-robin to the four warps (row r to warp r mod 4), so a warp's rows r - 8 and
    // r - 16, which last used the raw slot and the ring slot of row r, were its own and were
    // handled before r: every parity wait below is for the phase right after one this warp
    // has already seen (a parity wait cannot tell that phase from the one before it).
    const int cw = warp - kImpConv0;
    const uint16_t* x = static_cast<const uint16_t*>(xin);
    int n = u_begin / g.p, p = u_begin - n * g.p, f = 0;
    uint32_t i = 0;
    bool ok = true;
    for (int u = u_begin, k = 0; u < u_end && ok; ++u, ++k) {
      if ((k & 7) == 7 && __any_sync(0xffffffffu, hc::is_aborted(abort_flag))) break;
      for (int rr = f; rr < g.r; ++rr, ++i) {
        if ((int)(i % kImpConvWarps) != cw) continue;
        const uint32_t slot = i % kImpRing, fill = i / kImpRing, rs = i % kImpRaw;
        // the row's two barriers tested back to back; waited for only when not complete
        bool ready = mbar_test(bar_row_empty + 8 * slot, (fill & 1) ^ 1);
        if (g.rawtma) ready &= mbar_test(bar_raw_full + 8 * rs, (i / kImpRaw) & 1);
        if (!__all_sync(0xffffffffu, ready)) {
          bool got = mbar_wait_backoff(bar_row_empty + 8 * slot, (fill & 1) ^ 1, 256);
          if (g.rawtma) got = got && mbar_wait_backoff(bar_raw_full + 8 * rs, (i / kImpRaw) & 1, 256);
          if (!__all_sync(0xffffffffu, got)) {
            hc::set_abort(abort_flag, a.err, kErrWaitHalo);
            ok = false;
            break;
          }
        }
        const int h = p * g.stride - g.pad + rr;
        if (g.rawtma)
          imp_convert_row_smem(sbase + L.off_raw + rs * g.rawb, g, h, sbase + slot * g.rowb, lane);
        else
          imp_convert_row(x, g, n, h, sbase + slot * g.rowb, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (g.rawtma) mbar_arrive(bar_raw_empty + 8 * rs);
          mbar_arrive(bar_row_full + 8 * slot);
        }
      }
      const int pn = n, pp = p;
      if (++p == g.p) {
        p = 0;
        ++n;
      }
      f = imp_first_new(g, pn, pp, n, p);
    }
  } else if (warp == kImpMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer (whole warp)
    // The R x nmr MMAs of a unit run with compile-time trip counts for the common filters
    // (a runtime-bounded loop around the elected-lane MMA issues several times slower).
    const uint32_t idesc = make_idesc_f16(128, NOUT, BF16, false, false);
    const uint32_t ring = sbase, bmat = sbase + L.off_b;
    auto run_units = [&](auto kr, auto km) {
      constexpr int KR = decltype(kr)::value, KM = decltype(km)::value;
      const int R = KR ? KR : g.r, M = KM ? KM : g.nmr;
      int n = u_begin / g.p, p = u_begin - n * g.p;
      int f = 0;  // first new filter row of the current unit (the first unit appends all R)
      uint32_t iend = 0, it = 0;
      bool have_ready = false;  // this unit's barriers already seen complete (look-ahead)
      for (int u = u_begin; u < u_end; ++u, ++it) {
        if ((it & 7) == 7 && __any_sync(0xffffffffu, hc::is_aborted(abort_flag))) break;
        const uint32_t inew = iend;
        iend += (uint32_t)(R - f);
        const uint32_t s = it % kImpAcc, ph = (it / kImpAcc) & 1;
        // the unit's barriers are tested back to back (their latencies overlap); only one
        // that is not complete yet is then waited for
        bool ready = have_ready;
        if (!ready) {
          ready = mbar_test(bar_acc_empty + 8 * s, ph ^ 1);
          for (uint32_t j = inew; j < iend; ++j)
            ready &= mbar_test(bar_row_full + 8 * (j % kImpRing), (j / kImpRing) & 1);
          ready = __all_sync(0xffffffffu, ready);
        }
        if (!ready) {
          bool ok = mbar_wait(bar_acc_empty + 8 * s, ph ^ 1);
          for (uint32_t j = inew; j < iend && ok; ++j)
            ok = mbar_wait(bar_row_full + 8 * (j % kImpRing), (j / kImpRing) & 1);
          if (!__all_sync(0xffffffffu, ok)) {
            hc::set_abort(abort_flag, a.err, kErrWaitAccum);
            break;
          }
        }
        tc_fence_after();
        const uint32_t d = tmem_base + s * NOUT;
        const uint32_t row0 = iend - (uint32_t)R;
        // the next unit
        int n2 = n, p2 = p + 1;
        if (p2 == g.p) {
          p2 = 0;
          ++n2;
        }
        const int f2 = imp_first_new(g, n, p, n2, p2);
        bool ready_next = false;
        if constexpr (KR != 0 && KM != 0) {
#pragma unroll
          for (int rr = 0; rr < KR; ++rr) {
            if (rr == KR - 1 && u + 1 < u_end) {
              // look-ahead: test the next unit's barriers while this unit's last MMAs queue up
              const uint32_t s2 = (it + 1) % kImpAcc, ph2 = ((it + 1) / kImpAcc) & 1;
              const uint32_t iend2 = iend + (uint32_t)(R - f2);
              bool rn = mbar_test(bar_acc_empty + 8 * s2, ph2 ^ 1);
              for (uint32_t j = iend; j < iend2; ++j)
                rn &= mbar_test(bar_row_full + 8 * (j % kImpRing), (j / kImpRing) & 1);
              ready_next = __all_sync(0xffffffffu, rn);
            }
            const uint32_t arow = ring + ((row0 + rr) % kImpRing) * g.rowb;
#pragma unroll
            for (int m = 0; m < KM; ++m)
              mma_f16_ss_warp(d, make_noswz_desc(arow + 32u * m, 16, 128),
                              make_noswz_desc(bmat + (uint32_t)(rr * KM + m) * (NOUT * 32), NOUT * 16, 128), idesc,
                              (rr | m) ? 1u : 0u);
          }
        } else {
          uint32_t acc = 0;
          for (int rr = 0; rr < R; ++rr) {
            const uint32_t arow = ring + ((row0 + rr) % kImpRing) * g.rowb;
            for (int m = 0; m < M; ++m, acc = 1u)
              mma_f16_ss_warp(d, make_noswz_desc(arow + 32u * m, 16, 128),
                              make_noswz_desc(bmat + (uint32_t)(rr * M + m) * (NOUT * 32), NOUT * 16, 128), idesc, acc);
          }
        }
        mma_commit_warp(bar_acc_full + 8 * s);  // the epilogue also releases the unit's rows
        n = n2;
        p = p2;
        f = f2;
        have_ready = ready_next;
      }
    };
    if (g.r == 7 && g.nmr == 2)
      run_units(std::integral_constant<int, 7>{}, std::integral_constant<int, 2>{});
    else if (g.r == 5 && g.nmr == 3)
      run_units(std::integral_constant<int, 5>{}, std::integral_constant<int, 3>{});
    else
      run_units(std::integral_constant<int, 0>{}, std::integral_constant<int, 0>{});
    mma_commit_warp(bar_drain);
    mbar_wait(bar_drain, 0);
  } else {
    // ---------------------------------------------------------------- epilogue (ImpEpi warps)
    constexpr int kHalves = ImpEpi<NOUT>::kHalves;
    constexpr int kCPH = ImpEpi<NOUT>::kCPH;     // channels of one warp's block
    constexpr int kSB = kCPH < 32 ? kCPH : 32;
    constexpr int kNB = kCPH / kSB;
    constexpr int kSh = kSB == 32 ? 0 : 1;
    static_assert(kSB == 16 || kSB == 32, "the merge-scatter leaves channel lane >> kSh");
    constexpr uint32_t kSpan = kCPH * 2;         // staged row bytes = the TMA swizzle span
    constexpr uint32_t kSwz = kSpan / 16 - 1;    // 16-byte chunk bits XOR-ed with bits 7+ of the offset
    const int ew = warp - kImpEpiWarp0;
    const int quad = warp & 3;
    const int half = ew >> 2;
    const int e = quad * 32 + lane;
    float s1[kNB], s2[kNB];
#pragma unroll
    for (int b = 0; b < kNB; ++b) s1[b] = s2[b] = 0.f;
    constexpr bool kRegStats = kCPH <= 32;
    // r1, r2: running mean and M2 of this thread's rows (Welford), rn: their count
    float r1[kRegStats ? kCPH : 1], r2[kRegStats ? kCPH : 1];
    float rn = 0.f;
#pragma unroll
    for (int i = 0; i < (kRegStats ? kCPH : 1); ++i) r1[i] = r2[i] = 0.f;
    float sn = 0.f;  // rows merged into s1 / s2 (the mean and M2 of channel lane >> kSh)
    const bool stats = a.mode == kFpropStats;
    const bool bias_relu = a.mode == kFpropBiasRelu;
    const bool valid = e < g.q;
    const uint32_t stage0 = sbase + L.off_stage + (uint32_t)ew * 2 * ImpEpi<NOUT>::kStageBytes;
    // the unit sequence, to release ring rows: once a unit's MMAs are complete, the rows the
    // next unit does not read are free (first epilogue warp, lane 0)
    int n = u_begin / g.p, p = u_begin - n * g.p, f = 0;
    uint32_t iend = 0;
    uint32_t it = 0;
    for (int u = u_begin; u < u_end && !hc::is_aborted(abort_flag); ++u, ++it) {
      const uint32_t s = it % kImpAcc, ph = (it / kImpAcc) & 1;
      // the store that last read this unit's staging buffer (two units ago), waited for while
      // the accumulator is still being computed
      if (lane == 0) bulk_wait_group_read<1>();
      if (!mbar_wait_backoff(bar_acc_full + 8 * s, ph, 128)) {
        hc::set_abort(abort_flag, a.err, kErrWaitMma);
        break;
      }
      tc_fence_after();
      __syncwarp();
      {
        iend += (uint32_t)(g.r - f);
        const int pn = n, pp = p;
        if (++p == g.p) {
          p = 0;
          ++n;
        }
        f = imp_first_new(g, pn, pp, n, p);
        if (ew == 0 && lane == 0 && u + 1 < u_end)
          for (int j = 0; j < g.r - f; ++j) mbar_arrive(bar_row_empty + 8 * ((iend - g.r + j) % kImpRing));
      }
      if (half < kHalves) {
        const uint32_t sb = stage0 + (it & 1) * ImpEpi<NOUT>::kStageBytes;
#pragma unroll
        for (int b = 0; b < kNB; ++b) {
          const int c0 = half * kCPH + b * kSB;
          uint32_t r[kSB];
#pragma unroll
          for (int q16 = 0; q16 < kSB / 16; ++q16)
            tmem_ld16(tmem_base + ((uint32_t)(quad * 32) << 16) + s * NOUT + c0 + q16 * 16,
                      *reinterpret_cast<uint32_t(*)[16]>(r + q16 * 16));
          tmem_ld_wait();
          if (b == kNB - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_acc_empty + 8 * s);
          }
          float v[kSB];
#pragma unroll
          for (int i = 0; i < kSB; ++i) {
            float xv = __uint_as_float(r[i]);
            if (bias_relu) xv = fmaxf(xv + __ldg(a.bias + c0 + i), 0.f);
            // rows >= q are not stored (the TMA store clips them) and not counted by the
            // per-row Welford update; the warp merge of the 128-channel form weighs them by 0
            v[i] = (kRegStats || valid) ? xv : 0.f;
          }
#pragma unroll
          for (int cc = 0; cc < kSB / 8; ++cc) {
            const uint32_t logical = (uint32_t)lane * kSpan + (uint32_t)(b * kSB / 8 + cc) * 16u;
            st_shared_v4(sb + (logical ^ (((logical >> 7) & kSwz) << 4)),
                         make_uint4(pack2<BF16>(v[8 * cc + 0], v[8 * cc + 1]), pack2<BF16>(v[8 * cc + 2], v[8 * cc + 3]),
                                    pack2<BF16>(v[8 * cc + 4], v[8 * cc + 5]), pack2<BF16>(v[8 * cc + 6], v[8 * cc + 7])));
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
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (quad * 32 < g.q) tma_store_3d(&map_z, sb, half * kCPH, quad * 32, u);
          bulk_commit_group();
        }
      } else {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_acc_empty + 8 * s);
      }
    }
    if (lane == 0) bulk_wait_group<0>();
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
      // the ring is free: every MMA has completed
      float* red = reinterpret_cast<float*>(smem);
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
  if (a.mode == kFpropStats)
    hc::stats_partial_finalize<NOUT, ImpEpi<NOUT>::kThreads, 32768>(a, reinterpret_cast<const float*>(smem), smem, ticket_slot,
                                                          abort_flag);
  if (warp == kImpMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------------------ wgrad
// D[slot][k] = sum over the CTA's units of sum_q tile[q][slot] * dz[n,p,q][k]: the im2col tile
// is the MN-major A operand (M = K slot, two M = 128 tiles, so a fourth zero atom), the TMA-
// loaded dz rows of the unit are the MN-major B operand, the reduction runs over the unit's 128
// pixel rows (rows >= Q are zero in both).  Accumulators stay in TMEM for the whole kernel;
// warps 6-9 store them as this CTA's fp32 partial ([m tile][c16][v][row][4]).
constexpr uint32_t kFlWgTile = 4 * kFlAtomBytes;
constexpr int kFlWgThreads = (kFlEpiWarp0 + 4) * 32;  // 320
// four staged units in flight, two at NOUT = 128 (its dz stages take the room)
constexpr int fl_wg_xstages(int nout) { return nout > 64 ? 2 : kFlXStages; }

template <int NOUT, bool BF16>
__global__ void __launch_bounds__(kFlWgThreads, 1)
    first_wgrad_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_dz,
                       const FirstGeom g, const void* xin, float* part, uint32_t* err) {
  constexpr int kNkc = NOUT > 64 ? NOUT / 64 : 1;
  constexpr int kXS = fl_wg_xstages(NOUT);  // staged input rows in flight
  constexpr uint32_t kDzSub = 128 * 128;               // one 64-channel atom of the dz tile
  constexpr uint32_t kDzStage = kNkc * kDzSub;
  constexpr int kTmemCols = hc::pow2_at_least(2 * NOUT);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t xst = fl_xstage_bytes(g);
  const uint32_t off_a = kXS * xst, off_dz = off_a + 2 * kFlWgTile, off_bar = off_dz + 2 * kDzStage;
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + off_bar;
  const uint32_t bar_x_full = bar0, bar_x_empty = bar0 + 32, bar_a_full = bar0 + 64, bar_a_empty = bar0 + 80;
  const uint32_t bar_dz_full = bar0 + 96, bar_acc_full = bar0 + 112, bar_drain = bar0 + 120;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + off_bar + 128);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // zero the x stages (row margins and tails), the A stages (rows >= Q, unwritten slots, the
  // fourth atom) and the dz stages (rows >= Q)
  for (uint32_t i = threadIdx.x; i < off_bar / 16; i += kFlWgThreads)
    st_shared_v4(sbase + i * 16, make_uint4(0, 0, 0, 0));
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int i = 0; i < kXS; ++i) {
      mbar_init(bar_x_full + 8 * i, 1);
      mbar_init(bar_x_empty + 8 * i, kFlBuildWarps);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_a_full + 8 * i, kFlBuildWarps);
      mbar_init(bar_a_empty + 8 * i, 1);
      mbar_init(bar_dz_full + 8 * i, 1);
    }
    mbar_init(bar_acc_full, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------- input rows (x) and dz rows of each unit
    // One loop per unit for the whole warp: the input rows (TMA from lane 0, or a copy by all
    // lanes when the row pitch rules TMA out), then the unit's dz rows (TMA from lane 0).
    if (lane == 0) {
      if (g.tma) prefetch_tensormap(&map_x);
      prefetch_tensormap(&map_dz);
    }
    const uint32_t tx = (uint32_t)g.r * g.rowp;
    const uint16_t* xg = static_cast<const uint16_t*>(xin);
    const int row = g.w * 3;
    uint32_t it = 0;
    for (int u = blockIdx.x; u < g.units && !__any_sync(0xffffffffu, hc::is_aborted(abort_flag));
         u += gridDim.x, ++it) {
      const int n = u / g.p, p = u - n * g.p;
      const uint32_t s = it & 1, ph = (it >> 1) & 1;
      const uint32_t sx = it % kXS, phx = (it / kXS) & 1;
      if (!__all_sync(0xffffffffu, mbar_wait_backoff(bar_x_empty + 8 * sx, phx ^ 1, 64))) {
        hc::set_abort(abort_flag, err, kErrWaitHalo);
        break;
      }
      if (g.tma) {
        if (lane == 0) {
          mbar_arrive_expect_tx(bar_x_full + 8 * sx, tx);
          tma_load_3d(sbase + sx * xst, &map_x, -8, p * g.stride - g.pad, n, bar_x_full + 8 * sx);
        }
      } else {
        uint8_t* dst = smem + sx * xst;
        for (int i = lane; i < g.r * row; i += 32) {
          const int rr = i / row, e = i - rr * row;
          const int h = p * g.stride - g.pad + rr;
          *reinterpret_cast<uint16_t*>(dst + rr * g.rowp + 64 + 2 * e) =
              (h >= 0 && h < g.h) ? xg[((size_t)n * g.h + h) * row + e] : (uint16_t)0;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_x_full + 8 * sx);
      }
      // the dz stage is free once the MMAs of the unit that last used it have completed
      if (!__all_sync(0xffffffffu, mbar_wait_backoff(bar_a_empty + 8 * s, ph ^ 1, 64))) {
        hc::set_abort(abort_flag, err, kErrWaitOperand);
        break;
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_dz_full + 8 * s, (uint32_t)kNkc * g.q * 128);
        for (int kc = 0; kc < kNkc; ++kc)
          tma_load_2d(sbase + off_dz + s * kDzStage + kc * kDzSub, &map_dz, kc * 64, u * g.q, bar_dz_full + 8 * s);
      }
    }
    if (lane == 0) {
      if (g.tma)
        for (uint32_t k = (it > kXS ? it - kXS : 0); k < it; ++k)
          mbar_wait(bar_x_full + 8 * (k % kXS), (k / kXS) & 1);
      for (uint32_t k = (it > 2 ? it - 2 : 0); k < it; ++k) mbar_wait(bar_dz_full + 8 * (k & 1), (k >> 1) & 1);
    }
  } else if (warp <= kFlBuildWarps) {
    // ------------------------------------------------- im2col builders
    const int tid = threadIdx.x - 32;
    uint32_t it = 0;
    for (int u = blockIdx.x; u < g.units && !hc::is_aborted(abort_flag); u += gridDim.x, ++it) {
      const uint32_t s = it & 1, ph = (it >> 1) & 1;
      const uint32_t sx = it % kXS, phx = (it / kXS) & 1;
      if (!mbar_wait_backoff(bar_a_empty + 8 * s, ph ^ 1, 64) || !mbar_wait(bar_x_full + 8 * sx, phx)) {
        hc::set_abort(abort_flag, err, kErrWaitOperand);
        break;
      }
      fl_build_tile(sbase + off_a + s * kFlWgTile, sbase + sx * xst, g, tid);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar_x_empty + 8 * sx);
        mbar_arrive(bar_a_full + 8 * s);
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------- MMA issuer (whole warp, elected lane)
    const uint32_t idesc = make_idesc_f16(128, NOUT, BF16, true, true);
    uint32_t it = 0;
    for (int u = blockIdx.x; u < g.units && !__any_sync(0xffffffffu, hc::is_aborted(abort_flag));
         u += gridDim.x, ++it) {
      const uint32_t s = it & 1, ph = (it >> 1) & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar_a_full + 8 * s, ph) && mbar_wait(bar_dz_full + 8 * s, ph))) {
        hc::set_abort(abort_flag, err, kErrWaitOperand);
        break;
      }
      tc_fence_after();
      const uint64_t a0 = make_sw128_desc(sbase + off_a + s * kFlWgTile, kFlAtomBytes, 1024, 0);
      const uint64_t b0 = make_sw128_desc(sbase + off_dz + s * kDzStage, kDzSub, 1024, 0);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
          mma_f16_ss_warp(tmem_base + mt * NOUT, a0 + (uint64_t)((mt * 2 * kFlAtomBytes + kk * 2048) >> 4),
                          b0 + (uint64_t)((kk * 2048) >> 4), idesc, (it | kk) ? 1u : 0u);
      mma_commit_warp(bar_a_empty + 8 * s);
    }
    mma_commit_warp(bar_acc_full);
    mma_commit_warp(bar_drain);
    mbar_wait(bar_drain, 0);
  } else {
    // ------------------------------------------------- epilogue: TMEM -> fp32 partial
    const bool ok = mbar_wait_backoff(bar_acc_full, 0, 1024);
    if (!ok) hc::set_abort(abort_flag, err, kErrWaitMma);
    tc_fence_after();
    // a CTA without units never issued an MMA: its partial is zero
    const bool any = (int)blockIdx.x < g.units;
    if (ok) {
      const int quad = warp & 3;
      const int e = quad * 32 + lane;
#pragma unroll
      for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int c16 = 0; c16 < NOUT / 16; ++c16) {
          uint32_t r[16];
          tmem_ld16(tmem_base + ((uint32_t)(quad * 32) << 16) + mt * NOUT + c16 * 16, r);
          tmem_ld_wait();
          float4* dst = reinterpret_cast<float4*>(part) + (((size_t)blockIdx.x * 2 + mt) * (NOUT / 16) + c16) * 512 + e;
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v * 128] = any ? make_float4(__uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                             __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// dW[k][r][s][c] = sum over CTAs (fixed order: fp32 within four CTA slices, fp64 across them) of
// partial element (m tile, c16, v, row) with K slot = m tile*128 + row = r*24 + s*3 + c.
constexpr int kFlRedSpan = 64, kFlRedSlices = 4;

template <int NOUT>
__global__ void __launch_bounds__(kFlRedSpan * kFlRedSlices)
    first_wgrad_reduce_kernel(const float* __restrict__ part, float* __restrict__ dw, int grid, int R, int S) {
  __shared__ float4 red[kFlRedSlices][kFlRedSpan];
  const size_t per_cta = (size_t)2 * (NOUT / 16) * 512;  // float4
  const size_t f4 = (size_t)blockIdx.x * kFlRedSpan + threadIdx.x % kFlRedSpan;
  const int sl = threadIdx.x / kFlRedSpan;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (f4 < per_cta) {
    const float4* base = reinterpret_cast<const float4*>(part) + f4;
    for (int t0 = sl; t0 < grid; t0 += 8 * kFlRedSlices) {
      float4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int t = t0 + k * kFlRedSlices;
        v[k] = t < grid ? __ldg(base + (size_t)t * per_cta) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        acc.x += v[k].x;
        acc.y += v[k].y;
        acc.z += v[k].z;
        acc.w += v[k].w;
      }
    }
  }
  red[sl][threadIdx.x % kFlRedSpan] = acc;
  __syncthreads();
  if (sl != 0 || f4 >= per_cta) return;
  double t4[4] = {0.0, 0.0, 0.0, 0.0};
  for (int q = 0; q < kFlRedSlices; ++q) {
    const float4 v = red[q][threadIdx.x];
    t4[0] += v.x;
    t4[1] += v.y;
    t4[2] += v.z;
    t4[3] += v.w;
  }
  const int row = (int)(f4 % 128);
  const int vq = (int)((f4 / 128) % 4);
  const int c16 = (int)((f4 / 512) % (NOUT / 16));
  const int mt = (int)(f4 / (512 * (size_t)(NOUT / 16)));
  const int slot = mt * 128 + row;
  const int r = slot / 24, o = slot - r * 24;
  const int sx = o / 3, c = o - sx * 3;
  if (r >= R || sx >= S) return;
  for (int j = 0; j < 4; ++j) {
    const int k = c16 * 16 + vq * 4 + j;
    dw[((size_t)(k * R + r) * S + sx) * 3 + c] = (float)t4[j];
  }
}

// ------------------------------------------------------------------------------ wgrad, implicit im2col
// Weight gradient of the first layer for Cout = 64, stride 1 or 2, without an im2col tile
// (Tech-Renaissance CBR page, section 5.1: dW = sum over pixels of dz x im2col(x)).  The
// padded rows of the forward are the B operand, read MN-major through a descriptor without
// swizzle (16 bytes per K step = one output pixel, 16 bytes per N group of 8 K slots), and a
// pair of output rows p, p+1 is the A operand: the two 64-channel dz tiles stacked along M
// (M = 128).  The pair reads W = R + stride input rows; input row b of the window meets filter
// row b for row p (accumulator lanes 0-63) and filter row b - stride for row p+1 (lanes
// 64-127), so each window row has its own accumulator block of 16*nmr columns and one MMA
// per 16 output pixels.  Per CTA the blocks accumulate over a contiguous range of pairs; a
// fixed-order reduction then adds the two halves and the CTAs and maps K slots to (s, c).
constexpr int kIwRawWarp = 0, kIwDzWarp = 1, kIwConv0 = 2, kIwMmaWarp = 6, kIwRelWarp = 7, kIwEpiWarp0 = 8;
constexpr int kIwThreads = (kIwEpiWarp0 + 4) * 32;  // 384
constexpr int kIwDzStages = 3;
constexpr int kIwDone = 4;                           // pair-completion barriers in flight

struct IwGeom {
  int w;      // window rows per pair: r + stride
  int kq;     // K steps of 16 output pixels: ceil(q / 16)
  int pp;     // pairs per image: ceil(p / 2)
  int units;  // n_img * pp
  int ncol;   // accumulator columns per window row: 16 * nmr
};

struct IwLayout {
  uint32_t off_raw, off_dz, dztile, off_bar, total;
};

__host__ __device__ inline IwLayout iw_layout(const FirstGeom& g, const IwGeom& v) {
  IwLayout L;
  L.off_raw = imp_align((uint32_t)kImpRing * g.rowb);
  L.off_dz = imp_align(L.off_raw + (g.rawtma ? (uint32_t)kImpRaw * g.rawb : 0u));
  L.dztile = (uint32_t)v.kq * 16u * 128u;  // 16*kq pixels x 64 channels, SW128
  L.off_bar = L.off_dz + kIwDzStages * 2 * L.dztile;
  L.total = L.off_bar + 512;
  return L;
}

// First window row that pair j of image n appends, given the pair before it in the range.
__device__ __forceinline__ int iw_first_new(const FirstGeom& g, const IwGeom& v, int prev_n, int prev_j, int n, int j) {
  return (n == prev_n && j == prev_j + 1 && 2 * g.stride < v.w) ? v.w - 2 * g.stride : 0;
}

template <bool BF16>
__global__ void __launch_bounds__(kIwThreads, 1)
    first_wgrad_imp_kernel(const __grid_constant__ CUtensorMap map_dz, const FirstGeom g, const IwGeom v,
                           const void* xin, float* part, uint32_t* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const IwLayout L = iw_layout(g, v);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + L.off_bar;
  const uint32_t bar_row_full = bar0, bar_row_empty = bar0 + 8 * kImpRing;
  const uint32_t bar_raw_full = bar0 + 16 * kImpRing, bar_raw_empty = bar_raw_full + 8 * kImpRaw;
  const uint32_t bar_dz_full = bar_raw_empty + 8 * kImpRaw, bar_dz_empty = bar_dz_full + 8 * kIwDzStages;
  const uint32_t bar_done = bar_dz_empty + 8 * kIwDzStages, bar_drain = bar_done + 8 * kIwDone;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + (bar_drain + 8 - sbase));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u_begin = (int)(((long long)blockIdx.x * v.units) / gridDim.x);
  const int u_end = (int)(((long long)(blockIdx.x + 1) * v.units) / gridDim.x);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kImpRing; ++i) {
      mbar_init(bar_row_full + 8 * i, 1);
      mbar_init(bar_row_empty + 8 * i, 1);
    }
    for (int i = 0; i < kImpRaw; ++i) {
      mbar_init(bar_raw_full + 8 * i, 1);
      mbar_init(bar_raw_empty + 8 * i, 1);
    }
    for (int i = 0; i < kIwDzStages; ++i) {
      mbar_init(bar_dz_full + 8 * i, 1);
      mbar_init(bar_dz_empty + 8 * i, 1);
    }
    for (int i = 0; i < kIwDone; ++i) mbar_init(bar_done + 8 * i, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == kIwMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // the window's input rows: pair j of image n reads rows 2*j*stride - pad + b, b < w
  auto row_of = [&](int j, int b) { return 2 * j * g.stride - g.pad + b; };

  if (warp == kIwRawWarp) {
    // ---------------------------------------------------------------- raw input rows (bulk copies)
    if (g.rawtma && lane == 0) {
      const uint8_t* xb = static_cast<const uint8_t*>(xin);
      int prev_n = -1, prev_j = -2;
      uint32_t i = 0;
      bool ok = true;
      for (int u = u_begin; u < u_end && ok && !hc::is_aborted(abort_flag); ++u) {
        const int n = u / v.pp, j = u - n * v.pp;
        const int f = iw_first_new(g, v, prev_n, prev_j, n, j);
        prev_n = n;
        prev_j = j;
        for (int b = f; b < v.w; ++b, ++i) {
          const uint32_t rs = i % kImpRaw;
          if (!mbar_wait_backoff(bar_raw_empty + 8 * rs, ((i / kImpRaw) & 1) ^ 1, 32)) {
            hc::set_abort(abort_flag, err, kErrWaitHalo);
            ok = false;
            break;
          }
          const int h = row_of(j, b);
          if (h >= 0 && h < g.h) {
            mbar_arrive_expect_tx(bar_raw_full + 8 * rs, (uint32_t)g.rawb);
            bulk_load_1d(sbase + L.off_raw + rs * g.rawb, xb + ((size_t)n * g.h + h) * g.rawb, (uint32_t)g.rawb,
                         bar_raw_full + 8 * rs);
          } else {
            mbar_arrive(bar_raw_full + 8 * rs);
          }
        }
      }
    }
  } else if (warp == kIwDzWarp) {
    // ---------------------------------------------------------------- dz tiles of the pair (TMA)
    if (lane == 0) {
      prefetch_tensormap(&map_dz);
      uint32_t it = 0;
      for (int u = u_begin; u < u_end && !hc::is_aborted(abort_flag); ++u, ++it) {
        const int n = u / v.pp, j = u - n * v.pp;
        const uint32_t s = it % kIwDzStages;
        if (!mbar_wait_backoff(bar_dz_empty + 8 * s, ((it / kIwDzStages) & 1) ^ 1, 32)) {
          hc::set_abort(abort_flag, err, kErrWaitOperand);
          break;
        }
        // row 2j+1 past the image's last row loads as zeros (out-of-bounds fill), as do pixels
        // q >= Q of the last K step
        mbar_arrive_expect_tx(bar_dz_full + 8 * s, 2 * L.dztile);
        const uint32_t dst = sbase + L.off_dz + s * 2 * L.dztile;
        tma_load_4d(dst, &map_dz, 0, 0, 2 * j, n, bar_dz_full + 8 * s);
        tma_load_4d(dst + L.dztile, &map_dz, 0, 0, 2 * j + 1, n, bar_dz_full + 8 * s);
      }
    }
  } else if (warp < kIwConv0 + kImpConvWarps) {
    // ---------------------------------------------------------------- input-row converters
    const int cw = warp - kIwConv0;
    const uint16_t* x = static_cast<const uint16_t*>(xin);
    int prev_n = -1, prev_j = -2;
    uint32_t i = 0;
    bool ok = true;
    for (int u = u_begin; u < u_end && ok && !__any_sync(0xffffffffu, hc::is_aborted(abort_flag)); ++u) {
      const int n = u / v.pp, j = u - n * v.pp;
      const int f = iw_first_new(g, v, prev_n, prev_j, n, j);
      prev_n = n;
      prev_j = j;
      for (int b = f; b < v.w; ++b, ++i) {
        if ((int)(i % kImpConvWarps) != cw) continue;
        const uint32_t slot = i % kImpRing, fill = i / kImpRing, rs = i % kImpRaw;
        bool got = mbar_wait_backoff(bar_row_empty + 8 * slot, (fill & 1) ^ 1, 32);
        if (g.rawtma) got = got && mbar_wait_backoff(bar_raw_full + 8 * rs, (i / kImpRaw) & 1, 32);
        if (!__all_sync(0xffffffffu, got)) {
          hc::set_abort(abort_flag, err, kErrWaitHalo);
          ok = false;
          break;
        }
        const int h = row_of(j, b);
        if (g.rawtma)
          imp_convert_row_smem(sbase + L.off_raw + rs * g.rawb, g, h, sbase + slot * g.rowb, lane);
        else
          imp_convert_row(x, g, n, h, sbase + slot * g.rowb, lane);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (g.rawtma) mbar_arrive(bar_raw_empty + 8 * rs);
          mbar_arrive(bar_row_full + 8 * slot);
        }
      }
    }
  } else if (warp == kIwMmaWarp) {
    // ---------------------------------------------------------------- MMA issuer (whole warp)
    const uint32_t idesc = make_idesc_f16(128, (uint32_t)v.ncol, BF16, true, true);
    auto run_units = [&](auto w_c, auto kq_c) {
      constexpr int KW = decltype(w_c)::value, KQ = decltype(kq_c)::value;
      const int WR = KW ? KW : v.w, NQ = KQ ? KQ : v.kq;
      int n = u_begin / v.pp, j = u_begin - n * v.pp, f = 0;
      uint32_t iend = 0, it = 0;
      bool have_ready = false;  // this pair's barriers already seen complete (look-ahead)
      for (int u = u_begin; u < u_end; ++u, ++it) {
        if ((it & 7) == 7 && __any_sync(0xffffffffu, hc::is_aborted(abort_flag))) break;
        const uint32_t inew = iend;
        iend += (uint32_t)(WR - f);
        const uint32_t s = it % kIwDzStages;
        if (!have_ready) {
          // the pair's barriers are tested back to back (their latencies overlap); only one
          // that is not complete yet is then waited for
          bool ready = mbar_test(bar_dz_full + 8 * s, (it / kIwDzStages) & 1);
          for (uint32_t r = inew; r < iend; ++r)
            ready &= mbar_test(bar_row_full + 8 * (r % kImpRing), (r / kImpRing) & 1);
          if (!__all_sync(0xffffffffu, ready)) {
            bool ok = mbar_wait(bar_dz_full + 8 * s, (it / kIwDzStages) & 1);
            for (uint32_t r = inew; r < iend && ok; ++r)
              ok = mbar_wait(bar_row_full + 8 * (r % kImpRing), (r / kImpRing) & 1);
            if (!__all_sync(0xffffffffu, ok)) {
              hc::set_abort(abort_flag, err, kErrWaitAccum);
              break;
            }
          }
        }
        tc_fence_after();
        const uint32_t a0 = sbase + L.off_dz + s * 2 * L.dztile;
        const uint32_t row0 = iend - (uint32_t)WR;
        // the next pair
        int n2 = n, j2 = j + 1;
        if (j2 == v.pp) {
          j2 = 0;
          ++n2;
        }
        const int f2 = iw_first_new(g, v, n, j, n2, j2);
        bool ready_next = false;
        if constexpr (KW != 0 && KQ != 0) {
#pragma unroll
          for (int kk = 0; kk < KQ; ++kk) {
            if (kk == KQ - 1 && u + 1 < u_end) {
              // look-ahead: test the next pair's barriers while this pair's MMAs queue up,
              // so the next pair starts without a round of barrier latency
              const uint32_t s2 = (it + 1) % kIwDzStages, iend2 = iend + (uint32_t)(WR - f2);
              bool rn = mbar_test(bar_dz_full + 8 * s2, ((it + 1) / kIwDzStages) & 1);
              for (uint32_t r = iend; r < iend2; ++r)
                rn &= mbar_test(bar_row_full + 8 * (r % kImpRing), (r / kImpRing) & 1);
              ready_next = __all_sync(0xffffffffu, rn);
            }
            const uint64_t ad = make_sw128_desc(a0 + 2048u * kk, L.dztile, 1024, 0);
#pragma unroll
            for (int b = 0; b < KW; ++b)
              mma_f16_ss_warp(tmem_base + (uint32_t)(b * v.ncol),
                              ad, make_noswz_desc(sbase + ((row0 + b) % kImpRing) * g.rowb + 256u * kk, 128, 16),
                              idesc, (it | kk) ? 1u : 0u);
          }
        } else {
          for (int kk = 0; kk < NQ; ++kk) {
            const uint64_t ad = make_sw128_desc(a0 + 2048u * kk, L.dztile, 1024, 0);
            for (int b = 0; b < WR; ++b)
              mma_f16_ss_warp(tmem_base + (uint32_t)(b * v.ncol),
                              ad, make_noswz_desc(sbase + ((row0 + b) % kImpRing) * g.rowb + 256u * kk, 128, 16),
                              idesc, (it | kk) ? 1u : 0u);
          }
        }
        mma_commit_warp(bar_done + 8 * (it % kIwDone));
        n = n2;
        j = j2;
        f = f2;
        have_ready = ready_next;
      }
    };
    if (v.w == 9 && v.kq == 7)
      run_units(std::integral_constant<int, 9>{}, std::integral_constant<int, 7>{});
    else
      run_units(std::integral_constant<int, 0>{}, std::integral_constant<int, 0>{});
    mma_commit_warp(bar_drain);
    mbar_wait(bar_drain, 0);
  } else if (warp == kIwRelWarp) {
    // ---------------------------------------------------------------- releaser: once a pair's MMAs
    // are complete, its dz stage and the window rows the next pair does not read are free
    if (lane == 0) {
      int n = u_begin / v.pp, j = u_begin - n * v.pp, f = 0;
      uint32_t iend = 0, it = 0;
      for (int u = u_begin; u < u_end && !hc::is_aborted(abort_flag); ++u, ++it) {
        if (!mbar_wait_backoff(bar_done + 8 * (it % kIwDone), (it / kIwDone) & 1, 64)) {
          hc::set_abort(abort_flag, err, kErrWaitMma);
          break;
        }
        mbar_arrive(bar_dz_empty + 8 * (it % kIwDzStages));
        iend += (uint32_t)(v.w - f);
        const int pn = n, pj = j;
        if (++j == v.pp) {
          j = 0;
          ++n;
        }
        f = iw_first_new(g, v, pn, pj, n, j);
        if (u + 1 < u_end)
          for (int r = 0; r < v.w - f; ++r) mbar_arrive(bar_row_empty + 8 * ((iend - v.w + r) % kImpRing));
      }
    }
  } else {
    // ---------------------------------------------------------------- partials (4 warps, once)
    const int quad = warp & 3;
    const bool ok = mbar_wait_backoff(bar_drain, 0, 1024);
    tc_fence_after();
    if (!ok) {
      hc::set_abort(abort_flag, err, kErrWaitMma);
    } else {
      const int row = quad * 32 + lane;
      float* dst = part + ((size_t)blockIdx.x * v.w * 128 + row) * v.ncol;
      for (int b = 0; b < v.w; ++b) {
        for (int c0 = 0; c0 < v.ncol; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(b * v.ncol + c0), r);
          tmem_ld_wait();
          float4* d4 = reinterpret_cast<float4*>(dst + (size_t)b * 128 * v.ncol + c0);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            d4[k] = make_float4(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]), __uint_as_float(r[4 * k + 2]),
                                __uint_as_float(r[4 * k + 3]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kIwMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// dW[k][r][s][c] = sum over CTAs (in fixed order: fp32 within 8 slices of the CTAs, fp64
// across them) of the top half of window row r and the bottom half of window row r + stride,
// K slot (group t, element e) -> s = gpx*t + e / cpx - lead, c = e % cpx (c < 3).
constexpr int kIwRedSlices = 8;
__global__ void __launch_bounds__(128 * kIwRedSlices / 2)
    first_wgrad_imp_reduce_kernel(const float* __restrict__ part, float* __restrict__ dw, const FirstGeom g,
                                  const IwGeom v, int grid) {
  __shared__ float red[kIwRedSlices][64];
  const int rr = blockIdx.x / 64, k = blockIdx.x % 64;  // filter row, output channel
  const int col = threadIdx.x % 64, sl = threadIdx.x / 64;
  const size_t per_cta = (size_t)v.w * 128 * v.ncol;
  float acc = 0.f;
  if (col < v.ncol) {
    const float* top = part + ((size_t)rr * 128 + k) * v.ncol + col;
    const float* bot = part + ((size_t)(rr + g.stride) * 128 + 64 + k) * v.ncol + col;
    for (int c = sl; c < grid; c += kIwRedSlices) acc += __ldcg(top + c * per_cta) + __ldcg(bot + c * per_cta);
  }
  red[sl][col] = acc;
  __syncthreads();
  if (sl != 0 || col >= v.ncol) return;
  double t = 0.0;
  for (int q = 0; q < kIwRedSlices; ++q) t += red[q][col];
  const int grp = col / 8, e = col % 8;
  const int sx = g.gpx * grp + e / g.cpx - g.lead, c = e % g.cpx;
  if (c < 3 && sx >= 0 && sx < g.s) dw[((size_t)(k * g.r + rr) * g.s + sx) * 3 + c] = (float)t;
}

// ------------------------------------------------------------------------------ host helpers
bool first_geom(FirstGeom& g, const HaloGeom& hg, int stride) {
  g = FirstGeom{};
  g.n_img = hg.n_img;
  g.h = hg.h;
  g.w = hg.w;
  g.r = hg.r;
  g.s = hg.s;
  g.pad = hg.pad;
  g.stride = stride;
  g.p = (g.h + 2 * g.pad - g.r) / stride + 1;
  g.q = (g.w + 2 * g.pad - g.s) / stride + 1;
  if (g.p <= 0 || g.q <= 0 || g.q > 128 || g.r > 8 || g.s > 8) return false;
  g.units = g.n_img * g.p;
  const int row = g.w * 3;
  // staged row: 8 zero units (64 bytes, at least 3*pad elements), the row, a zero tail that
  // covers the right padding and the 26 elements a run read may pass its last value
  if (3 * g.pad > 30) return false;
  const int data_units = (row + 3) / 4;
  const int tail_units = (3 * g.pad + 32 + 3) / 4;
  const int wunits = (8 + data_units + tail_units + 1) / 2 * 2;
  g.rowp = wunits * 8;
  g.nk = (g.r * 24 + 15) / 16;
  g.tma = (row * 2) % 16 == 0 && wunits <= 256;
  g.imp = 0;
  if (stride == 1 || stride == 2) {
    g.gpx = stride;
    g.cpx = 8 / stride;
    g.jm = (g.pad + g.gpx - 1) / g.gpx;
    g.lead = g.gpx * g.jm - g.pad;
    const int nch = (g.lead + g.s + g.gpx - 1) / g.gpx;  // groups of one filter row's run
    g.nmr = (nch + 1) / 2;
    g.rowb = (128 + 2 * g.nmr) * 16;                     // output pixel 127 reads groups < 128 + 2*nmr
    g.imp = 128 + 2 * g.nmr <= 32 * kImpGroupsPerLane && 2 * g.r <= kImpRing;
  }
  return true;
}

bool first_x_map(CUtensorMap* m, const FirstGeom& g, const void* x, bool bf16) {
  // x viewed in 8-byte units (4 elements): a whole staged row is one box row
  (void)bf16;
  const uint64_t dims[3] = {(uint64_t)g.w * 3 / 4, (uint64_t)g.h, (uint64_t)g.n_img};
  const uint64_t strides[2] = {(uint64_t)g.w * 3 * 2, (uint64_t)g.h * g.w * 3 * 2};
  const uint32_t box[3] = {(uint32_t)g.rowp / 8, (uint32_t)g.r, 1};
  return encode_tiled_plain(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, x, dims, strides, box);
}

}  // namespace

int launch_first_fprop(const FpropArgs& f, int stride, int c_out, bool bf16, const void* x, const void* w,
                       int num_sms, cudaStream_t st) {
  ConvArgs a{};
  a.out = f.z;
  a.out_c = c_out;
  a.mode = f.mode;
  a.part = f.part;
  a.ticket = f.ticket;
  a.gamma = f.gamma;
  a.beta = f.beta;
  a.running_mean = f.running_mean;
  a.running_var = f.running_var;
  a.saved_mean = f.saved_mean;
  a.saved_inv_var = f.saved_inv_var;
  a.eq = f.eq;
  a.moments = f.moments;
  a.defer = f.defer;
  a.bias = f.bias;
  a.momentum = f.momentum;
  a.eps = f.eps;
  a.m_count = f.m_count;
  a.inv_m = 1.0 / (double)f.m_count;
  a.unbias = f.m_count > 1 ? (float)((double)f.m_count / (double)(f.m_count - 1)) : 1.f;
  a.err = f.err;
  FirstGeom g;
  if (!first_geom(g, f.g, stride)) return 3;
  CUtensorMap mx{};
  if (g.tma && !first_x_map(&mx, g, x, bf16)) return 6;
  const int nout = nout_for(c_out);
  if (nout != c_out) return 3;
  if (g.imp) {
    // implicit im2col: output written by TMA in blocks of 32 pixels x (channels / halves)
    g.xal4 = (reinterpret_cast<uintptr_t>(x) & 3) == 0;
    g.rawb = g.w * 6;
    g.rawtma = (g.rawb % 16) == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0;
    const int cph = nout == 128 ? 64 : 16;  // ImpEpi<nout>::kCPH
    CUtensorMap mz{};
    const uint64_t dims[3] = {(uint64_t)c_out, (uint64_t)g.q, (uint64_t)g.units};
    const uint64_t strides[2] = {(uint64_t)c_out * 2, (uint64_t)g.q * c_out * 2};
    const uint32_t box[3] = {(uint32_t)cph, 32, 1};
    uint32_t total = 0;
    switch (nout) {
      case 16: total = imp_layout<16>(g).total; break;
      case 32: total = imp_layout<32>(g).total; break;
      case 64: total = imp_layout<64>(g).total; break;
      default: total = imp_layout<128>(g).total; break;
    }
    const uint32_t ismem = total + 1024;
    if (ismem <= 227 * 1024 &&
        encode_tiled_span(&mz, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, f.z,
                          dims, strides, box, cph * 2)) {
      const int igrid = std::min(g.units, num_sms);
      if (f.parts_out) *f.parts_out = igrid;
      auto go = [&](auto kern, int threads) {
        if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), 227 * 1024)) return 6;
        kern<<<igrid, threads, ismem, st>>>(mz, a, g, w, x);
        return cudaGetLastError() == cudaSuccess ? 0 : 6;
      };
      switch (nout * 2 + (bf16 ? 1 : 0)) {
        case 16 * 2: return go(first_fprop_imp_kernel<16, false>, ImpEpi<16>::kThreads);
        case 16 * 2 + 1: return go(first_fprop_imp_kernel<16, true>, ImpEpi<16>::kThreads);
        case 32 * 2: return go(first_fprop_imp_kernel<32, false>, ImpEpi<32>::kThreads);
        case 32 * 2 + 1: return go(first_fprop_imp_kernel<32, true>, ImpEpi<32>::kThreads);
        case 64 * 2: return go(first_fprop_imp_kernel<64, false>, ImpEpi<64>::kThreads);
        case 64 * 2 + 1: return go(first_fprop_imp_kernel<64, true>, ImpEpi<64>::kThreads);
        case 128 * 2: return go(first_fprop_imp_kernel<128, false>, ImpEpi<128>::kThreads);
        case 128 * 2 + 1: return go(first_fprop_imp_kernel<128, true>, ImpEpi<128>::kThreads);
        default: return 3;
      }
    }
  }
  const uint32_t smem = kFlXStages * fl_xstage_bytes(g) + 2 * kFlTile + kFlAtoms * nout * 128 + 256 + 1024;
  if (smem > 227 * 1024) return 3;
  const int grid = std::min(g.units, num_sms);
  if (f.parts_out) *f.parts_out = grid;
  auto go = [&](auto kern) {
    if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), 227 * 1024)) return 6;
    kern<<<grid, kFlThreads, smem, st>>>(mx, a, g, w, x);
    return cudaGetLastError() == cudaSuccess ? 0 : 6;
  };
  switch (nout * 2 + (bf16 ? 1 : 0)) {
    case 16 * 2: return go(first_fprop_kernel<16, false>);
    case 16 * 2 + 1: return go(first_fprop_kernel<16, true>);
    case 32 * 2: return go(first_fprop_kernel<32, false>);
    case 32 * 2 + 1: return go(first_fprop_kernel<32, true>);
    case 64 * 2: return go(first_fprop_kernel<64, false>);
    case 64 * 2 + 1: return go(first_fprop_kernel<64, true>);
    case 128 * 2: return go(first_fprop_kernel<128, false>);
    case 128 * 2 + 1: return go(first_fprop_kernel<128, true>);
    default: return 3;
  }
}


size_t first_wgrad_partial_floats(int num_sms, int c_out) {
  // builder kernel: 2 x 128 x nout per CTA; implicit kernel: at most 512 columns x 128 lanes
  return (size_t)num_sms * std::max(2 * 128 * nout_for(c_out), 512 * 128);
}

int launch_first_wgrad(const HaloGeom& hg, int stride, int c_out, bool bf16, const void* x, const void* dz,
                       float* part, float* dw, uint32_t* err, int num_sms, cudaStream_t st,
                       void (*between)(void*), void* ctx) {
  FirstGeom g;
  if (!first_geom(g, hg, stride)) return 3;
  const int nout = nout_for(c_out);
  if (nout != c_out) return 3;
  if (g.imp && c_out == 64) {
    // implicit im2col (pairs of output rows, see first_wgrad_imp_kernel)
    IwGeom v;
    v.w = g.r + g.stride;
    v.kq = (g.q + 15) / 16;
    v.pp = (g.p + 1) / 2;
    v.units = g.n_img * v.pp;
    v.ncol = 16 * g.nmr;
    g.xal4 = (reinterpret_cast<uintptr_t>(x) & 3) == 0;
    g.rawb = g.w * 6;
    g.rawtma = (g.rawb % 16) == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0;
    const IwLayout L = iw_layout(g, v);
    CUtensorMap mdz4{};
    const uint64_t dims[4] = {64, (uint64_t)g.q, (uint64_t)g.p, (uint64_t)g.n_img};
    const uint64_t strides[3] = {128, (uint64_t)g.q * 128, (uint64_t)g.p * g.q * 128};
    const uint32_t box[4] = {64, (uint32_t)(16 * v.kq), 1, 1};
    if (v.w * v.ncol <= 512 && L.total + 1024 <= 227 * 1024 &&
        encode_tiled(&mdz4, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, dz, dims,
                     strides, box)) {
      const int grid = std::min(v.units, num_sms);
      auto go = [&](auto kern) {
        if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), 227 * 1024)) return 6;
        kern<<<grid, kIwThreads, L.total + 1024, st>>>(mdz4, g, v, x, part, err);
        if (cudaGetLastError() != cudaSuccess) return 6;
        if (between) between(ctx);
        first_wgrad_imp_reduce_kernel<<<g.r * 64, 64 * kIwRedSlices, 0, st>>>(part, dw, g, v, grid);
        return cudaGetLastError() == cudaSuccess ? 0 : 6;
      };
      return bf16 ? go(first_wgrad_imp_kernel<true>) : go(first_wgrad_imp_kernel<false>);
    }
  }
  CUtensorMap mx{}, mdz;
  if (g.tma && !first_x_map(&mx, g, x, bf16)) return 6;
  {
    const uint64_t dims[2] = {(uint64_t)c_out, (uint64_t)g.units * g.q};
    const uint64_t strides[1] = {(uint64_t)c_out * 2};
    const uint32_t box[2] = {64, (uint32_t)g.q};
    if (!encode_tiled(&mdz, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, dz, dims,
                      strides, box))
      return 6;
  }
  const int nkc = nout > 64 ? nout / 64 : 1;
  const uint32_t smem = fl_wg_xstages(nout) * fl_xstage_bytes(g) + 2 * kFlWgTile + 2 * nkc * 128 * 128 + 256 + 1024;
  if (smem > 227 * 1024) return 3;
  const int grid = num_sms;  // every CTA writes a partial (zero when it has no unit)
  auto go = [&](auto kern, auto red) {
    if (!ensure_smem_attr(reinterpret_cast<const void*>(kern), 227 * 1024)) return 6;
    kern<<<grid, kFlWgThreads, smem, st>>>(mx, mdz, g, x, part, err);
    if (cudaGetLastError() != cudaSuccess) return 6;
    if (between) between(ctx);
    const size_t per_cta = (size_t)2 * (nout / 16) * 512;
    const int rgrid = (int)((per_cta + kFlRedSpan - 1) / kFlRedSpan);
    red<<<rgrid, kFlRedSpan * kFlRedSlices, 0, st>>>(part, dw, grid, g.r, g.s);
    return cudaGetLastError() == cudaSuccess ? 0 : 6;
  };
  switch (nout * 2 + (bf16 ? 1 : 0)) {
    case 16 * 2: return go(first_wgrad_kernel<16, false>, first_wgrad_reduce_kernel<16>);
    case 16 * 2 + 1: return go(first_wgrad_kernel<16, true>, first_wgrad_reduce_kernel<16>);
    case 32 * 2: return go(first_wgrad_kernel<32, false>, first_wgrad_reduce_kernel<32>);
    case 32 * 2 + 1: return go(first_wgrad_kernel<32, true>, first_wgrad_reduce_kernel<32>);
    case 64 * 2: return go(first_wgrad_kernel<64, false>, first_wgrad_reduce_kernel<64>);
    case 64 * 2 + 1: return go(first_wgrad_kernel<64, true>, first_wgrad_reduce_kernel<64>);
    case 128 * 2: return go(first_wgrad_kernel<128, false>, first_wgrad_reduce_kernel<128>);
    case 128 * 2 + 1: return go(first_wgrad_kernel<128, true>, first_wgrad_reduce_kernel<128>);
    default: return 3;
  }
}

}  // namespace cbr
