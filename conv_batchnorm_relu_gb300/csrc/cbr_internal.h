// Host-side interface between the C ABI (cbr_api.cu) and the kernel launchers.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace cbr {

// Workspace sizing constants (cbr_api.cu): the first kWsHeaderBytes of every workspace hold
// arrival counters, and per-CTA partial buffers are sized for at most kMaxCtas CTAs (the grids
// never exceed the SM count, clamped to this).
constexpr size_t kWsHeaderBytes = 256;
constexpr int kMaxCtas = 256;
constexpr size_t align256(size_t v) { return (v + 255) / 256 * 256; }
// Training-forward workspace with the conv output kept by the caller: the counters, 2*Cout
// floats of apply coefficients and, per CTA, the partial statistics (2*Cout moments and a row
// count, padded to 2*Cout + 4 floats).
constexpr size_t forward_scratch_bytes(int c_out) {
  return align256(align256(kWsHeaderBytes + 2 * (size_t)c_out * 4) + (size_t)kMaxCtas * (2 * c_out + 4) * 4);
}

// Geometry of a stride-1 convolution computed over "padded-linear" rows.
//
// Output pixel (p, q) of image n is row m = p*wp + q of a per-image row space whose width is
// the padded input width wp = w + 2*pad; the wp - q_out columns past the last output column
// are computed and discarded.  In that space, filter tap (r, s) of output row m reads row
// m + r*wp + s of the zero-padded input, so each tap is the same contiguous slab of a halo
// tile shifted by r*wp + s rows.  A work unit is `um` consecutive rows of one image; its halo
// is `hr` input rows (wp wide) starting at input row floor(m0/wp) - pad.
struct HaloGeom {
  int n_img, h, w;   // conv input (NHWC)
  int p, q;          // conv output rows / cols
  int r, s, pad;     // filter taps; stride 1
  int wp;            // padded width
  int hr;            // halo rows per unit
  int um;            // output rows per unit (U * 128)
  int upi;           // units per image
  int total_units;
  int box_rows;      // halo rows per TMA box (the halo is fetched as ceil(hr/box_rows) boxes)
};

struct FpropArgs {
  HaloGeom g;
  void* z;                  // [n][p][q][cout] conv output (storage dtype)
  float* part;              // [grid][2][cout] per-CTA sum / sum of squares
  uint32_t* ticket;         // wrap-around arrival counter (must start at 0)
  const float* gamma;
  const float* beta;
  float* running_mean;
  float* running_var;
  float* saved_mean;
  float* saved_inv_var;
  float* eq;                // [2][cout] eq_scale, eq_bias for the apply pass
  // split (synchronised) forward: when set, the last CTA writes the merged moments of this
  // call's rows here, [mean cout][M2 cout][row count], instead of finalizing
  float* moments;
  // training forward whose apply pass merges the statistics: the CTAs write their partials
  // and no CTA finalizes (eq, the saved and the running statistics are left to the apply)
  int defer;
  int* parts_out;           // host: set to the number of partials (the grid) before the launch
  const float* bias;        // inference: per-channel bias added before ReLU
  // epilogue-only inference (launch_fprop_bn): BatchNorm parameters, conv bias (may be null)
  const float* bn_gamma;
  const float* bn_beta;
  const float* bn_mean;
  const float* bn_var;
  const float* conv_bias;
  float momentum;
  float eps;
  long long m_count;        // n*p*q
  uint32_t* err;            // device error word
  int mode;                 // FpropMode
};

enum FpropMode : int {
  kFpropStats = 0,   // z + per-channel statistics + finalize (training forward)
  kFpropPlain = 1,   // z only (recompute for backward)
  kFpropBiasRelu = 2 // y = relu(conv + bias) (folded inference)
};

// Opt `func` into `bytes` of dynamic shared memory on the current device (once per
// device and kernel; thread-safe).  Returns false if the runtime refuses.
bool ensure_smem_attr(const void* func, int bytes);

// The argument checks cbr_forward_train makes before it enqueues anything (descriptor,
// pointers, scalars, alignment, supported shape), but not the workspace or the device; on
// success *ws_need is the workspace the call needs (cbr_api.cu).  Returns a CBR status.
int check_forward_train(const void* desc, const void* x, const void* w, const float* gamma,
                        const float* beta, const float* running_mean, const float* running_var,
                        float momentum, float eps, const void* y, const uint32_t* relu_mask,
                        const void* z_saved, const float* saved_mean, const float* saved_inv_var,
                        size_t* ws_need);
// CBR_OK if the current device is one this library runs on (compute 10.3), else CBR_ERR_DEVICE.
int check_device();

// Tensor-map helpers (cbr_api.cu).
bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                  const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box);
// Same, without swizzle (plain row-major boxes).
bool encode_tiled_plain(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                  const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box);

// Same, with the swizzle span given in bytes (128, 64, 32; anything else: none).
bool encode_tiled_span(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       int swizzle_bytes);

// Launchers (one per kernel family).  Each validates only what its kernel needs beyond the
// C-ABI checks and returns a CBR status.
// First-layer forward (Cin = 3, any stride, R, S <= 8, Q <= 128): first_layer.cu.
int launch_first_fprop(const FpropArgs& f, int stride, int c_out, bool bf16, const void* x, const void* w,
                       int num_sms, cudaStream_t st);
// First-layer wgrad (dz read by TMA) and its fixed-order partial reduction: first_layer.cu.
int launch_first_wgrad(const HaloGeom& hg, int stride, int c_out, bool bf16, const void* x, const void* dz,
                       float* part, float* dw, uint32_t* err, int num_sms, cudaStream_t st,
                       void (*between)(void*) = nullptr, void* ctx = nullptr);
size_t first_wgrad_partial_floats(int num_sms, int c_out);
int launch_fprop(const FpropArgs& a, int c_in, int c_out, bool bf16, const void* x,
                 const void* w, int num_sms, cudaStream_t st);
// The persistent training forward (conv_fprop.cu): z, statistics, finalize, y and the mask in
// one cooperative launch; `ready` is a workspace word the kernel increments once per call.
bool fprop_apply_supported(const HaloGeom& g, int c_in, int c_out, int num_sms);
int launch_fprop_apply(const FpropArgs& f, void* y, uint32_t* mask, uint32_t* ready, int c_in, int c_out, bool bf16,
                       const void* x, const void* w, int num_sms, cudaStream_t st);
size_t fprop_partial_floats(int num_sms, int c_out);
// Inference forward with BatchNorm applied to the fp32 accumulator: relu(conv(x, W)*scale +
// shift), stride-1 layers (conv_infer_bn.cu).
int launch_fprop_bn(const FpropArgs& a, int c_in, int c_out, bool bf16, const void* x, const void* w,
                    int num_sms, cudaStream_t st);

struct ApplyArgs {
  const void* z;
  void* y;
  uint8_t* mask;            // bit-packed, bit i of byte j <-> element 8j+i; may be null
  const float* eq;          // [2][c] (unused when part is set)
  long long total;          // elements
  int c;
  // When set, the forward convolution left `nparts` partial moments here (FpropArgs::defer):
  // every block merges them into eq in its prologue and block 0 writes the finalize's outputs.
  const float* part;
  int nparts;
  const float* gamma;
  const float* beta;
  float* running_mean;
  float* running_var;
  float* saved_mean;
  float* saved_inv_var;
  float momentum;
  float eps;
  float inv_m;              // 1 / rows
  float unbias;             // rows / (rows - 1)
  uint32_t* err;
};
// Whether the apply pass can merge the statistics of a forward with c channels and at most
// max_parts partials (the staged partials must fit in shared memory).
bool apply_merge_supported(int c, int max_parts);
int launch_apply(const ApplyArgs& a, bool bf16, int num_sms, cudaStream_t st);

struct BwdReduceArgs {
  const void* dy;
  const void* z;
  const void* y;            // mask source when mask == null (y > 0)
  const uint8_t* mask;      // bit-packed mask or null
  const float* gamma;
  const float* mean;
  const float* inv_std;
  float* dgamma;
  float* dbeta;
  float* coef;              // [3][c]: a, d, e with dz = a*g - d*z + e
  // split (synchronised) backward: when set, the last block writes the raw per-channel sums
  // [sum g c][sum g*(z - mean) c] here instead of dgamma, dbeta and the coefficients
  float* sums_out;
  float* part;              // [grid][2][c]
  uint32_t* ticket;
  long long m_count;
  double inv_m;             // 1 / m_count (set by the launcher)
  int c;
  uint32_t* err;
};
int launch_bwd_reduce(const BwdReduceArgs& a, bool bf16, int num_sms, cudaStream_t st);
// Split forward, second half: merge `world` moment sets ([mean c][M2 c][count] each, in order)
// and finalize the statistics as the forward does (bn_kernels.cu).
int launch_merge_finalize(const float* moments, int world, int c, const float* gamma, const float* beta,
                          float* running_mean, float* running_var, float momentum, float eps,
                          float* saved_mean, float* saved_inv_var, float* eq, cudaStream_t st);
// Split backward, second half: dgamma, dbeta and the dz coefficients from reduced sums.
int launch_bwd_coef(const float* sums, int c, long long m_count, const float* gamma, const float* mean,
                    const float* inv_std, float* dgamma, float* dbeta, float* coef, cudaStream_t st);
size_t bwd_reduce_partial_floats(int num_sms, int c);

struct DgradArgs {
  HaloGeom g;               // geometry of the dgrad conv: input = dz (P x Q), output = dx
  void* dx;
  const void* dz_full;      // materialised dz [n][p][dz_pitch][cout]
  int dz_pitch;             // row pitch of dz_full in pixels (>= q, zero beyond q)
  uint32_t* err;
};
// MMA N width used for `c` output channels: the next of 16, 32, 64, 128.
inline int nout_for(int c) { return c <= 16 ? 16 : (c <= 32 ? 32 : (c <= 64 ? 64 : 128)); }
int launch_dgrad(const DgradArgs& a, int c_in, int c_out, bool bf16, const void* w, int num_sms,
                 cudaStream_t st);

struct WgradArgs {
  HaloGeom g;               // geometry of the forward conv
  float* part;              // [grid][taps*cin][cout] per-CTA partial dW
  float* dw;                // [cout][r][s][cin]
  // materialised dz [n][p][wp][cout] in the padded-linear row layout of the forward geometry
  // (row pitch wp = w + 2*pad, columns q..wp-1 zero)
  const void* dz_full;
  uint32_t* err;
};

// How the filter taps of a weight gradient are paired into M = 128 MMAs (two 64-channel atoms)
// and how the pairs and 64-channel input chunks are split across CTAs (conv_bwd.cu).
constexpr int kWgMaxGroups = 64;
constexpr int kWgMaxSplits = 8;
struct WgPlan {
  int nsplit, gmax, ngroups;
  int split_chunk[kWgMaxSplits], split_g0[kWgMaxSplits], split_ng[kWgMaxSplits];
  int ta[kWgMaxGroups], tb[kWgMaxGroups];
};
bool make_wg_plan(WgPlan& P, int taps, int c_in, int nout);
// Fixed-order sum of the per-CTA wgrad partials ([cta][group][c16][v][row][4]) into dW.
int launch_wgrad_reduce(const float* part, float* dw, const WgPlan& plan, int grid, int c_in, int taps,
                        int nout, cudaStream_t st);

// Fused backward convolutions (conv_bwd_fused.cu): one kernel evaluates dz = a*g - d*z + e once
// per tile in shared memory and feeds it to both the data gradient and the weight gradient.
struct BwdFusedArgs {
  HaloGeom g;               // geometry of the forward conv (stride 1, padding (R-1)/2)
  const void* dy;
  const void* z;
  const void* y;            // mask source when mask == null (y > 0)
  const uint8_t* mask;      // bit-packed ReLU mask or null
  const float* coef;        // [3][cout]: a, d, e
  void* dx;                 // [n][h][w][cin] or null (weight gradient only)
  float* part;              // per-CTA partial dW (wgrad_partial_floats)
  float* dw;
  uint32_t* err;
};
// Whether the fused kernel takes this layer (and so the backward needs no materialised dz).
bool bwd_fused_supported(int n, int h, int w, int c_in, int c_out, int r, int s, int stride, int pad);
int launch_bwd_fused(const BwdFusedArgs& a, int c_in, int c_out, bool bf16, const void* x, const void* w,
                     int num_sms, cudaStream_t st, void (*between)(void*) = nullptr, void* ctx = nullptr);
// Whether the TMA-fed wgrad (dz read from HBM) fits shared memory for this geometry.
bool wgrad_dz_tma_fits(const HaloGeom& g, int c_out);

// Unsigned 32-bit division by a run-time invariant divisor through a multiply-high
// (Granlund and Montgomery, "Division by invariant integers using multiplication", PLDI 1994,
// the round-up method): n / d = (t + ((n - t) >> s1)) >> s2 with t = umulhi(m, n), exact for
// every 32-bit n and 1 <= d < 2^31.
struct FastDiv {
  uint32_t d, m, s1, s2;
};
inline FastDiv make_fastdiv(uint32_t d) {
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  const uint64_t m = ((1ull << 32) * ((1ull << l) - d)) / d + 1;
  return FastDiv{d, (uint32_t)m, l ? 1u : 0u, l ? l - 1 : 0u};
}

struct DzArgs {
  const void* dy;
  const void* z;
  const void* y;            // mask source when mask == null (y > 0)
  const uint8_t* mask;
  const float* coef;        // [3][c]
  void* dz;                 // output, storage dtype: [n][p][pitch][c] (see below)
  long long total;          // elements of dy / z (n*p*q*c)
  int c;
  int q;                    // output columns of one image row
  int pitch;                // dz row pitch in pixels (>= q); columns q..pitch-1 are written as zero
  FastDiv fd_cvec, fd_q;    // division by c/8 and by q (set by the launcher)
};
// ReLU-mask transcoding, bit-packed <-> one byte per element (mask.cu).  count = elements.
int launch_mask_bytes_to_bits(const uint8_t* bytes, uint32_t* bits, long long count, int num_sms, cudaStream_t st);
int launch_mask_bits_to_bytes(const uint32_t* bits, uint8_t* bytes, long long count, int num_sms, cudaStream_t st);

// One warp that gives up on a never-completed barrier after limit_ns (selftest.cu).
int launch_selftest_wait(uint32_t* err, uint64_t limit_ns, cudaStream_t st);
// dz = a*(dy*mask) - d*z + e, elementwise (bn_kernels.cu).
int launch_dz(const DzArgs& a, bool bf16, int num_sms, cudaStream_t st);
// Launches the wgrad kernel, calls `between(ctx)` (if set), then the fixed-order reduction.
int launch_wgrad(const WgradArgs& a, int c_in, int c_out, bool bf16, const void* x, int num_sms,
                 cudaStream_t st, void (*between)(void*) = nullptr, void* ctx = nullptr);
size_t wgrad_partial_floats(int num_sms, int c_in, int c_out, int taps);

}  // namespace cbr
