// K1 + K2: forward convolution with BatchNorm statistics generated in the epilogue
// ("conv_fprop + genstats", Tech-Renaissance CBR page, section 4.1) and bn_finalize (section
// 4.2) run by the last CTA; the same kernel serves the z recompute for backward and the
// folded inference form relu(conv(x, W_fold) + b_fold) (sections 2 and 6).
// The kernel body is the shared halo-conv template (halo_conv.cuh) with TMA-loaded A.
#include <algorithm>

#include "halo_conv.cuh"

namespace cbr {

// per CTA: the means and M2s of its rows, then its row count (stats.cuh)
size_t fprop_partial_floats(int num_sms, int c_out) { return (size_t)num_sms * st::partial_floats(c_out); }

int launch_fprop(const FpropArgs& f, int c_in, int c_out, bool bf16, const void* x, const void* w,
                 int num_sms, cudaStream_t st) {
  ConvArgs a{};
  a.g = f.g;
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
  HaloGeom& g = a.g;
  const int nch = c_in <= 64 ? 1 : (c_in <= 128 ? 2 : 0);
  if (nch == 0) return 3;
  // Two M tiles per unit (um = 256 rows) wherever they fit: at 128 output channels that is all
  // 512 TMEM columns (two accumulator stages) and needs the streamed-filter layout to fit smem;
  // each filter slab then feeds twice the MMAs.
  int U = 2;
  if (!hc::finish_geom(g, U)) return 3;
  if (c_out > 64 && hc::layout(g, kKindFprop, nch, c_out, false).total + 1024 > 227 * 1024) {
    U = 1;
    g = f.g;
    if (!hc::finish_geom(g, U)) return 3;
  }
  bool wres = hc::layout(g, kKindFprop, nch, c_out, true).total + 1024 <= 227 * 1024;

  const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap mx, mw;
  {
    const uint64_t dims[4] = {(uint64_t)c_in, (uint64_t)g.w, (uint64_t)g.h, (uint64_t)g.n_img};
    const uint64_t strides[3] = {(uint64_t)c_in * 2, (uint64_t)g.w * c_in * 2, (uint64_t)g.h * g.w * c_in * 2};
    const uint32_t box[4] = {64, (uint32_t)g.wp, (uint32_t)g.box_rows, 1};
    if (!encode_tiled(&mx, dt, 4, x, dims, strides, box)) return 6;
  }
  {
    const uint64_t dims[3] = {(uint64_t)c_in, (uint64_t)(g.r * g.s), (uint64_t)c_out};
    const uint64_t strides[2] = {(uint64_t)c_in * 2, (uint64_t)g.r * g.s * c_in * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)c_out};
    if (!encode_tiled(&mw, dt, 3, w, dims, strides, box)) return 6;
  }
  const int grid = std::min(g.total_units, num_sms);
  if (f.parts_out) *f.parts_out = grid;

#define CBR_FPROP_CASE(NCH_, COUT_, U_, WRES_)                                                        \
  if (nch == NCH_ && c_out == COUT_ && U == U_ && (WRES_ == wres)) {                                 \
    return bf16 ? hc::launch_halo_conv<kKindFprop, NCH_, COUT_, U_, WRES_, true>(a, mx, mw, grid, st) \
                : hc::launch_halo_conv<kKindFprop, NCH_, COUT_, U_, WRES_, false>(a, mx, mw, grid, st); \
  }
  // a resident filter where an instantiation has one, else the streamed filter
  for (int pass = 0; pass < 2; ++pass, wres = false) {
    CBR_FPROP_CASE(1, 16, 2, true)
    CBR_FPROP_CASE(1, 32, 2, true)
    CBR_FPROP_CASE(1, 64, 2, true)
    CBR_FPROP_CASE(1, 64, 2, false)
    CBR_FPROP_CASE(1, 128, 2, false)
    CBR_FPROP_CASE(1, 128, 1, true)
    CBR_FPROP_CASE(1, 128, 1, false)
    CBR_FPROP_CASE(2, 64, 2, false)
    CBR_FPROP_CASE(2, 128, 2, false)
    CBR_FPROP_CASE(2, 128, 1, false)
  }
#undef CBR_FPROP_CASE
  return 3;
}

// Whether the persistent forward (conv + statistics + finalize + apply in one cooperative
// launch) takes this layer: a halo convolution with one 64-channel input chunk, 32 or 64 output
// channels, two 128-row tiles per unit and at most kPersistMaxUnits units per CTA (all
// accumulators resident in TMEM), with the filter resident in shared memory.
bool fprop_apply_supported(const HaloGeom& g_in, int c_in, int c_out, int num_sms) {
  if (c_in > 64 || (c_out != 32 && c_out != 64)) return false;
  HaloGeom g = g_in;
  if (!hc::finish_geom(g, 2)) return false;
  const int grid = std::min(g.total_units, num_sms);
  if ((g.total_units + grid - 1) / grid > kPersistMaxUnits) return false;
  return hc::layout(g, kKindFpropApply, 1, c_out, true).total + 1024 <= 227 * 1024;
}

int launch_fprop_apply(const FpropArgs& f, void* y, uint32_t* mask, uint32_t* ready, int c_in, int c_out, bool bf16,
                       const void* x, const void* w, int num_sms, cudaStream_t st) {
  if (!fprop_apply_supported(f.g, c_in, c_out, num_sms)) return 3;
  ConvArgs a{};
  a.g = f.g;
  a.out = f.z;
  a.out_c = c_out;
  a.mode = kFpropStats;
  a.part = f.part;
  a.ticket = f.ticket;
  a.gamma = f.gamma;
  a.beta = f.beta;
  a.running_mean = f.running_mean;
  a.running_var = f.running_var;
  a.saved_mean = f.saved_mean;
  a.saved_inv_var = f.saved_inv_var;
  a.eq = f.eq;
  a.y = y;
  a.mask = mask;
  a.ready = ready;
  a.momentum = f.momentum;
  a.eps = f.eps;
  a.m_count = f.m_count;
  a.inv_m = 1.0 / (double)f.m_count;
  a.unbias = f.m_count > 1 ? (float)((double)f.m_count / (double)(f.m_count - 1)) : 1.f;
  a.err = f.err;
  HaloGeom& g = a.g;
  hc::finish_geom(g, 2);
  const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap mx, mw;
  {
    const uint64_t dims[4] = {(uint64_t)c_in, (uint64_t)g.w, (uint64_t)g.h, (uint64_t)g.n_img};
    const uint64_t strides[3] = {(uint64_t)c_in * 2, (uint64_t)g.w * c_in * 2, (uint64_t)g.h * g.w * c_in * 2};
    const uint32_t box[4] = {64, (uint32_t)g.wp, (uint32_t)g.box_rows, 1};
    if (!encode_tiled(&mx, dt, 4, x, dims, strides, box)) return 6;
  }
  {
    const uint64_t dims[3] = {(uint64_t)c_in, (uint64_t)(g.r * g.s), (uint64_t)c_out};
    const uint64_t strides[2] = {(uint64_t)c_in * 2, (uint64_t)g.r * g.s * c_in * 2};
    const uint32_t box[3] = {64, 1, (uint32_t)c_out};
    if (!encode_tiled(&mw, dt, 3, w, dims, strides, box)) return 6;
  }
  const int grid = std::min(g.total_units, num_sms);
  if (c_out == 64)
    return bf16 ? hc::launch_halo_conv<kKindFpropApply, 1, 64, 2, true, true>(a, mx, mw, grid, st)
                : hc::launch_halo_conv<kKindFpropApply, 1, 64, 2, true, false>(a, mx, mw, grid, st);
  return bf16 ? hc::launch_halo_conv<kKindFpropApply, 1, 32, 2, true, true>(a, mx, mw, grid, st)
              : hc::launch_halo_conv<kKindFpropApply, 1, 32, 2, true, false>(a, mx, mw, grid, st);
}

}  // namespace cbr
