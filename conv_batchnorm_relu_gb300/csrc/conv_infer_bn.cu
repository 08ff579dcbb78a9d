// Inference in the CBR page's single-graph form (Tech-Renaissance CBR page, section 6:
// conv_fprop, then MUL by eq_scale, ADD eq_bias, ReLU, as one graph): the forward convolution
// whose epilogue applies y = relu(acc*scale + shift) to the fp32 accumulator, with
// scale = gamma/sqrt(running_var + eps) and shift = beta + (conv_bias - running_mean)*scale.
// Unlike the folded form (fold.cu + conv_fprop.cu), the filter is used as trained, so nothing
// is rounded to the storage dtype before the convolution.  Same halo-conv template and tiling
// as the training forward (conv_fprop.cu).
#include <algorithm>

#include "halo_conv.cuh"

namespace cbr {

int launch_fprop_bn(const FpropArgs& f, int c_in, int c_out, bool bf16, const void* x, const void* w,
                    int num_sms, cudaStream_t st) {
  ConvArgs a{};
  a.g = f.g;
  a.out = f.z;
  a.out_c = c_out;
  a.mode = kFpropPlain;
  a.eps = f.eps;
  a.bn_gamma = f.bn_gamma;
  a.bn_beta = f.bn_beta;
  a.bn_mean = f.bn_mean;
  a.bn_var = f.bn_var;
  a.conv_bias = f.conv_bias;
  a.m_count = f.m_count;
  a.err = f.err;
  HaloGeom& g = a.g;
  const int nch = c_in <= 64 ? 1 : (c_in <= 128 ? 2 : 0);
  if (nch == 0) return 3;
  int U = 2;
  if (!hc::finish_geom(g, U)) return 3;
  if (c_out > 64 && hc::layout(g, kKindFpropBn, nch, c_out, false).total + 1024 > 227 * 1024) {
    U = 1;
    g = f.g;
    if (!hc::finish_geom(g, U)) return 3;
  }
  bool wres = hc::layout(g, kKindFpropBn, nch, c_out, true).total + 1024 <= 227 * 1024;
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
#define CBR_INFER_BN_CASE(NCH_, COUT_, U_, WRES_)                                                        \
  if (nch == NCH_ && c_out == COUT_ && U == U_ && (WRES_ == wres)) {                                    \
    return bf16 ? hc::launch_halo_conv<kKindFpropBn, NCH_, COUT_, U_, WRES_, true>(a, mx, mw, grid, st) \
                : hc::launch_halo_conv<kKindFpropBn, NCH_, COUT_, U_, WRES_, false>(a, mx, mw, grid, st); \
  }
  // a resident filter where an instantiation has one, else the streamed filter
  for (int pass = 0; pass < 2; ++pass, wres = false) {
    CBR_INFER_BN_CASE(1, 16, 2, true)
    CBR_INFER_BN_CASE(1, 32, 2, true)
    CBR_INFER_BN_CASE(1, 64, 2, true)
    CBR_INFER_BN_CASE(1, 64, 2, false)
    CBR_INFER_BN_CASE(1, 128, 2, false)
    CBR_INFER_BN_CASE(1, 128, 1, true)
    CBR_INFER_BN_CASE(1, 128, 1, false)
    CBR_INFER_BN_CASE(2, 64, 2, false)
    CBR_INFER_BN_CASE(2, 128, 2, false)
    CBR_INFER_BN_CASE(2, 128, 1, false)
  }
#undef CBR_INFER_BN_CASE
  return 3;
}

}  // namespace cbr
