// DGrad: dx = stride-1 convolution of dz (P x Q, Cout channels) with the filter rotated by 180
// degrees and its channel roles swapped (CBR page, section 5.2; padding R-1-pad), for the
// layers the fused backward kernel (conv_bwd_fused.cu) does not take.  The A operand is the
// zero-padded dz halo, loaded by TMA from the materialised dz (its stored zero columns past q
// and the out-of-bounds fill supply the padding).
#include <algorithm>

#include "halo_conv.cuh"

namespace cbr {

int launch_dgrad(const DgradArgs& d, int c_in, int c_out, bool bf16, const void* w, int num_sms,
                 cudaStream_t st) {
  ConvArgs a{};
  a.g = d.g;
  a.out = d.dx;
  a.out_c = c_in;
  if (c_in % 8 != 0) return 3;  // dx rows are stored in 16-byte groups of 8 channels
  a.mode = kFpropPlain;
  a.err = d.err;
  if (d.dz_full == nullptr) return 3;
  const int nch = (c_out + 63) / 64;
  const int nout = nout_for(c_in);
  if (nch > 2 || c_in > 128) return 3;
  // two M tiles per unit wherever the streamed-filter layout fits (see launch_fprop)
  int U = 2;
  HaloGeom& g = a.g;
  if (!hc::finish_geom(g, U)) return 3;
  if (nout > 64 && hc::layout(g, kKindDgradTma, nch, nout, false).total + 1024 > 227 * 1024) {
    U = 1;
    g = d.g;
    if (!hc::finish_geom(g, U)) return 3;
  }
  bool wres = hc::layout(g, kKindDgradTma, nch, nout, true).total + 1024 <= 227 * 1024;
  const CUtensorMapDataType dt = bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap mx, mw;  // mx: the materialised dz
  {
    // dz rows have a pitch of dz_pitch >= q pixels, zero past q: the halo's right padding reads
    // those zeros (or the out-of-bounds fill past the pitch), its left padding the fill
    const uint64_t pitch = (uint64_t)d.dz_pitch;
    if (pitch < (uint64_t)g.w) return 3;
    const uint64_t dims[4] = {(uint64_t)c_out, pitch, (uint64_t)g.h, (uint64_t)g.n_img};
    const uint64_t strides[3] = {(uint64_t)c_out * 2, pitch * c_out * 2, (uint64_t)g.h * pitch * c_out * 2};
    const uint32_t box[4] = {64, (uint32_t)g.wp, (uint32_t)g.box_rows, 1};
    if (!encode_tiled(&mx, dt, 4, d.dz_full, dims, strides, box)) return 6;
  }
  {
    const uint64_t dims[3] = {(uint64_t)c_in, (uint64_t)(g.r * g.s), (uint64_t)c_out};
    const uint64_t strides[2] = {(uint64_t)c_in * 2, (uint64_t)g.r * g.s * c_in * 2};
    const uint32_t box[3] = {64, 1, 64};
    if (!encode_tiled(&mw, dt, 3, w, dims, strides, box)) return 6;
  }
  const int grid = std::min(g.total_units, num_sms);
#define CBR_DGRAD_KIND(K_, NCH_, NOUT_, U_, WRES_)                                               \
  (bf16 ? hc::launch_halo_conv<K_, NCH_, NOUT_, U_, WRES_, true>(a, mx, mw, grid, st)            \
        : hc::launch_halo_conv<K_, NCH_, NOUT_, U_, WRES_, false>(a, mx, mw, grid, st))
#define CBR_DGRAD_CASE(NCH_, NOUT_, U_, WRES_)                                                   \
  if (nch == NCH_ && nout == NOUT_ && U == U_ && (WRES_ == wres)) {                             \
    return CBR_DGRAD_KIND(kKindDgradTma, NCH_, NOUT_, U_, WRES_);                               \
  }
  // a resident filter where an instantiation has one, else the streamed filter
  for (int pass = 0; pass < 2; ++pass, wres = false) {
    CBR_DGRAD_CASE(1, 16, 2, true)
    CBR_DGRAD_CASE(1, 32, 2, true)
    CBR_DGRAD_CASE(1, 64, 2, true)
    CBR_DGRAD_CASE(1, 16, 2, false)
    CBR_DGRAD_CASE(1, 32, 2, false)
    CBR_DGRAD_CASE(1, 64, 2, false)
    CBR_DGRAD_CASE(2, 64, 2, false)
    CBR_DGRAD_CASE(1, 128, 2, false)
    CBR_DGRAD_CASE(2, 128, 2, false)
    CBR_DGRAD_CASE(1, 128, 1, false)
    CBR_DGRAD_CASE(2, 128, 1, false)
  }
#undef CBR_DGRAD_CASE
#undef CBR_DGRAD_KIND
  return 3;
}

}  // namespace cbr
