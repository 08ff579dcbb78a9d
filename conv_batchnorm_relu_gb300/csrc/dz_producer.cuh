// The BN + ReLU backward expression, evaluated while building an MMA operand tile.
//
// dz = gamma*inv_std*(g - dbeta/M - xhat*dgamma/M) with g = dy*mask and
// xhat = (z - mean)*inv_std (Tech-Renaissance CBR page, section 5.1; BatchNorm CUDA page,
// section 3.1) is affine in (g, z) per channel, so with the coefficients a, d, e produced by
// the backward reduction pass it is dz = a*g - d*z + e: two FMAs per element.  dz is never
// written to HBM; producer threads read dy, z and the mask (or y) with 128-bit loads, evaluate
// dz in fp32, round it to the storage dtype and store it into a 128-byte-swizzled smem tile
// that the tensor cores read directly.  Positions outside the image (conv padding) are 0.
#pragma once
#include "common.cuh"

namespace cbr {

struct DzSrc {
  const void* dy;          // [n][p][q][cout] storage dtype
  const void* z;           // [n][p][q][cout] storage dtype
  const void* y;           // mask source when mask == nullptr: y > 0
  const uint8_t* mask;     // bit-packed ReLU mask (bit i of byte j <-> element 8j+i)
  const float* coef;       // [3][cout]: a, d, e
  int p, q, cout;
};

// Fill rows [0, nrows) of a tile of 128-byte rows (64 channels of channel chunk `kc`).
// Row i holds dz at pixel (pp, qq) = ((row0+i)/wsp + prow, (row0+i)%wsp - coff) of image n,
// or zeros when that pixel is outside [0,p) x [0,q).  Executed by `nthr` threads (a multiple
// of 8) with rank `tid`; each thread always handles the same 8 channels.  `dst` must be
// 1024-byte aligned (the swizzle phase is the row index mod 8).
template <bool BF16>
__device__ __forceinline__ void fill_dz_rows(uint32_t dst, int nrows, int row0, int wsp, int prow,
                                             int coff, int n, const DzSrc& s, int kc, int tid,
                                             int nthr) {
  constexpr int kUnroll = 4;
  const int c8 = tid & 7;
  const int ch0 = kc * 64 + c8 * 8;
  const bool ch_ok = ch0 < s.cout;
  float ca[8], cd[8], ce[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    ca[j] = ch_ok ? __ldg(s.coef + ch0 + j) : 0.f;
    cd[j] = ch_ok ? __ldg(s.coef + s.cout + ch0 + j) : 0.f;
    ce[j] = ch_ok ? __ldg(s.coef + 2 * s.cout + ch0 + j) : 0.f;
  }
  const uint8_t* dyb = static_cast<const uint8_t*>(s.dy);
  const uint8_t* zb = static_cast<const uint8_t*>(s.z);
  const uint8_t* yb = static_cast<const uint8_t*>(s.y);
  const int items = nrows * 8;
  for (int it0 = tid; it0 < items; it0 += nthr * kUnroll) {
    uint4 dv[kUnroll], zv[kUnroll], yv[kUnroll];
    uint32_t mb[kUnroll];
    bool ok[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int it = it0 + k * nthr;
      const int i = it >> 3;
      const int lin = row0 + i;
      const int pr = lin / wsp;
      const int pp = pr + prow, qq = lin - pr * wsp - coff;
      ok[k] = it < items && ch_ok && pp >= 0 && pp < s.p && qq >= 0 && qq < s.q;
      if (ok[k]) {
        const size_t v = (((size_t)n * s.p + pp) * s.q + qq) * s.cout + ch0;  // element index
        dv[k] = ld_global_nc_v4(dyb + v * 2);
        zv[k] = ld_global_nc_v4(zb + v * 2);
        if (s.mask) mb[k] = s.mask[v >> 3];
        else yv[k] = ld_global_nc_v4(yb + v * 2);
      }
    }
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      const int it = it0 + k * nthr;
      if (it >= items) break;
      uint4 o = make_uint4(0, 0, 0, 0);
      if (ok[k]) {
        uint32_t bits;
        if (s.mask) {
          bits = mb[k];
        } else {
          const uint32_t yw[4] = {yv[k].x, yv[k].y, yv[k].z, yv[k].w};
          bits = 0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 yy = unpack2<BF16>(yw[j]);
            bits |= (yy.x > 0.f ? 1u : 0u) << (2 * j);
            bits |= (yy.y > 0.f ? 1u : 0u) << (2 * j + 1);
          }
        }
        const uint32_t dw[4] = {dv[k].x, dv[k].y, dv[k].z, dv[k].w};
        const uint32_t zw[4] = {zv[k].x, zv[k].y, zv[k].z, zv[k].w};
        uint32_t ow[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 d = unpack2<BF16>(dw[j]);
          const float2 z = unpack2<BF16>(zw[j]);
          const float g0 = (bits >> (2 * j)) & 1u ? d.x : 0.f;
          const float g1 = (bits >> (2 * j + 1)) & 1u ? d.y : 0.f;
          const float r0 = fmaf(ca[2 * j], g0, fmaf(-cd[2 * j], z.x, ce[2 * j]));
          const float r1 = fmaf(ca[2 * j + 1], g1, fmaf(-cd[2 * j + 1], z.y, ce[2 * j + 1]));
          ow[j] = pack2<BF16>(r0, r1);
        }
        o = make_uint4(ow[0], ow[1], ow[2], ow[3]);
      }
      const int i = it >> 3;
      st_shared_v4(dst + swz_off((uint32_t)i, (uint32_t)c8, 128), o);
    }
  }
}

}  // namespace cbr
