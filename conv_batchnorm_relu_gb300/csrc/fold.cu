// BN folding for inference (Tech-Renaissance CBR page, section 2; BatchNorm CUDA page,
// section 4.4): w_fold = w*gamma/sqrt(rv+eps) and b_fold = (b - rm)*gamma/sqrt(rv+eps) + beta,
// computed in fp32 and stored in the filter's storage dtype.
#include "cbr_internal.h"
#include "common.cuh"

namespace cbr {
namespace {

template <bool BF16>
__global__ void fold_kernel(const uint16_t* __restrict__ w, const float* __restrict__ conv_bias,
                            const float* __restrict__ gamma, const float* __restrict__ beta,
                            const float* __restrict__ rm, const float* __restrict__ rv, float eps,
                            uint16_t* __restrict__ w_fold, float* __restrict__ b_fold, int cout,
                            int rsc) {
  const int k = blockIdx.x;
  const float scale = gamma[k] / sqrtf(rv[k] + eps);
  for (int j = threadIdx.x; j < rsc; j += blockDim.x) {
    const size_t i = (size_t)k * rsc + j;
    float v;
    if constexpr (BF16) {
      v = __bfloat162float(__ushort_as_bfloat16(w[i])) * scale;
      w_fold[i] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    } else {
      v = __half2float(__ushort_as_half(w[i])) * scale;
      w_fold[i] = __half_as_ushort(__float2half_rn(v));
    }
  }
  if (threadIdx.x == 0) {
    const float b = conv_bias ? conv_bias[k] : 0.f;
    b_fold[k] = (b - rm[k]) * scale + beta[k];
  }
}

}  // namespace

int launch_fold(const void* w, const float* conv_bias, const float* gamma, const float* beta,
                const float* rm, const float* rv, float eps, void* w_fold, float* b_fold, int cout,
                int rsc, bool bf16, cudaStream_t st) {
  const uint16_t* wi = static_cast<const uint16_t*>(w);
  uint16_t* wo = static_cast<uint16_t*>(w_fold);
  if (bf16)
    fold_kernel<true><<<cout, 256, 0, st>>>(wi, conv_bias, gamma, beta, rm, rv, eps, wo, b_fold, cout, rsc);
  else
    fold_kernel<false><<<cout, 256, 0, st>>>(wi, conv_bias, gamma, beta, rm, rv, eps, wo, b_fold, cout, rsc);
  return cudaGetLastError() == cudaSuccess ? 0 : 6;
}

}  // namespace cbr
