// ReLU-mask transcoding between the bit-packed form this library writes (one bit per element,
// bit i of 32-bit word j <-> NHWC element 32j+i) and a byte-per-element form (0 or 1), as a
// standalone ReLU stores it (Tech-Renaissance CBR page, sections 8 and 9: the fused operator's
// BOOLEAN bit mask against the standalone ReLU's per-element INT8 mask, which its tests
// transcode to compare the two paths).  A byte counts as set when it is non-zero.
//
// Both directions are HBM streams: one thread per 32-bit word, 32 bytes on the byte side
// (two 16-byte vectors), grid-stride over a one-wave grid.
#include <algorithm>

#include "cbr_internal.h"
#include "common.cuh"

namespace cbr {
namespace {

constexpr int kMaskThreads = 256;

// Bits of 16 bytes: bit b set when byte b is non-zero.
__device__ __forceinline__ uint32_t bits_of(uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t r = 0;
#pragma unroll
  for (int k = 0; k < 4; ++k)
#pragma unroll
    for (int b = 0; b < 4; ++b) r |= ((w[k] >> (8 * b)) & 0xffu ? 1u : 0u) << (4 * k + b);
  return r;
}

// 16 bytes (0 or 1) of 16 bits.
__device__ __forceinline__ uint4 bytes_of(uint32_t bits16) {
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    w[k] = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) w[k] |= ((bits16 >> (4 * k + b)) & 1u) << (8 * b);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// Words [0, full) are whole (32 elements each); the last word, when count % 32 != 0, covers
// count % 32 elements and its higher bits are written as 0.
__global__ void __launch_bounds__(kMaskThreads) mask_bytes_to_bits_kernel(const uint8_t* __restrict__ bytes,
                                                                          uint32_t* __restrict__ bits, long long count) {
  const long long words = (count + 31) / 32, full = count / 32;
  for (long long j = (long long)blockIdx.x * kMaskThreads + threadIdx.x; j < words;
       j += (long long)gridDim.x * kMaskThreads) {
    uint32_t r = 0;
    if (j < full) {
      const uint4 lo = ld_global_nc_v4(bytes + j * 32);
      const uint4 hi = ld_global_nc_v4(bytes + j * 32 + 16);
      r = bits_of(lo) | (bits_of(hi) << 16);
    } else {
      for (long long e = j * 32; e < count; ++e) r |= (bytes[e] ? 1u : 0u) << (e - j * 32);
    }
    bits[j] = r;
  }
}

__global__ void __launch_bounds__(kMaskThreads) mask_bits_to_bytes_kernel(const uint32_t* __restrict__ bits,
                                                                          uint8_t* __restrict__ bytes, long long count) {
  const long long words = (count + 31) / 32, full = count / 32;
  for (long long j = (long long)blockIdx.x * kMaskThreads + threadIdx.x; j < words;
       j += (long long)gridDim.x * kMaskThreads) {
    const uint32_t r = __ldg(bits + j);
    if (j < full) {
      st_global_v4(bytes + j * 32, bytes_of(r & 0xffffu));
      st_global_v4(bytes + j * 32 + 16, bytes_of(r >> 16));
    } else {
      for (long long e = j * 32; e < count; ++e) bytes[e] = (uint8_t)((r >> (e - j * 32)) & 1u);
    }
  }
}

int mask_grid(long long count, int num_sms) {
  const long long words = (count + 31) / 32;
  const long long want = std::max<long long>(1, (words + kMaskThreads - 1) / kMaskThreads);
  return (int)std::min<long long>(want, (long long)num_sms * 8);
}

}  // namespace

int launch_mask_bytes_to_bits(const uint8_t* bytes, uint32_t* bits, long long count, int num_sms, cudaStream_t st) {
  if (count <= 0) return 0;
  mask_bytes_to_bits_kernel<<<mask_grid(count, num_sms), kMaskThreads, 0, st>>>(bytes, bits, count);
  return cudaGetLastError() == cudaSuccess ? 0 : 6;
}

int launch_mask_bits_to_bytes(const uint32_t* bits, uint8_t* bytes, long long count, int num_sms, cudaStream_t st) {
  if (count <= 0) return 0;
  mask_bits_to_bytes_kernel<<<mask_grid(count, num_sms), kMaskThreads, 0, st>>>(bits, bytes, count);
  return cudaGetLastError() == cudaSuccess ? 0 : 6;
}

}  // namespace cbr
