// Device-side helpers shared by the CBR kernels: storage-dtype packing, named barriers,
// the device error word and the 128-byte-swizzled row layout used for smem tiles.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"

namespace cbr {

// Bits of the device error word (OR-ed in by any CTA that gives up on a wait).
enum : uint32_t {
  kErrWaitHalo = 1u << 0,
  kErrWaitWeights = 1u << 1,
  kErrWaitAccum = 1u << 2,
  kErrWaitMma = 1u << 3,
  kErrWaitOperand = 1u << 4,
  kErrBadLaunch = 1u << 8,
};

__device__ __forceinline__ void report_error(uint32_t* err, uint32_t bits) {
  if (err) atomicOr(err, bits);
}

// Pack two fp32 values into one 32-bit word of the storage dtype (RNE rounding).
template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (BF16) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&w);
    return __bfloat1622float2(v);
  } else {
    __half2 v = *reinterpret_cast<__half2*>(&w);
    return __half22float2(v);
  }
}

// Named barrier among `count` threads (ids 1..15; id 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Named barrier that also ANDs a predicate across the participating threads, so every
// participant takes the same branch afterwards.
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// Byte offset of 16-byte chunk `ch` of row `row` in a tile whose rows are `pitch` bytes
// (a multiple of 128) and whose chunks are XOR-swizzled within each 128-byte segment by the
// row's phase -- the same pattern TMA's 128-byte swizzle writes.  Conflict-free when eight
// consecutive threads touch the eight chunks of one row, or one chunk of eight rows.
__device__ __forceinline__ uint32_t swz_off(uint32_t row, uint32_t ch, uint32_t pitch) {
  return row * pitch + (((ch & ~7u) | ((ch ^ row) & 7u)) << 4);
}

// 32-byte store (sm_100+ vector width); p must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* p, uint4 a, uint4 b) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a.x), "r"(a.y),
               "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}

__device__ __forceinline__ void st_global_v4(void* p, uint4 v) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint4 ld_global_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint32_t ld_shared_b32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

}  // namespace cbr
