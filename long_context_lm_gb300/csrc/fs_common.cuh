// fs_common.cuh -- small device helpers shared by the FS-L kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "fs.h"
#include "fs_internal.h"

namespace fs {

constexpr int kD = 64;       // head dim the kernels are built for
constexpr int kS = 32;       // tokens per cell
constexpr int kBq = 128;     // query block / query tile
constexpr int kMaxP = 64;    // largest P the prune kernels keep
constexpr int kMaxK = 8;     // largest K the select kernel keeps


// ---------------------------------------------------------------------------
// warp helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Three-input maximum (one instruction on this architecture).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Packed fp32 pairs: (a.x*b.x + c.x, a.y*b.y + c.y) and (a.x+b.x, a.y+b.y),
// each element rounded exactly as the scalar fmaf / add would round it.
__device__ __forceinline__ unsigned long long f2_bits(float x, float y) {
  return (unsigned long long)__float_as_uint(x) | ((unsigned long long)__float_as_uint(y) << 32);
}
__device__ __forceinline__ void fma2(float &rx, float &ry, float ax, float ay, float b, float c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(f2_bits(ax, ay)), "l"(f2_bits(b, b)),
      "l"(f2_bits(c, c)));
  rx = __uint_as_float((uint32_t)r);
  ry = __uint_as_float((uint32_t)(r >> 32));
}
// (a - b) on the two fp32 halves packed in 64-bit words (as bits).
__device__ __forceinline__ unsigned long long sub2_bits(unsigned long long a,
                                                       unsigned long long b) {
  unsigned long long r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ void add2(float &ax, float &ay, float bx, float by) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2_bits(ax, ay)), "l"(f2_bits(bx, by)));
  ax = __uint_as_float((uint32_t)r);
  ay = __uint_as_float((uint32_t)(r >> 32));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // .x = lo (low half)
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);  // .x = lo (low half)
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float bf16_lo(uint32_t x) {
  return __uint_as_float(x << 16);
}
__device__ __forceinline__ float bf16_hi(uint32_t x) {
  return __uint_as_float(x & 0xffff0000u);
}

// ---------------------------------------------------------------------------
// cp.async (Ampere-style async copy, still the simplest way to gather small
// scattered 16-byte pieces into shared memory)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)),
               "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::);
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Byte offset of 16-byte chunk `ch` (0..7) of row `r` in a tile whose rows
// are 128 bytes (64 bf16): chunks are XOR-swizzled by the row index so that
// eight rows read at the same logical chunk hit eight different bank groups.
__device__ __forceinline__ uint32_t swz128(int r, int ch) {
  return static_cast<uint32_t>(r * 128 + ((ch ^ (r & 7)) << 4));
}

}  // namespace fs
