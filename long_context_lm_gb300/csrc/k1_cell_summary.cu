// k1_cell_summary.cu -- cell summaries of the unrotated keys.
//
// FreeSolo (paper.rainbus.top summary, 方法步骤详情 ③; ai.info summary, "Key
// Contributions" 2): every s-token cell is summarised by its mean key
// kbar_c (used for content routing) and its largest token-key L2 norm a_c (a
// query-independent priority used for pruning).
//
// HBM-bound streaming reduction: one warp per 32-token cell (4 KB of bf16
// keys); every lane issues all eight of its 16-byte loads before using any, a
// warp reads 512 contiguous bytes per load instruction, and the CTA's eight
// warps cover eight consecutive cells (32 KB).  Per token-head it reads 128 B
// and writes 8 B (kbar fp32 and a_c, amortised over the 32 tokens).
#include "fs_common.cuh"
#include "fs_internal.h"

namespace fs {

template <bool kF32>
__global__ void __launch_bounds__(256) k1_cell_summary_kernel(
    const void *__restrict__ k, long long ncells, float *__restrict__ kbar,
    float *__restrict__ amax) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long cell = (long long)blockIdx.x * 8 + warp;
  if (cell >= ncells) return;
  const int g = lane & 7;      // dims 8g .. 8g+7
  const int t0 = lane >> 3;    // tokens t0 + 4i

  float x[8][8];
  if constexpr (!kF32) {
    const uint4 *src = reinterpret_cast<const uint4 *>(k) + cell * (kS * kD / 8);
    uint4 raw[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) raw[i] = __ldg(src + (t0 + 4 * i) * 8 + g);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[i][2 * j] = bf16_lo(w[j]);
        x[i][2 * j + 1] = bf16_hi(w[j]);
      }
    }
  } else {
    const float4 *src = reinterpret_cast<const float4 *>(k) + cell * (kS * kD / 4);
    float4 raw[8][2];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      raw[i][0] = __ldg(src + (t0 + 4 * i) * 16 + 2 * g);
      raw[i][1] = __ldg(src + (t0 + 4 * i) * 16 + 2 * g + 1);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float f[8] = {raw[i][0].x, raw[i][0].y, raw[i][0].z, raw[i][0].w,
                          raw[i][1].x, raw[i][1].y, raw[i][1].z, raw[i][1].w};
#pragma unroll
      for (int j = 0; j < 8; ++j) x[i][j] = __bfloat162float(__float2bfloat16_rn(f[j]));
    }
  }

  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.f;
  float best = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    float sq = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      acc[j] += x[i][j];
      sq = fmaf(x[i][j], x[i][j], sq);
    }
    // the eight lanes holding token t0+4i: full squared norm
    sq += __shfl_xor_sync(0xffffffffu, sq, 1);
    sq += __shfl_xor_sync(0xffffffffu, sq, 2);
    sq += __shfl_xor_sync(0xffffffffu, sq, 4);
    best = fmaxf(best, sq);
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], 8);
    acc[j] += __shfl_xor_sync(0xffffffffu, acc[j], 16);
  }
  best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, 8));
  best = fmaxf(best, __shfl_xor_sync(0xffffffffu, best, 16));
  if (lane < 8) {
    const float inv = 1.0f / kS;
    float4 *dst = reinterpret_cast<float4 *>(kbar + cell * kD) + 2 * g;
    dst[0] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    dst[1] = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
  }
  if (lane == 0) amax[cell] = sqrtf(best);
}

cudaError_t launch_cell_summary(const void *k, bool f32, const Shape &sh, float *kbar,
                                float *amax, cudaStream_t st) {
  const long long ncells = (long long)sh.BH() * sh.C();
  const long long grid = (ncells + 7) / 8;
  if (f32)
    k1_cell_summary_kernel<true><<<(unsigned)grid, 256, 0, st>>>(k, ncells, kbar, amax);
  else
    k1_cell_summary_kernel<false><<<(unsigned)grid, 256, 0, st>>>(k, ncells, kbar, amax);
  return cudaGetLastError();
}

}  // namespace fs
