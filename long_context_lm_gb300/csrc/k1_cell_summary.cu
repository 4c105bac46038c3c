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
#include "cell_summary.cuh"
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
  float x[8][8];
  if constexpr (!kF32) {
    load_cell_bf16<true>(reinterpret_cast<const uint4 *>(k) + cell * (kS * kD / 8), lane, x);
  } else {
    const int g = lane & 7, t0 = lane >> 3;
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
  cell_summary_warp(x, lane, kbar + cell * kD, amax + cell);
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
