// cell_summary.cuh -- the per-cell key summary shared by the prefill pass
// and the decode step: mean key kbar_c and largest token-key norm a_c of one
// 32-token cell (FreeSolo, paper.rainbus.top summary, 方法步骤详情 ③).
#pragma once

#include "fs_common.cuh"

namespace fs {

// One warp summarises one 32-token cell of bf16 keys (x[i][j] = dim 8g+j of
// token t0+4i, g = lane & 7, t0 = lane >> 3).  The reduction order is fixed
// (per-lane sums over i, then xor-shuffles), so every caller of this function
// gets bit-identical kbar and amax for the same cell.  Lanes 0-7 write
// kbar[8g .. 8g+7]; lane 0 writes *amax.
__device__ __forceinline__ void cell_summary_warp(const float (&x)[8][8], int lane,
                                                  float *__restrict__ kbar_c,
                                                  float *__restrict__ amax_c) {
  const int g = lane & 7;
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
    float4 *dst = reinterpret_cast<float4 *>(kbar_c) + 2 * g;
    dst[0] = make_float4(acc[0] * inv, acc[1] * inv, acc[2] * inv, acc[3] * inv);
    dst[1] = make_float4(acc[4] * inv, acc[5] * inv, acc[6] * inv, acc[7] * inv);
  }
  if (lane == 0) *amax_c = sqrtf(best);
}

// Load one cell of bf16 keys (32 rows of 64, contiguous) in the lane layout
// cell_summary_warp expects; every lane issues its eight 16-byte loads first.
// kReadOnly: the keys do not change during the kernel (read-only cache path);
// otherwise plain coherent loads (a kernel that wrote some of the rows).
template <bool kReadOnly>
__device__ __forceinline__ void load_cell_bf16(const uint4 *__restrict__ src, int lane,
                                               float (&x)[8][8]) {
  const int g = lane & 7, t0 = lane >> 3;
  uint4 raw[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    raw[i] = kReadOnly ? __ldg(src + (t0 + 4 * i) * 8 + g) : src[(t0 + 4 * i) * 8 + g];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t w[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[i][2 * j] = bf16_lo(w[j]);
      x[i][2 * j + 1] = bf16_hi(w[j]);
    }
  }
}

}  // namespace fs
