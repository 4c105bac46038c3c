// k3_select.cu -- per-query cell scores and top-K selection.
//
// FreeSolo (paper.rainbus.top summary, 核心方法 and 方法步骤详情 ⑤; 局限与改进
// for the erf factor g_h >= erf(2); ai.info summary, "Methodology in Plain
// English"): a candidate cell c of query n scores
//     u = q_n . kbar_c + lambda_h * a_c * erf(sigma_h * (n - p_c) / s),
// p_c = c*s + s/2, with the unrotated query, and the K best cells are read.
// Candidates are the block's FS-L pool (<= P+W cells) or, in FS mode, every
// cell that ends at or before the block start.
//
// One CTA per (head, 128-query block), one thread per query.  Candidate mean
// keys are staged in shared memory in chunks of 64 cells and every thread
// computes its dot products in fp32 (the scores decide integer indices, so
// they are kept fp32-accurate).  The top-K list lives in registers and is
// ranked by (u desc, c asc).
#include "fs_common.cuh"
#include "fs_internal.h"

namespace fs {

constexpr int kSelChunk = 64;

__device__ __forceinline__ bool ranks_before(float u, int c, float u2, int c2) {
  return u > u2 || (u == u2 && c < c2);
}

template <bool kFS>
__global__ void __launch_bounds__(128) k3_select_kernel(
    const __nv_bfloat16 *__restrict__ q, const float *__restrict__ kbar,
    const float *__restrict__ amax, const int32_t *__restrict__ pool,
    const int32_t *__restrict__ pool_count, const float *__restrict__ lambda,
    const float *__restrict__ sigma, int H, int N, int K, int cap,
    int32_t *__restrict__ sel, float *__restrict__ sel_score) {
  __shared__ __align__(16) float s_kb[kSelChunk][kD];
  __shared__ float s_a[kSelChunk];
  __shared__ int s_c[kSelChunk];

  const int beta = blockIdx.x, bh = blockIdx.y, h = bh % H;
  const int C = N / kS;
  const int n = beta * kBq + threadIdx.x;
  const size_t row = (size_t)bh * N + n;

  float qf[kD];
  {
    const uint4 *src = reinterpret_cast<const uint4 *>(q + row * kD);
#pragma unroll
    for (int i = 0; i < kD / 8; ++i) {
      const uint4 r = __ldg(src + i);
      const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        qf[8 * i + 2 * j] = bf16_lo(w[j]);
        qf[8 * i + 2 * j + 1] = bf16_hi(w[j]);
      }
    }
  }
  const float lam = lambda[h], sig = sigma[h];
  const float inv_s = 1.0f / kS;

  float bu[kMaxK];
  int bc[kMaxK];
#pragma unroll
  for (int r = 0; r < kMaxK; ++r) {
    bu[r] = -INFINITY;
    bc[r] = 0x7fffffff;
  }

  const int A = beta * (kBq / kS);
  const int count = kFS ? A : min(pool_count[(size_t)bh * (N / kBq) + beta], cap);
  int nvalid = 0;
  const int32_t *pl = kFS ? nullptr : pool + ((size_t)bh * (N / kBq) + beta) * cap;

  for (int base = 0; base < count; base += kSelChunk) {
    const int m = min(kSelChunk, count - base);
    __syncthreads();
    if (threadIdx.x < m) {
      int c = kFS ? base + threadIdx.x : pl[base + threadIdx.x];
      if (c < 0 || c >= A) c = -1;  // not a cell this block may read: skipped
      s_c[threadIdx.x] = c;
      s_a[threadIdx.x] = c >= 0 ? amax[(size_t)bh * C + c] : 0.f;
    }
    __syncthreads();
    // stage the m mean keys: m*16 float4 pieces over 128 threads
    for (int i = threadIdx.x; i < m * (kD / 4); i += blockDim.x) {
      const int cc = i / (kD / 4), part = i % (kD / 4);
      const int c = s_c[cc];
      reinterpret_cast<float4 *>(s_kb[cc])[part] =
          c >= 0 ? __ldg(reinterpret_cast<const float4 *>(kbar + ((size_t)bh * C + c) * kD) + part)
                 : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    for (int j = 0; j < m; ++j) {
      if (s_c[j] < 0) continue;
      const float4 *kb = reinterpret_cast<const float4 *>(s_kb[j]);
      float d0 = 0.f, d1 = 0.f;
#pragma unroll
      for (int i = 0; i < kD / 4; i += 2) {
        const float4 x = kb[i], y = kb[i + 1];
        d0 = fmaf(qf[4 * i], x.x, d0);
        d0 = fmaf(qf[4 * i + 1], x.y, d0);
        d0 = fmaf(qf[4 * i + 2], x.z, d0);
        d0 = fmaf(qf[4 * i + 3], x.w, d0);
        d1 = fmaf(qf[4 * i + 4], y.x, d1);
        d1 = fmaf(qf[4 * i + 5], y.y, d1);
        d1 = fmaf(qf[4 * i + 6], y.z, d1);
        d1 = fmaf(qf[4 * i + 7], y.w, d1);
      }
      const int c = s_c[j];
      const float pc = (float)(c * kS) + 0.5f * kS;
      float u = (d0 + d1) + lam * s_a[j] * erff(sig * ((float)n - pc) * inv_s);
      int cu = c;
      ++nvalid;
#pragma unroll
      for (int r = 0; r < kMaxK; ++r) {
        if (r < K && ranks_before(u, cu, bu[r], bc[r])) {
          const float tu = bu[r];
          const int tc = bc[r];
          bu[r] = u;
          bc[r] = cu;
          u = tu;
          cu = tc;
        }
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kMaxK; ++r) {
    if (r < K) {
      const bool valid = r < nvalid;
      sel[row * K + r] = valid ? bc[r] : -1;
      if (sel_score) sel_score[row * K + r] = valid ? bu[r] : 0.f;
    }
  }
}

cudaError_t launch_select(const void *q, const float *kbar, const float *amax,
                          const int32_t *pool, const int32_t *pool_count, const float *lambda,
                          const float *sigma, const Shape &sh, int K, int cap, bool fs_mode,
                          int32_t *sel, float *sel_score, cudaStream_t st) {
  dim3 grid(sh.nblk(), sh.BH());
  const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(q);
  if (fs_mode)
    k3_select_kernel<true><<<grid, kBq, 0, st>>>(qb, kbar, amax, pool, pool_count, lambda, sigma,
                                                 sh.H, sh.N, K, cap, sel, sel_score);
  else
    k3_select_kernel<false><<<grid, kBq, 0, st>>>(qb, kbar, amax, pool, pool_count, lambda,
                                                  sigma, sh.H, sh.N, K, cap, sel, sel_score);
  return cudaGetLastError();
}

}  // namespace fs
