// k7_qkv.cu -- the shared q / k / v projection of an FS-L layer: RMSNorm of
// the hidden state, then W_q, W_k, W_v in one tcgen05 GEMM whose epilogue
// applies the norm's row scale and writes q, k, v in the [batch, H, N, d]
// layout the attention kernels read.
//
// FreeSolo (paper.rainbus.top summary, 方法步骤详情 ①): "the hidden state
// goes through RMSNorm and W_q, W_k, W_v to give q, k, v, shared by both
// branches".  With RMSNorm(x) = x * r * g, r = 1 / sqrt(mean(x^2) + eps):
//     [q | k | v][row, j] = r[row] * sum_i x[row, i] * (g[i] * w_qkv[j, i])
// so the gain folds into the weights (w' = bf16(w * g), once per call) and
// the row scale r into the epilogue (computed by a streaming pass over x).
//
// GEMM: D[128 x 192] tiles of x (K-major, M = 128 rows) times w'^T (w' rows
// are K-major: the [out, in] weight layout), K = D in steps of 64 staged by
// TMA through a 5-deep ring (16 KB of x + 24 KB of w' per stage).  192
// output columns are three heads of one of q, k, v (3*H*64 is always a
// multiple of 192).  Persistent CTAs, one per SM; warp 0 loads, warp 1 issues
// the MMAs (accumulators double buffered in TMEM, 2 x 192 columns), warps
// 4-7 run the epilogue of the previous tile: one thread per row, TMEM ->
// registers -> * r -> bf16 -> 64-byte row segments of q, k or v.
#include <cuda.h>
#include <string.h>

#include "fs_common.cuh"
#include "fs_internal.h"
#include "tc05.cuh"

namespace fs {
namespace {

constexpr int kBM = 128, kBN = 192, kBK = 64;
constexpr int kStages = 5;
constexpr int kThreads = 256;
constexpr uint32_t kStageA = kBM * kBK * 2;  // 16 KB
constexpr uint32_t kStageB = kBN * kBK * 2;  // 24 KB
constexpr uint32_t kSmem = kStages * (kStageA + kStageB) + 1024;
constexpr uint32_t kAccCols = 256;  // per accumulator buffer (192 used), power-of-two stride

struct GemmParams {
  const float *rscale;   // [M] row scales
  uint16_t *q, *k, *v;   // [batch, H, N, 64] bf16
  int M, D, H, N, ntn, ntiles;  // ntn: column tiles
  int *err;
};

__device__ __forceinline__ bool wait_nth(uint64_t *bar, uint32_t k, int *err) {
  return tc::mbar_wait(bar, k & 1, err);
}

struct Bars {
  uint64_t full[kStages], empty[kStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t fin;
  uint32_t tmem;
};

__global__ void __launch_bounds__(kThreads, 1) k7_qkv_gemm_kernel(
    const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
    const GemmParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Bars bar;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = p.D / kBK;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&bar.full[s], 1);
      tc::mbar_init(&bar.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bar.acc_full[b], 1);
      tc::mbar_init(&bar.acc_empty[b], 4);
    }
    tc::mbar_init(&bar.fin, 1);
    tc::mbar_fence_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&bar.tmem, 2 * kAccCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bar.tmem;
  const uint32_t sbase = smem_u32(smem);

  if (warp == 0 && lane == 0) {
    // TMA producer: stage s of the ring holds x[m0.., k0..] and w'[n0.., k0..]
    uint32_t it = 0;
    bool ok = true;
    for (int g = blockIdx.x; g < p.ntiles && ok; g += gridDim.x) {
      const int m0 = (g / p.ntn) * kBM, n0 = (g % p.ntn) * kBN;
      for (int kk = 0; kk < nk; ++kk, ++it) {
        const int s = it % kStages;
        if (it >= kStages && !wait_nth(&bar.empty[s], it / kStages - 1, p.err)) {
          ok = false;
          break;
        }
        unsigned char *a = smem + s * (kStageA + kStageB);
        tc::mbar_arrive_expect_tx(&bar.full[s], kStageA + kStageB);
        tc::tma_load_2d(a, &xmap, &bar.full[s], kk * kBK, m0);
        tc::tma_load_2d(a + kStageA, &wmap, &bar.full[s], kk * kBK, n0);
      }
    }
    // every load issued has landed before the CTA exits
    for (uint32_t j = it > (uint32_t)kStages ? it - kStages : 0; j < it; ++j)
      tc::mbar_wait(&bar.full[j % kStages], j / kStages, nullptr);
  } else if (warp == 1 && lane == 0) {
    // MMA issuer: D (tmem buffer) = sum over k of x_tile . w'_tile^T
    const uint32_t idesc = tc::idesc_bf16(kBM, kBN, 0);
    uint32_t it = 0, tcount = 0;
    for (int g = blockIdx.x; g < p.ntiles; g += gridDim.x, ++tcount) {
      const uint32_t ab = tcount & 1;
      if (tcount >= 2 && !wait_nth(&bar.acc_empty[ab], tcount / 2 - 1, p.err)) break;
      tc::fence_after_sync();
      const uint32_t d = tmem + ab * kAccCols;
      bool ok = true;
      for (int kk = 0; kk < nk; ++kk, ++it) {
        const int s = it % kStages;
        if (!wait_nth(&bar.full[s], it / kStages, p.err)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t a = sbase + s * (kStageA + kStageB);
        const uint64_t da = tc::desc_sw128(a), db = tc::desc_sw128(a + kStageA);
#pragma unroll
        for (int k16 = 0; k16 < kBK / 16; ++k16)
          tc::mma_ss(d, da + (uint64_t)(2 * k16), db + (uint64_t)(2 * k16), idesc,
                     (kk > 0 || k16 > 0) ? 1u : 0u);
        tc::mma_commit(&bar.empty[s]);
      }
      if (!ok) break;
      tc::mma_commit(&bar.acc_full[ab]);
    }
    tc::mma_commit(&bar.fin);
    tc::mbar_wait(&bar.fin, 0, nullptr);
  } else if (warp >= 4) {
    // epilogue: warp 4+w reads TMEM lanes 32w.., one thread per row
    const int r = (warp - 4) * 32 + lane;
    const uint32_t lane_base = (uint32_t)((warp - 4) * 32) << 16;
    const int hd = p.H * kD;
    uint32_t tcount = 0;
    for (int g = blockIdx.x; g < p.ntiles; g += gridDim.x, ++tcount) {
      const uint32_t ab = tcount & 1;
      const bool ok = wait_nth(&bar.acc_full[ab], tcount / 2, p.err);
      if (!__all_sync(0xffffffffu, ok)) break;
      tc::fence_after_sync();
      const int m0 = (g / p.ntn) * kBM, n0 = (g % p.ntn) * kBN;
      const int row = m0 + r;              // row of x: (batch, position)
      const int b = row / p.N, n = row % p.N;
      const float rs = p.rscale[row];
#pragma unroll 1
      for (int c = 0; c < kBN / 32; ++c) {
        uint32_t acc[32];
        tc::tmem_ld32(tmem + ab * kAccCols + lane_base + 32 * c, acc);
        tc::tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack_bf16(__uint_as_float(acc[2 * e]) * rs, __uint_as_float(acc[2 * e + 1]) * rs);
        const int j0 = n0 + 32 * c;         // output column
        const int which = j0 / hd, h = (j0 % hd) / kD, dim0 = j0 % kD;
        uint16_t *base = which == 0 ? p.q : (which == 1 ? p.k : p.v);
        uint4 *dst = reinterpret_cast<uint4 *>(base + (((size_t)b * p.H + h) * p.N + n) * kD + dim0);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          dst[e] = make_uint4(pk[4 * e], pk[4 * e + 1], pk[4 * e + 2], pk[4 * e + 3]);
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar.acc_empty[ab]);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 2 * kAccCols);
  }
}

// r[row] = 1 / sqrt(mean(x[row]^2) + eps): one warp per row of D bf16
__global__ void __launch_bounds__(256) k7_rowscale_kernel(const uint4 *__restrict__ x, int M, int D,
                                                           float eps, float *__restrict__ r) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (row >= M) return;
  const uint4 *src = x + (size_t)row * (D / 8);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int c = lane; c < D / 8; c += 32) {
    const uint4 u = __ldg(src + c);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      acc[j] = fmaf(bf16_lo(w[j]), bf16_lo(w[j]), acc[j]);
      acc[j] = fmaf(bf16_hi(w[j]), bf16_hi(w[j]), acc[j]);
    }
  }
  const float ss = warp_sum((acc[0] + acc[1]) + (acc[2] + acc[3]));
  if (lane == 0) r[row] = rsqrtf(ss / D + eps);
}

// w'[j, i] = bf16(w[j, i] * g[i])
__global__ void k7_fold_gain_kernel(const uint32_t *__restrict__ w, const float *__restrict__ g,
                                    int D, size_t n2, uint32_t *__restrict__ wf) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n2;
       i += (size_t)gridDim.x * blockDim.x) {
    const int col = (int)((2 * i) % D);
    const uint32_t x = __ldg(w + i);
    wf[i] = pack_bf16(bf16_lo(x) * __ldg(g + col), bf16_hi(x) * __ldg(g + col + 1));
  }
}

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  if (!fn) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(ptr);
  }
  return fn;
}

// [rows, cols] bf16 row-major, boxes of box_rows x 64 with the 128-byte swizzle
bool make_map(CUtensorMap *map, const void *ptr, size_t rows, int cols, int box_rows) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

}  // namespace

size_t qkv_workspace_bytes(int M, int D, int H) {
  const size_t w = (size_t)3 * H * kD * D * 2;
  return (w + 255) / 256 * 256 + ((size_t)M * 4 + 255) / 256 * 256;
}

cudaError_t launch_qkv(const QkvArgs &a, cudaStream_t st) {
  const int M = a.batch * a.N, nout = 3 * a.H * kD;
  unsigned char *ws = static_cast<unsigned char *>(a.ws);
  const size_t wbytes = ((size_t)nout * a.D * 2 + 255) / 256 * 256;
  float *rscale = reinterpret_cast<float *>(ws + wbytes);
  const void *w = a.w;
  if (a.gain) {
    const size_t n2 = (size_t)nout * a.D / 2;
    k7_fold_gain_kernel<<<(unsigned)((n2 + 255) / 256 < 4096 ? (n2 + 255) / 256 : 4096), 256, 0,
                          st>>>(static_cast<const uint32_t *>(a.w), a.gain, a.D, n2,
                                reinterpret_cast<uint32_t *>(ws));
    w = ws;
  }
  k7_rowscale_kernel<<<(M + 7) / 8, 256, 0, st>>>(static_cast<const uint4 *>(a.x), M, a.D, a.eps,
                                                  rscale);
  CUtensorMap xm, wm;
  memset(&xm, 0, sizeof(xm));
  memset(&wm, 0, sizeof(wm));
  if (!make_map(&xm, a.x, (size_t)M, a.D, kBM) || !make_map(&wm, w, (size_t)nout, a.D, kBN))
    return cudaErrorInvalidValue;
  GemmParams p;
  p.rscale = rscale;
  p.q = static_cast<uint16_t *>(a.q);
  p.k = static_cast<uint16_t *>(a.k);
  p.v = static_cast<uint16_t *>(a.v);
  p.M = M;
  p.D = a.D;
  p.H = a.H;
  p.N = a.N;
  p.ntn = nout / kBN;
  p.ntiles = (M / kBM) * p.ntn;
  p.err = a.err;
  cudaError_t e =
      cudaFuncSetAttribute(k7_qkv_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  if (e != cudaSuccess) return e;
  const int grid = p.ntiles < sm_count() ? p.ntiles : sm_count();
  k7_qkv_gemm_kernel<<<grid, kThreads, kSmem, st>>>(xm, wm, p);
  return cudaGetLastError();
}

}  // namespace fs
