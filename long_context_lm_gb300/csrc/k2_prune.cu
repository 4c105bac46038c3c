// k2_prune.cu -- FS-L availability sets (pools), linear in N.
//
// FreeSolo (paper.rainbus.top summary, 核心方法 and 方法步骤详情 ④; ai.info
// summary, "Methodology in Plain English"): before any query-dependent
// scoring each head keeps only the W most recent available cells plus the P
// cells with the largest max key norm a_c, a pool that changes only at
// query-block boundaries.
//
// For block beta with A = beta*Bq/s available cells and L = A - min(W, A)
// older cells, the kept older cells are the top-P of cells [0, L) ranked by
// (a_c desc, c asc).  Recomputing that per block from scratch is
// Theta(N^2/(Bq*s)); instead:
//   1. k2_chunk_sort: cells are cut into 64-cell chunks and each chunk is
//      sorted (one warp, bitonic network on 64-bit keys).
//   2. k2_chunk_scan: an inclusive prefix "merge, keep the top 64" over the
//      chunks (Hillis-Steele, one CTA per head; the merge is associative).
//   3. k2_emit: every block independently merges the prefix list of the
//      chunks below L with the sorted partial chunk [64*floor(L/64), L) and
//      writes the recent cells plus the first min(P, L) ranked cells.
// Steps 1 and 2 run as one kernel per head (k2_sort_scan) with the lists in
// shared memory while a head has at most kScanSmemChunks chunks (N up to
// 393216 at s = 32); longer heads take the two global-memory kernels.
// Keys are (float bits of a_c << 32) | (0xffffffff - c): larger key = higher
// rank, so the order is exact and equal norms rank the older cell first.
// Key 0 is padding and ranks below every real cell.
#include "fs_common.cuh"
#include "fs_internal.h"

namespace fs {

__device__ __forceinline__ uint64_t cell_key(float a, int c) {
  return (static_cast<uint64_t>(__float_as_uint(fmaxf(a, 0.f))) << 32) |
         static_cast<uint64_t>(0xffffffffu - static_cast<uint32_t>(c));
}
__device__ __forceinline__ int key_cell(uint64_t key) {
  return static_cast<int>(0xffffffffu - static_cast<uint32_t>(key & 0xffffffffu));
}
__device__ __forceinline__ uint64_t shfl_xor64(uint64_t x, int m) {
  uint32_t lo = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(x), m);
  uint32_t hi = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(x >> 32), m);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t shfl64(uint64_t x, int src) {
  uint32_t lo = __shfl_sync(0xffffffffu, static_cast<uint32_t>(x), src);
  uint32_t hi = __shfl_sync(0xffffffffu, static_cast<uint32_t>(x >> 32), src);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}

// One compare-exchange stage of a 64-element bitonic network held as two
// elements per lane (element e = 2*lane + r).  `k` is the size of the blocks
// being sorted (a block is descending when (e & k) == 0), `j` the distance.
__device__ __forceinline__ void bitonic_stage(uint64_t &x0, uint64_t &x1, int lane,
                                              int k, int j) {
  if (j == 1) {
    const bool desc = ((2 * lane) & k) == 0;
    const uint64_t hi = x0 > x1 ? x0 : x1, lo = x0 > x1 ? x1 : x0;
    x0 = desc ? hi : lo;
    x1 = desc ? lo : hi;
    return;
  }
  const int m = j >> 1;  // partner lane distance
  const uint64_t y0 = shfl_xor64(x0, m), y1 = shfl_xor64(x1, m);
  const int e0 = 2 * lane;
  const bool desc = (e0 & k) == 0;     // same for both elements of the lane
  const bool lower = (e0 & j) == 0;    // this lane holds the lower index
  const bool keep_max = (lower == desc);
  x0 = keep_max ? (x0 > y0 ? x0 : y0) : (x0 < y0 ? x0 : y0);
  x1 = keep_max ? (x1 > y1 ? x1 : y1) : (x1 < y1 ? x1 : y1);
}

// Sort 64 keys descending (two per lane, element 2*lane + r).
__device__ __forceinline__ void warp_sort64_desc(uint64_t &x0, uint64_t &x1, int lane) {
#pragma unroll
  for (int k = 2; k <= 64; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j >= 1; j >>= 1) bitonic_stage(x0, x1, lane, k, j);
}

// (a0,a1) and (b0,b1): two descending 64-lists.  Leaves the 64 largest keys of
// their union, descending, in (a0,a1).  max(A[i], B[63-i]) is the top half of
// the union as a bitonic sequence; a bitonic merge then sorts it.
__device__ __forceinline__ void warp_merge64_desc(uint64_t &a0, uint64_t &a1, uint64_t b0,
                                                  uint64_t b1, int lane) {
  const uint64_t rb0 = shfl64(b1, 31 - lane);  // B[63 - (2*lane)]
  const uint64_t rb1 = shfl64(b0, 31 - lane);  // B[63 - (2*lane+1)]
  a0 = a0 > rb0 ? a0 : rb0;
  a1 = a1 > rb1 ? a1 : rb1;
#pragma unroll
  for (int j = 32; j >= 1; j >>= 1) bitonic_stage(a0, a1, lane, 64, j);
}

__global__ void __launch_bounds__(128) k2_chunk_sort_kernel(
    const float *__restrict__ amax, int BH, int C, int nchunks, uint64_t *__restrict__ lists) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long gid = (long long)blockIdx.x * 4 + warp;
  if (gid >= (long long)BH * nchunks) return;
  const int bh = static_cast<int>(gid / nchunks), ch = static_cast<int>(gid % nchunks);
  const float *a = amax + (size_t)bh * C;
  const int c0 = ch * 64 + 2 * lane;
  uint64_t x0 = c0 < C ? cell_key(a[c0], c0) : 0ull;
  uint64_t x1 = c0 + 1 < C ? cell_key(a[c0 + 1], c0 + 1) : 0ull;
  warp_sort64_desc(x0, x1, lane);
  uint64_t *dst = lists + (size_t)gid * 64;
  dst[2 * lane] = x0;
  dst[2 * lane + 1] = x1;
}

// Inclusive prefix over the chunk lists of one head: after the call list i of
// the returned buffer holds the top 64 of chunks 0..i.
__global__ void __launch_bounds__(1024) k2_chunk_scan_kernel(uint64_t *buf0, uint64_t *buf1,
                                                             int nchunks) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const size_t base = (size_t)blockIdx.x * nchunks * 64;
  uint64_t *in = buf0 + base, *out = buf1 + base;
  for (int off = 1; off < nchunks; off <<= 1) {
    for (int i = warp; i < nchunks; i += nw) {
      uint64_t a0 = in[(size_t)i * 64 + 2 * lane], a1 = in[(size_t)i * 64 + 2 * lane + 1];
      if (i >= off) {
        const uint64_t b0 = in[(size_t)(i - off) * 64 + 2 * lane];
        const uint64_t b1 = in[(size_t)(i - off) * 64 + 2 * lane + 1];
        warp_merge64_desc(a0, a1, b0, b1, lane);
      }
      out[(size_t)i * 64 + 2 * lane] = a0;
      out[(size_t)i * 64 + 2 * lane + 1] = a1;
    }
    __syncthreads();
    uint64_t *t = in;
    in = out;
    out = t;
  }
}

// Steps 1 and 2 for one head in shared memory: every warp sorts chunks
// (warp w: chunks w, w + 32, ...), then the same inclusive prefix as
// k2_chunk_scan between two shared buffers; the result goes to `prefix`.
constexpr int kScanSmemChunks = 192;

__global__ void __launch_bounds__(1024) k2_sort_scan_kernel(const float *__restrict__ amax,
                                                            int C, int nchunks,
                                                            uint64_t *__restrict__ prefix,
                                                            uint64_t *__restrict__ sorted) {
  extern __shared__ uint64_t lists[];  // two buffers of nchunks x 64 keys
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int bh = blockIdx.x;
  const float *a = amax + (size_t)bh * C;
  uint64_t *in = lists, *out = lists + (size_t)nchunks * 64;
  for (int ch = warp; ch < nchunks; ch += nw) {
    const int c0 = ch * 64 + 2 * lane;
    uint64_t x0 = c0 < C ? cell_key(a[c0], c0) : 0ull;
    uint64_t x1 = c0 + 1 < C ? cell_key(a[c0 + 1], c0 + 1) : 0ull;
    warp_sort64_desc(x0, x1, lane);
    in[ch * 64 + 2 * lane] = x0;
    in[ch * 64 + 2 * lane + 1] = x1;
    uint64_t *sd = sorted + ((size_t)bh * nchunks + ch) * 64;  // for the emit's partial chunks
    sd[2 * lane] = x0;
    sd[2 * lane + 1] = x1;
  }
  __syncthreads();
  for (int off = 1; off < nchunks; off <<= 1) {
    for (int i = warp; i < nchunks; i += nw) {
      uint64_t a0 = in[i * 64 + 2 * lane], a1 = in[i * 64 + 2 * lane + 1];
      if (i >= off)
        warp_merge64_desc(a0, a1, in[(i - off) * 64 + 2 * lane], in[(i - off) * 64 + 2 * lane + 1],
                          lane);
      out[i * 64 + 2 * lane] = a0;
      out[i * 64 + 2 * lane + 1] = a1;
    }
    __syncthreads();
    uint64_t *t = in;
    in = out;
    out = t;
  }
  uint64_t *dst = prefix + (size_t)bh * nchunks * 64;
  for (int e = threadIdx.x; e < nchunks * 64; e += blockDim.x) dst[e] = in[e];
}

// The partial chunk [64 ci, L) in descending order: sorted here from the
// norms, or (kSorted) taken from the chunk's sorted list by keeping the cells
// below L in their order (the same keys in the same order as sorting them).
template <bool kSorted>
__global__ void __launch_bounds__(128) k2_emit_kernel(
    const float *__restrict__ amax, const uint64_t *__restrict__ prefix,
    const uint64_t *__restrict__ sorted, int BH, int C, int nchunks, int nblk,
    int cells_per_blk, int P, int W, int32_t *__restrict__ pool,
    int32_t *__restrict__ pool_count) {
  __shared__ uint64_t s_part[4][64];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long gid = (long long)blockIdx.x * 4 + warp;
  if (gid >= (long long)BH * nblk) return;
  const int bh = static_cast<int>(gid / nblk), beta = static_cast<int>(gid % nblk);
  const int A = beta * cells_per_blk;
  const int nrec = A < W ? A : W;
  const int L = A - nrec;
  const int cap = P + W;
  int32_t *pl = pool + (size_t)gid * cap;
  for (int r = lane; r < nrec; r += 32) pl[r] = L + r;
  const int keep = L < P ? L : P;
  if (L > 0) {
    const int ci = L / 64, rem = L % 64;
    uint64_t x0 = 0ull, x1 = 0ull;
    if (kSorted) {
      if (rem > 0) {
        // compact the chunk's sorted keys of cells below L, order kept
        const uint64_t *sd = sorted + ((size_t)bh * nchunks + ci) * 64;
        const uint64_t y0 = sd[2 * lane], y1 = sd[2 * lane + 1];
        const bool k0 = y0 != 0ull && key_cell(y0) < L, k1 = y1 != 0ull && key_cell(y1) < L;
        const uint32_t b0 = __ballot_sync(0xffffffffu, k0), b1 = __ballot_sync(0xffffffffu, k1);
        const uint32_t below = (1u << lane) - 1u;
        const int pos = __popc(b0 & below) + __popc(b1 & below);
        __syncwarp();
        if (k0) s_part[warp][pos] = y0;
        if (k1) s_part[warp][pos + (k0 ? 1 : 0)] = y1;
        __syncwarp();
        x0 = 2 * lane < rem ? s_part[warp][2 * lane] : 0ull;
        x1 = 2 * lane + 1 < rem ? s_part[warp][2 * lane + 1] : 0ull;
      }
    } else {
      const float *a = amax + (size_t)bh * C;
      const int c0 = ci * 64 + 2 * lane;
      if (2 * lane < rem) x0 = cell_key(a[c0], c0);
      if (2 * lane + 1 < rem) x1 = cell_key(a[c0 + 1], c0 + 1);
      warp_sort64_desc(x0, x1, lane);
    }
    if (ci > 0) {
      const uint64_t *pf = prefix + ((size_t)bh * nchunks + (ci - 1)) * 64;
      warp_merge64_desc(x0, x1, pf[2 * lane], pf[2 * lane + 1], lane);
    }
    if (2 * lane < keep) pl[nrec + 2 * lane] = key_cell(x0);
    if (2 * lane + 1 < keep) pl[nrec + 2 * lane + 1] = key_cell(x1);
  }
  for (int r = nrec + keep + lane; r < cap; r += 32) pl[r] = -1;
  if (lane == 0) pool_count[gid] = nrec + keep;
}

size_t prune_workspace_bytes(const Shape &sh) {
  const size_t nchunks = (size_t)(sh.C() + 63) / 64;
  return 2 * (size_t)sh.BH() * nchunks * 64 * sizeof(uint64_t);
}

cudaError_t launch_prune(const float *amax, const Shape &sh, int P, int W, int32_t *pool,
                         int32_t *pool_count, void *ws, cudaStream_t st) {
  const int C = sh.C();
  const int nchunks = (C + 63) / 64;
  const int BH = sh.BH();
  uint64_t *buf0 = static_cast<uint64_t *>(ws);
  uint64_t *buf1 = buf0 + (size_t)BH * nchunks * 64;
  const uint64_t *prefix = buf0;
  const long long nwarps = (long long)BH * sh.nblk();
  const unsigned egrid = (unsigned)((nwarps + 3) / 4);
  if (nchunks <= kScanSmemChunks) {
    const int smem = 2 * nchunks * 64 * (int)sizeof(uint64_t);
    cudaError_t e = cudaFuncSetAttribute(k2_sort_scan_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    k2_sort_scan_kernel<<<BH, 1024, smem, st>>>(amax, C, nchunks, buf0, buf1);
    k2_emit_kernel<true><<<egrid, 128, 0, st>>>(amax, buf0, buf1, BH, C, nchunks, sh.nblk(),
                                                kBq / kS, P, W, pool, pool_count);
  } else {
    const long long nlists = (long long)BH * nchunks;
    k2_chunk_sort_kernel<<<(unsigned)((nlists + 3) / 4), 128, 0, st>>>(amax, BH, C, nchunks,
                                                                       buf0);
    int levels = 0;
    for (int off = 1; off < nchunks; off <<= 1) ++levels;
    if (levels > 0) k2_chunk_scan_kernel<<<BH, 1024, 0, st>>>(buf0, buf1, nchunks);
    prefix = (levels % 2 == 0) ? buf0 : buf1;
    k2_emit_kernel<false><<<egrid, 128, 0, st>>>(amax, prefix, nullptr, BH, C, nchunks,
                                                 sh.nblk(), kBq / kS, P, W, pool, pool_count);
  }
  return cudaGetLastError();
}

}  // namespace fs
