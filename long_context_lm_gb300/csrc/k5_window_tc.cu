// k5_window_tc.cu -- sliding-window RoPE branch on the 5th-generation tensor
// cores (tcgen05 + TMEM), with the branch mix fused into the epilogue.
//
// FreeSolo (paper.rainbus.top summary, 方法步骤详情 ② "在 w=512 窗口内做 RoPE
// 注意力" and ⑥ "与局部分支相加"; 前置知识 RoPE; ai.info summary, "Methodology
// in Plain English"):
//     o_win[n] = softmax_j((R(n) q_n . R(j) k_j) / sqrt(d)) v_j,  j in [n-w+1, n]
//     out[n]   = o_win[n] + mix_h * o_long[n].
//
// One CTA (12 warps, one per SM) owns two adjacent 128-query tiles A and B of
// one head and walks the 64-key tiles that cover both windows:
//   warps 0-3   softmax of tile A (thread = query row = TMEM lane)
//   warps 4-7   softmax of tile B
//   warp  8     TMEM allocation and the single MMA-issuing thread
//   warp  9     TMA producer: raw key tile and value tile of each key tile
//   warps 10-11 rotate the queries once and every raw key tile once
// RoPE is applied relative to tile A's first position b: q_n.k_j after
// rotations by n-b and j-b equals the absolute-position product (R is
// orthogonal and depends only on differences), so both query tiles share one
// rotated copy of each key tile, and the angles stay small (|j-b| < w+256).
// The rotated q and k are split into bf16 hi + lo halves; S = Q.K^T takes
// three tcgen05.mma chains (hi.hi + hi.lo + lo.hi) accumulating in TMEM, which
// keeps logits at ~2^-16 relative error (a single bf16 rounding of the
// rotated vectors exceeds the output tolerance on lognormal keys).  P is
// written as bf16 into a swizzled shared tile and P.V accumulates into a TMEM
// O that the softmax threads rescale when their running max grows.
#include <cuda.h>

#include "fs_common.cuh"
#include "fs_internal.h"
#include "tc05.cuh"

namespace fs {
namespace {

constexpr int kKT = 64;       // keys per tile
constexpr int kRing = 3;      // raw-key / value ring depth
constexpr int kRot = 2;       // rotated-key ring depth
constexpr int kThreads = 384;

// shared-memory layout, offsets from a 1024-byte aligned base
constexpr uint32_t kOffQ = 0;           // [A hi, A lo, B hi, B lo] x 16 KB
constexpr uint32_t kOffP = 65536;       // [A, B] x 16 KB
constexpr uint32_t kOffKT = 98304;      // kRot x [hi 8 KB, lo 8 KB]
constexpr uint32_t kOffV = kOffKT + kRot * 16384;       // kRing x 8 KB
constexpr uint32_t kOffKRaw = kOffV + kRing * 8192;     // kRing x 8 KB
constexpr uint32_t kSmemUsed = kOffKRaw + kRing * 8192; // 176 KB
constexpr uint32_t kSmemBytes = kSmemUsed + 1024;       // + alignment slack

// TMEM columns: S_A, O_A, S_B, O_B (64 fp32 columns each)
constexpr uint32_t kTmemCols = 256;

struct Barriers {
  uint64_t q_full;
  uint64_t raw_full[kRing];
  uint64_t raw_empty[kRing];
  uint64_t v_empty[kRing];
  uint64_t kt_full[kRot];
  uint64_t kt_empty[kRot];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t fin;
  uint32_t tmem;
};

struct Params {
  const __nv_bfloat16 *q;
  const float *o_long;
  const float *mix;
  const float2 *rel;  // (cos, sin) of t*theta_i, row t + rel_off
  int rel_off;
  int H, N, w, nblk;
  float *out;
  int *err;
};

// Rotate one 64-element row (bf16, 8 chunks of 8) by the angles of table row
// `cs` and write bf16 hi / lo halves into two swizzled tiles at row r.
__device__ __forceinline__ void rotate_row(const uint4 (&x)[8], const float2 *__restrict__ cs,
                                           unsigned char *hi, unsigned char *lo, int r) {
#pragma unroll
  for (int ig = 0; ig < 4; ++ig) {
    const uint32_t wa[4] = {x[ig].x, x[ig].y, x[ig].z, x[ig].w};
    const uint32_t wb[4] = {x[ig + 4].x, x[ig + 4].y, x[ig + 4].z, x[ig + 4].w};
    uint32_t ah[4], al[4], bh[4], bl[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 t = __ldg(reinterpret_cast<const float4 *>(cs + 8 * ig + 2 * j));
      float y0[2], y1[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float c = e ? t.z : t.x, s = e ? t.w : t.y;
        const float x0 = e ? bf16_hi(wa[j]) : bf16_lo(wa[j]);
        const float x1 = e ? bf16_hi(wb[j]) : bf16_lo(wb[j]);
        y0[e] = x0 * c - x1 * s;
        y1[e] = x0 * s + x1 * c;
      }
      ah[j] = pack_bf16(y0[0], y0[1]);
      al[j] = pack_bf16(y0[0] - bf16_lo(ah[j]), y0[1] - bf16_hi(ah[j]));
      bh[j] = pack_bf16(y1[0], y1[1]);
      bl[j] = pack_bf16(y1[0] - bf16_lo(bh[j]), y1[1] - bf16_hi(bh[j]));
    }
    *reinterpret_cast<uint4 *>(hi + swz128(r, ig)) = make_uint4(ah[0], ah[1], ah[2], ah[3]);
    *reinterpret_cast<uint4 *>(hi + swz128(r, ig + 4)) = make_uint4(bh[0], bh[1], bh[2], bh[3]);
    *reinterpret_cast<uint4 *>(lo + swz128(r, ig)) = make_uint4(al[0], al[1], al[2], al[3]);
    *reinterpret_cast<uint4 *>(lo + swz128(r, ig + 4)) = make_uint4(bl[0], bl[1], bl[2], bl[3]);
  }
}

struct TileRange {
  int kt0;      // first key of tile 0
  int ntiles;   // tiles walked by the CTA
  int begin[2]; // first tile of query tile A / B
  int end[2];   // one past the last tile of A / B (end <= begin: tile absent)
  int q0[2];    // first query of A / B
};

__device__ __forceinline__ TileRange tile_range(int pair, int nblk, int w) {
  TileRange tr;
  const bool has_b = 2 * pair + 1 < nblk;
  tr.q0[0] = pair * 2 * kBq;
  tr.q0[1] = tr.q0[0] + kBq;
  tr.kt0 = max(0, tr.q0[0] - w + 1) / kKT * kKT;
  const int last = has_b ? tr.q0[1] + kBq : tr.q0[0] + kBq;
  tr.ntiles = (last - tr.kt0) / kKT;
  tr.begin[0] = 0;
  tr.end[0] = (tr.q0[0] + kBq - tr.kt0) / kKT;
  tr.begin[1] = (max(0, tr.q0[1] - w + 1) / kKT * kKT - tr.kt0) / kKT;
  tr.end[1] = has_b ? tr.ntiles : tr.begin[1];
  return tr;
}

__device__ __forceinline__ bool uses(const TileRange &tr, int x, int t) {
  return t >= tr.begin[x] && t < tr.end[x];
}

// --------------------------------------------------------------------------
// roles
// --------------------------------------------------------------------------

__device__ void role_mma(const TileRange &tr, Barriers &bar, uint32_t tmem, uint32_t base,
                         int *err) {
  const uint32_t id_qk = tc::idesc_bf16(128, kKT, 0);
  const uint32_t id_pv = tc::idesc_bf16(128, kD, 1);
  const uint32_t sQ = base + kOffQ, sP = base + kOffP;
  if (!tc::mbar_wait(&bar.q_full, 0, err)) return;
  for (int t = 0; t <= tr.ntiles; ++t) {
    const bool tile = t < tr.ntiles;
    if (tile) {
      if (!tc::mbar_wait(&bar.kt_full[t % kRot], (t / kRot) & 1, err)) return;
    }
    tc::fence_after_sync();
    const uint32_t sKh = base + kOffKT + (t % kRot) * 16384, sKl = sKh + 8192;
    bool any_pv = false;
    for (int x = 0; x < 2; ++x) {
      const uint32_t s_col = tmem + x * 128, o_col = s_col + 64;
      // P.V of this query tile's previous key tile
      if (t > 0 && uses(tr, x, t - 1)) {
        const int i = t - 1 - tr.begin[x];
        if (!tc::mbar_wait(&bar.p_full[x], i & 1, err)) return;
        tc::fence_after_sync();
        const uint32_t sV = base + kOffV + ((t - 1) % kRing) * 8192;
        const uint32_t pa = sP + x * 16384;
#pragma unroll
        for (int k = 0; k < kKT / 16; ++k)
          tc::mma_ss(o_col, tc::desc_sw128(pa + 32 * k), tc::desc_sw128(sV + 2048 * k), id_pv,
                     (i > 0 || k > 0) ? 1u : 0u);
        any_pv = true;
        if (t == tr.end[x]) tc::mma_commit(&bar.o_done[x]);
      }
      // S = Q.K^T of this key tile (three split-precision chains)
      if (tile && uses(tr, x, t)) {
        const uint32_t qh = sQ + x * 32768, ql = qh + 16384;
#pragma unroll
        for (int part = 0; part < 3; ++part) {
          const uint32_t a = part == 2 ? ql : qh, b = part == 1 ? sKl : sKh;
#pragma unroll
          for (int k = 0; k < kD / 16; ++k)
            tc::mma_ss(s_col, tc::desc_sw128(a + 32 * k), tc::desc_sw128(b + 32 * k), id_qk,
                       (part > 0 || k > 0) ? 1u : 0u);
        }
        tc::mma_commit(&bar.s_full[x]);
      }
    }
    if (any_pv) tc::mma_commit(&bar.v_empty[(t - 1) % kRing]);
    if (tile) tc::mma_commit(&bar.kt_empty[t % kRot]);
  }
}

__device__ void role_tma(const TileRange &tr, Barriers &bar, unsigned char *smem,
                         const CUtensorMap *tk, const CUtensorMap *tv, int row0, int *err) {
  for (int t = 0; t < tr.ntiles; ++t) {
    const int slot = t % kRing;
    if (t >= kRing) {
      const uint32_t ph = ((t / kRing) - 1) & 1;
      if (!tc::mbar_wait(&bar.raw_empty[slot], ph, err)) return;
      if (!tc::mbar_wait(&bar.v_empty[slot], ph, err)) return;
    }
    tc::mbar_arrive_expect_tx(&bar.raw_full[slot], 2 * kKT * kD * 2);
    const int y = row0 + tr.kt0 + t * kKT;
    tc::tma_load_2d(smem + kOffKRaw + slot * 8192, tk, &bar.raw_full[slot], 0, y);
    tc::tma_load_2d(smem + kOffV + slot * 8192, tv, &bar.raw_full[slot], 0, y);
  }
}

__device__ void role_rotate(const TileRange &tr, Barriers &bar, unsigned char *smem,
                            const Params &p, size_t head, int tr_id, int *err) {
  // queries: rows tr_id and tr_id + 64 of A and of B (B only if present)
  for (int x = 0; x < 2; ++x) {
    if (tr.end[x] <= tr.begin[x]) continue;
    for (int rr = 0; rr < 2; ++rr) {
      const int r = tr_id + 64 * rr;
      const int n = tr.q0[x] + r;
      const uint4 *src = reinterpret_cast<const uint4 *>(p.q + (head + n) * kD);
      uint4 raw[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) raw[c] = __ldg(src + c);
      unsigned char *qh = smem + kOffQ + x * 32768;
      rotate_row(raw, p.rel + (size_t)(n - tr.q0[0] + p.rel_off) * (kD / 2), qh, qh + 16384, r);
    }
  }
  tc::fence_async_smem();
  tc::mbar_arrive(&bar.q_full);
  for (int t = 0; t < tr.ntiles; ++t) {
    const int slot = t % kRing, s = t % kRot;
    if (!tc::mbar_wait(&bar.raw_full[slot], (t / kRing) & 1, err)) return;
    if (t >= kRot && !tc::mbar_wait(&bar.kt_empty[s], ((t / kRot) - 1) & 1, err)) return;
    const unsigned char *kr = smem + kOffKRaw + slot * 8192;
    uint4 raw[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) raw[c] = *reinterpret_cast<const uint4 *>(kr + swz128(tr_id, c));
    const int j = tr.kt0 + t * kKT + tr_id;
    unsigned char *kh = smem + kOffKT + s * 16384;
    rotate_row(raw, p.rel + (size_t)(j - tr.q0[0] + p.rel_off) * (kD / 2), kh, kh + 8192, tr_id);
    tc::fence_async_smem();
    tc::mbar_arrive(&bar.kt_full[s]);
    tc::mbar_arrive(&bar.raw_empty[slot]);
  }
}

__device__ void role_softmax(const TileRange &tr, Barriers &bar, unsigned char *smem,
                             uint32_t tmem, const Params &p, size_t head, int h, int x, int r,
                             int *err) {
  const int warp = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t s_addr = tmem + x * 128 + lane_base, o_addr = s_addr + 64;
  const int n = tr.q0[x] + r;
  const float sl2 = 1.4426950408889634f * 0.125f;  // log2(e) / sqrt(64)
  unsigned char *prow = smem + kOffP + x * 16384;
  float m = -INFINITY, l = 0.f;
  for (int t = tr.begin[x]; t < tr.end[x]; ++t) {
    const int i = t - tr.begin[x];
    if (!tc::mbar_wait(&bar.s_full[x], i & 1, err)) return;
    tc::fence_after_sync();
    const int kt = tr.kt0 + t * kKT;
    const int lo = max(0, n - p.w + 1 - kt), hi = min(kKT - 1, n - kt);
    const bool any = lo <= hi;
    uint32_t pk[32];
    if (__any_sync(0xffffffffu, any)) {
      uint32_t s0[32], s1[32];
      tc::tmem_ld32(s_addr, s0);
      tc::tmem_ld32(s_addr + 32, s1);
      tc::tmem_wait_ld();
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        if (c >= lo && c <= hi) mx = fmaxf(mx, __uint_as_float(s0[c]));
        if (c + 32 >= lo && c + 32 <= hi) mx = fmaxf(mx, __uint_as_float(s1[c]));
      }
      const float mnew = fmaxf(m, mx * sl2);
      const float alpha = (mnew == m) ? 1.f : tc::ex2(m - mnew);
      float ls = 0.f;
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        float e0 = (c >= lo && c <= hi) ? tc::ex2(fmaf(__uint_as_float(s0[c]), sl2, -mnew)) : 0.f;
        float e1 = (c + 1 >= lo && c + 1 <= hi)
                       ? tc::ex2(fmaf(__uint_as_float(s0[c + 1]), sl2, -mnew)) : 0.f;
        float f0 = (c + 32 >= lo && c + 32 <= hi)
                       ? tc::ex2(fmaf(__uint_as_float(s1[c]), sl2, -mnew)) : 0.f;
        float f1 = (c + 33 >= lo && c + 33 <= hi)
                       ? tc::ex2(fmaf(__uint_as_float(s1[c + 1]), sl2, -mnew)) : 0.f;
        ls += (e0 + e1) + (f0 + f1);
        pk[c / 2] = pack_bf16(e0, e1);
        pk[16 + c / 2] = pack_bf16(f0, f1);
      }
      l = l * alpha + ls;
      m = mnew;
      if (i > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        uint32_t o0[32], o1[32];
        tc::tmem_ld32(o_addr, o0);
        tc::tmem_ld32(o_addr + 32, o1);
        tc::tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          o0[c] = __float_as_uint(__uint_as_float(o0[c]) * alpha);
          o1[c] = __float_as_uint(__uint_as_float(o1[c]) * alpha);
        }
        tc::tmem_st32(o_addr, o0);
        tc::tmem_st32(o_addr + 32, o1);
        tc::tmem_wait_st();
      }
    } else {
#pragma unroll
      for (int c = 0; c < 32; ++c) pk[c] = 0u;
    }
#pragma unroll
    for (int ch = 0; ch < 8; ++ch)
      *reinterpret_cast<uint4 *>(prow + swz128(r, ch)) =
          make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&bar.p_full[x]);
  }
  // epilogue: O / l (+ mix_h * o_long)
  if (!tc::mbar_wait(&bar.o_done[x], 0, err)) return;
  tc::fence_after_sync();
  uint32_t o0[32], o1[32];
  tc::tmem_ld32(o_addr, o0);
  tc::tmem_ld32(o_addr + 32, o1);
  tc::tmem_wait_ld();
  const float inv = 1.f / l;
  const float mh = p.mix ? p.mix[h] : 0.f;
  float4 *dst = reinterpret_cast<float4 *>(p.out + (head + n) * kD);
  const float4 *ol = p.o_long ? reinterpret_cast<const float4 *>(p.o_long + (head + n) * kD) : nullptr;
#pragma unroll
  for (int c4 = 0; c4 < 16; ++c4) {
    const uint32_t *src = c4 < 8 ? o0 : o1;
    const int b = (c4 & 7) * 4;
    float4 v = make_float4(__uint_as_float(src[b]) * inv, __uint_as_float(src[b + 1]) * inv,
                           __uint_as_float(src[b + 2]) * inv, __uint_as_float(src[b + 3]) * inv);
    if (ol) {
      const float4 u = __ldg(ol + c4);
      v.x = fmaf(mh, u.x, v.x);
      v.y = fmaf(mh, u.y, v.y);
      v.z = fmaf(mh, u.z, v.z);
      v.w = fmaf(mh, u.w, v.w);
    }
    dst[c4] = v;
  }
}

__global__ void __launch_bounds__(kThreads, 1) k5_window_tc_kernel(
    const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
    const Params p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Barriers bar;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = blockIdx.x, bh = blockIdx.y, h = bh % p.H;
  const size_t head = (size_t)bh * p.N;
  const TileRange tr = tile_range(pair, p.nblk, p.w);

  if (threadIdx.x == 0) {
    tc::mbar_init(&bar.q_full, 64);
    for (int i = 0; i < kRing; ++i) {
      tc::mbar_init(&bar.raw_full[i], 1);
      tc::mbar_init(&bar.raw_empty[i], 64);
      tc::mbar_init(&bar.v_empty[i], 1);
    }
    for (int i = 0; i < kRot; ++i) {
      tc::mbar_init(&bar.kt_full[i], 64);
      tc::mbar_init(&bar.kt_empty[i], 1);
    }
    for (int x = 0; x < 2; ++x) {
      tc::mbar_init(&bar.s_full[x], 1);
      tc::mbar_init(&bar.p_full[x], 4);
      tc::mbar_init(&bar.o_done[x], 1);
    }
    tc::mbar_init(&bar.fin, 1);
    tc::mbar_fence_init();
  }
  if (warp == 8) {
    tc::tmem_alloc(&bar.tmem, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bar.tmem;
  const uint32_t sbase = smem_u32(smem);

  if (warp < 8) {
    const int x = warp >> 2;
    if (tr.end[x] > tr.begin[x])
      role_softmax(tr, bar, smem, tmem, p, head, h, x, threadIdx.x & 127, p.err);
  } else if (warp == 8) {
    if (lane == 0) {
      role_mma(tr, bar, tmem, sbase, p.err);
      tc::mma_commit(&bar.fin);  // every issued MMA has completed once this arrives
      tc::mbar_wait(&bar.fin, 0, p.err);
    }
  } else if (warp == 9) {
    if (lane == 0) role_tma(tr, bar, smem, &tmap_k, &tmap_v, (int)head, p.err);
  } else {
    role_rotate(tr, bar, smem, p, head, threadIdx.x - 320, p.err);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 8) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

__global__ void rel_rope_table_kernel(float2 *__restrict__ tab, int rows, int off, double base) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * (kD / 2)) return;
  const int row = idx / (kD / 2), i = idx % (kD / 2);
  const double theta = pow(base, -2.0 * (double)i / (double)kD);
  double s, c;
  sincos((double)(row - off) * theta, &s, &c);
  tab[idx] = make_float2((float)c, (float)s);
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

// [rows, 64] bf16 row-major, boxes of 64 x 64 with the 128-byte swizzle.
bool make_rows_map(CUtensorMap *map, const void *ptr, size_t rows) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kD, (cuuint32_t)kKT};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Relative-angle table rows: offsets t in [-rel_off, 2*kBq).
int window_rel_offset(int w) { return (w + 62 + kKT - 1) / kKT * kKT; }
size_t window_table_bytes(int w) {
  return (size_t)(window_rel_offset(w) + 2 * kBq) * (kD / 2) * sizeof(float2);
}

cudaError_t launch_window_tc(const void *q, const void *k, const void *v, const float *o_long,
                             const float *mix, void *table, const Shape &sh, int w, float base,
                             float *out, int *err, cudaStream_t st) {
  const int off = window_rel_offset(w);
  const int rows = off + 2 * kBq;
  float2 *tab = static_cast<float2 *>(table);
  rel_rope_table_kernel<<<(rows * (kD / 2) + 255) / 256, 256, 0, st>>>(tab, rows, off, (double)base);
  CUtensorMap mk, mv;
  const size_t nrows = (size_t)sh.BH() * sh.N;
  if (!make_rows_map(&mk, k, nrows) || !make_rows_map(&mv, v, nrows)) return cudaErrorInvalidValue;
  Params p;
  p.q = static_cast<const __nv_bfloat16 *>(q);
  p.o_long = o_long;
  p.mix = mix;
  p.rel = tab;
  p.rel_off = off;
  p.H = sh.H;
  p.N = sh.N;
  p.w = w;
  p.nblk = sh.nblk();
  p.out = out;
  p.err = err;
  cudaError_t e = cudaFuncSetAttribute(k5_window_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid((sh.nblk() + 1) / 2, sh.BH());
  k5_window_tc_kernel<<<grid, kThreads, kSmemBytes, st>>>(mk, mv, p);
  return cudaGetLastError();
}

}  // namespace fs
