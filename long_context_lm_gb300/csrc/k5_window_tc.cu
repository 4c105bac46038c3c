// k5_window_tc.cu -- sliding-window RoPE branch on the 5th-generation tensor
// cores (tcgen05 + TMEM), with the branch mix fused into the epilogue.
//
// FreeSolo (paper.rainbus.top summary, 方法步骤详情 ② "在 w=512 窗口内做 RoPE
// 注意力" and ⑥ "与局部分支相加"; 前置知识 RoPE; ai.info summary, "Methodology
// in Plain English"):
//     o_win[n] = softmax_j((R(n) q_n . R(j) k_j) / sqrt(d)) v_j,  j in [n-w+1, n]
//     out[n]   = o_win[n] + mix_h * o_long[n].
//
// One CTA (14 warps, one per SM) owns two adjacent 128-query tiles A and B of
// one head and walks the 64-key tiles that cover both windows:
//   warps 0-3   softmax of tile A (thread = query row = TMEM lane)
//   warps 4-7   softmax of tile B
//   warp  8     TMEM allocation and the single MMA-issuing thread
//   warp  9     TMA producer: key tile and value tile of each key tile
//   warps 10-13 rotate the queries once and every key tile once, in place
//               (two threads per 64-element row, disjoint 16-byte chunks)
// RoPE is applied relative to tile A's first position b: q_n.k_j after
// rotations by n-b and j-b equals the absolute-position product (R is
// orthogonal and depends only on differences), so both query tiles share one
// rotated copy of each key tile, and the angles stay small (|j-b| < w+256).
// An offset t = 64*u + r is rotated with cos/sin of t*theta_i formed by the
// angle-sum identity from two small shared tables (r*theta_i for r < 64 and
// the few tile bases 64*u*theta_i), both taken from an fp64-computed table.
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
constexpr int kRing = 3;      // key / value ring depth (keys rotated in place)
constexpr int kThreads = 448;

// shared-memory layout, offsets from a 1024-byte aligned base
constexpr uint32_t kOffQ = 0;                           // [A hi, A lo, B hi, B lo] x 16 KB
constexpr uint32_t kOffP = 65536;                       // [A, B] x 16 KB
constexpr uint32_t kOffK = 98304;                       // kRing x [hi 8 KB, lo 8 KB]
constexpr uint32_t kOffV = kOffK + kRing * 16384;       // kRing x 8 KB
constexpr uint32_t kOffT64 = kOffV + kRing * 8192;      // 64 x 32 (cos, sin): 16 KB
constexpr uint32_t kOffTB = kOffT64 + 64 * 256;         // bases x 32 (cos, sin)
// key tiles a CTA walks at most, and the dynamic shared memory it needs
__host__ __device__ constexpr int max_tiles(int w) { return (w + 318) / kKT + 1; }
__host__ __device__ constexpr uint32_t smem_bytes(int w) {
  return kOffTB + (4 + max_tiles(w)) * 256 + 1024;
}

// TMEM columns: S_A, O_A, S_B, O_B (64 fp32 columns each)
constexpr uint32_t kTmemCols = 256;

struct Barriers {
  uint64_t q_full;
  uint64_t raw_full[kRing];   // TMA: key and value tile landed
  uint64_t kt_full[kRing];    // key tile rotated
  uint64_t kt_empty[kRing];   // S MMAs of the tile done
  uint64_t v_empty[kRing];    // P.V MMAs of the tile done
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

// Rotate half of one 64-element row in place: pairs i in [16*half, 16*half+16)
// (dims 16*half.. and 32+16*half..), angles from the shared tables t64 (row
// offset r) and tb (tile base), composed by the angle-sum identity.  The raw
// row is read from `hi` (chunks 2*half, 2*half+1, 4+2*half, 5+2*half) and the
// rotated bf16 hi / lo halves are written back to the same chunks of `hi`
// and `lo`.
__device__ __forceinline__ void rotate_half_row(unsigned char *hi, unsigned char *lo, int r,
                                                int half, const float2 *t64r,
                                                const float2 *tbr) {
  uint4 xa[2], xb[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    xa[k] = *reinterpret_cast<const uint4 *>(hi + swz128(r, 2 * half + k));
    xb[k] = *reinterpret_cast<const uint4 *>(hi + swz128(r, 4 + 2 * half + k));
  }
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const uint32_t wa[4] = {xa[k].x, xa[k].y, xa[k].z, xa[k].w};
    const uint32_t wb[4] = {xb[k].x, xb[k].y, xb[k].z, xb[k].w};
    uint32_t ah[4], al[4], bh[4], bl[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i0 = 16 * half + 8 * k + 2 * j;  // first pair of this 32-bit word
      const float4 rr = *reinterpret_cast<const float4 *>(t64r + i0);
      const float4 bb = *reinterpret_cast<const float4 *>(tbr + i0);
      float y0[2], y1[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float cr = e ? rr.z : rr.x, sr = e ? rr.w : rr.y;
        const float cb = e ? bb.z : bb.x, sb = e ? bb.w : bb.y;
        const float c = fmaf(cb, cr, -sb * sr), sn = fmaf(sb, cr, cb * sr);
        const float x0 = e ? bf16_hi(wa[j]) : bf16_lo(wa[j]);
        const float x1 = e ? bf16_hi(wb[j]) : bf16_lo(wb[j]);
        y0[e] = fmaf(x0, c, -x1 * sn);
        y1[e] = fmaf(x0, sn, x1 * c);
      }
      ah[j] = pack_bf16(y0[0], y0[1]);
      al[j] = pack_bf16(y0[0] - bf16_lo(ah[j]), y0[1] - bf16_hi(ah[j]));
      bh[j] = pack_bf16(y1[0], y1[1]);
      bl[j] = pack_bf16(y1[0] - bf16_lo(bh[j]), y1[1] - bf16_hi(bh[j]));
    }
    const int ca = 2 * half + k, cb = 4 + 2 * half + k;
    *reinterpret_cast<uint4 *>(hi + swz128(r, ca)) = make_uint4(ah[0], ah[1], ah[2], ah[3]);
    *reinterpret_cast<uint4 *>(hi + swz128(r, cb)) = make_uint4(bh[0], bh[1], bh[2], bh[3]);
    *reinterpret_cast<uint4 *>(lo + swz128(r, ca)) = make_uint4(al[0], al[1], al[2], al[3]);
    *reinterpret_cast<uint4 *>(lo + swz128(r, cb)) = make_uint4(bl[0], bl[1], bl[2], bl[3]);
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
      if (!tc::mbar_wait(&bar.kt_full[t % kRing], (t / kRing) & 1, err)) return;
    }
    tc::fence_after_sync();
    const uint32_t sKh = base + kOffK + (t % kRing) * 16384, sKl = sKh + 8192;
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
    if (tile) tc::mma_commit(&bar.kt_empty[t % kRing]);
  }
}

__device__ void role_tma(const TileRange &tr, Barriers &bar, unsigned char *smem,
                         const CUtensorMap *tk, const CUtensorMap *tv, int row0, int *err) {
  for (int t = 0; t < tr.ntiles; ++t) {
    const int slot = t % kRing;
    if (t >= kRing) {
      const uint32_t ph = ((t / kRing) - 1) & 1;
      if (!tc::mbar_wait(&bar.kt_empty[slot], ph, err)) return;
      if (!tc::mbar_wait(&bar.v_empty[slot], ph, err)) return;
    }
    tc::mbar_arrive_expect_tx(&bar.raw_full[slot], 2 * kKT * kD * 2);
    const int y = row0 + tr.kt0 + t * kKT;
    tc::tma_load_2d(smem + kOffK + slot * 16384, tk, &bar.raw_full[slot], 0, y);
    tc::tma_load_2d(smem + kOffV + slot * 8192, tv, &bar.raw_full[slot], 0, y);
  }
}

// Table rows of the tile bases: [0, 4) query bases 0, 64, 128, 192 relative to
// tile A; [4, 4 + ntiles) key-tile bases kt0 + 64 t - q0[A].
__device__ void role_rotate(const TileRange &tr, Barriers &bar, unsigned char *smem,
                            const Params &p, size_t head, int tid_r, int *err) {
  const float2 *t64 = reinterpret_cast<const float2 *>(smem + kOffT64);
  const float2 *tb = reinterpret_cast<const float2 *>(smem + kOffTB);
  const int r = tid_r >> 1, half = tid_r & 1;  // key row 0..63, half row
  // queries: raw rows -> hi tile, then rotate in place; thread handles rows
  // r and r + 64 (half of each) of A and of B
  for (int x = 0; x < 2; ++x) {
    if (tr.end[x] <= tr.begin[x]) continue;
    unsigned char *qh = smem + kOffQ + x * 32768;
    for (int rr = 0; rr < 2; ++rr) {
      const int row = r + 64 * rr;
      const uint4 *src = reinterpret_cast<const uint4 *>(p.q + (head + tr.q0[x] + row) * kD);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int ca = 2 * half + k, cb = 4 + 2 * half + k;
        *reinterpret_cast<uint4 *>(qh + swz128(row, ca)) = __ldg(src + ca);
        *reinterpret_cast<uint4 *>(qh + swz128(row, cb)) = __ldg(src + cb);
      }
      rotate_half_row(qh, qh + 16384, row, half, t64 + r * (kD / 2),
                      tb + (2 * x + rr) * (kD / 2));
    }
  }
  tc::fence_async_smem();
  tc::mbar_arrive(&bar.q_full);
  for (int t = 0; t < tr.ntiles; ++t) {
    const int slot = t % kRing;
    if (!tc::mbar_wait(&bar.raw_full[slot], (t / kRing) & 1, err)) return;
    unsigned char *kh = smem + kOffK + slot * 16384;
    rotate_half_row(kh, kh + 8192, r, half, t64 + r * (kD / 2), tb + (4 + t) * (kD / 2));
    tc::fence_async_smem();
    tc::mbar_arrive(&bar.kt_full[slot]);
  }
}

// One row of a 64-key score tile: running max m and sum l (log2 domain,
// scale sl2 folded in), bf16 probabilities packed two per word into pk, and
// the factor alpha that rescales the row's earlier accumulation.  kMask:
// only columns [lo, hi] are inside the row's window.
template <bool kMask>
__device__ __forceinline__ void softmax_row(const uint32_t (&s0)[32], const uint32_t (&s1)[32],
                                            int lo, int hi, float sl2, float &m, float &l,
                                            float &alpha, uint32_t (&pk)[32]) {
  auto in = [&](int c) { return !kMask || (c >= lo && c <= hi); };
  float mx = -INFINITY;
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    if (in(c)) mx = fmaxf(mx, __uint_as_float(s0[c]));
    if (in(c + 32)) mx = fmaxf(mx, __uint_as_float(s1[c]));
  }
  const float mnew = fmaxf(m, mx * sl2);
  alpha = (mnew == m) ? 1.f : tc::ex2(m - mnew);
  float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
  for (int c = 0; c < 32; c += 2) {
    const float e0 = in(c) ? tc::ex2(fmaf(__uint_as_float(s0[c]), sl2, -mnew)) : 0.f;
    const float e1 = in(c + 1) ? tc::ex2(fmaf(__uint_as_float(s0[c + 1]), sl2, -mnew)) : 0.f;
    const float f0 = in(c + 32) ? tc::ex2(fmaf(__uint_as_float(s1[c]), sl2, -mnew)) : 0.f;
    const float f1 = in(c + 33) ? tc::ex2(fmaf(__uint_as_float(s1[c + 1]), sl2, -mnew)) : 0.f;
    ls0 += e0 + e1;
    ls1 += f0 + f1;
    pk[c / 2] = pack_bf16(e0, e1);
    pk[16 + c / 2] = pack_bf16(f0, f1);
  }
  l = l * alpha + (ls0 + ls1);
  m = mnew;
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
      float alpha;
      if (__all_sync(0xffffffffu, lo == 0 && hi == kKT - 1))
        softmax_row<false>(s0, s1, lo, hi, sl2, m, l, alpha, pk);
      else
        softmax_row<true>(s0, s1, lo, hi, sl2, m, l, alpha, pk);
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
    tc::mbar_init(&bar.q_full, 128);
    for (int i = 0; i < kRing; ++i) {
      tc::mbar_init(&bar.raw_full[i], 1);
      tc::mbar_init(&bar.kt_full[i], 128);
      tc::mbar_init(&bar.kt_empty[i], 1);
      tc::mbar_init(&bar.v_empty[i], 1);
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
    // rotation warps: stage the angle tables, sync among themselves, rotate
    const int tid_r = threadIdx.x - 320;
    float4 *t64 = reinterpret_cast<float4 *>(smem + kOffT64);
    for (int i = tid_r; i < 64 * 16; i += 128)
      t64[i] = __ldg(reinterpret_cast<const float4 *>(p.rel + (size_t)p.rel_off * (kD / 2)) + i);
    float4 *tb = reinterpret_cast<float4 *>(smem + kOffTB);
    for (int i = tid_r; i < (4 + tr.ntiles) * 16; i += 128) {
      const int row = i >> 4, part = i & 15;
      const int off = row < 4 ? 64 * row : tr.kt0 + (row - 4) * kKT - tr.q0[0];
      tb[i] = __ldg(reinterpret_cast<const float4 *>(p.rel + (size_t)(off + p.rel_off) * (kD / 2)) + part);
    }
    asm volatile("bar.sync 1, 128;\n" ::: "memory");
    role_rotate(tr, bar, smem, p, head, tid_r, p.err);
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
  const uint32_t smem = smem_bytes(w);
  cudaError_t e = cudaFuncSetAttribute(k5_window_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((sh.nblk() + 1) / 2, sh.BH());
  k5_window_tc_kernel<<<grid, kThreads, smem, st>>>(mk, mv, p);
  return cudaGetLastError();
}

}  // namespace fs
