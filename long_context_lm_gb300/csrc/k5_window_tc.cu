// k5_window_tc.cu -- sliding-window RoPE branch on the 5th-generation tensor
// cores (tcgen05 + TMEM), with the branch mix fused into the epilogue.
//
// FreeSolo (paper.rainbus.top summary, 方法步骤详情 ② "在 w=512 窗口内做 RoPE
// 注意力" and ⑥ "与局部分支相加"; 前置知识 RoPE; ai.info summary, "Methodology
// in Plain English"):
//     o_win[n] = softmax_j((R(n) q_n . R(j) k_j) / sqrt(d)) v_j,  j in [n-w+1, n]
//     out[n]   = o_win[n] + mix_h * o_long[n].
//
// One CTA (15 warps, one per SM) owns two adjacent 128-query tiles A and B of
// one head and walks the 128-key tiles that cover both windows:
//   warps 0-3   softmax of tile A (thread = query row = TMEM lane)
//   warps 4-7   softmax of tile B
//   warp  8     TMEM allocation; lane 0 issues every MMA of tile A
//   warp  9     lane 0 issues every MMA of tile B (one issuing thread caps at
//               roughly one tcgen05.mma per ~100 cycles, so the two query
//               tiles get their own issuer)
//   warp  10    TMA producer: key tile and value tile of each key tile
//   warps 11-14 rotate the queries once and every key tile once, in place
// RoPE is applied relative to tile A's first position b: q_n.k_j after
// rotations by n-b and j-b equals the absolute-position product (R is
// orthogonal and depends only on differences), so both query tiles share one
// rotated copy of each key tile and the angles stay small (|j-b| < w+256).
// An offset t = 64*u + r is rotated with cos/sin of t*theta_i formed by the
// angle-sum identity from two small shared tables (r*theta_i for r < 64 and
// the few tile bases 64*u*theta_i), both taken from an fp64-computed table.
// The rotated q and k are split into bf16 hi + lo halves; S = Q.K^T takes
// three tcgen05.mma chains (hi.hi + hi.lo + lo.hi) accumulating in TMEM, which
// keeps logits at ~2^-16 relative error (a single bf16 rounding of the
// rotated vectors exceeds the output tolerance on lognormal keys).  The
// softmax threads write P as bf16 back into TMEM; P.V reads A = P from TMEM
// and accumulates into a TMEM O that the softmax threads rescale when their
// running max grows.
#include <cuda.h>

#include "fs_common.cuh"
#include "fs_internal.h"
#include "tc05.cuh"

namespace fs {
namespace {

// Pipeline timeline probe (builds with -DFS_TRACE only): clock64() stamps of
// each role's hand-offs for one sampled CTA, event e of tile t at [e*64 + t].
#ifdef FS_TRACE
__device__ long long *g_trace = nullptr;
#define FS_TR(e, t)                                                              \
  do {                                                                           \
    if (g_trace && blockIdx.x == gridDim.x / 2 && blockIdx.y == 0 && (t) < 64)   \
      g_trace[(e) * 64 + (t)] = clock64();                                       \
  } while (0)
#else
#define FS_TR(e, t) \
  do {              \
  } while (0)
#endif

constexpr int kKT = 128;         // keys per tile
constexpr int kRing = 2;         // key / value ring depth (keys rotated in place)
constexpr int kThreads = 480;
constexpr int kT64Stride = 272;  // bytes per row of the r*theta table (padded: no bank conflicts)

// shared-memory layout, offsets from a 1024-byte aligned base
constexpr uint32_t kOffQ = 0;                           // [A hi, A lo, B hi, B lo] x 16 KB
constexpr uint32_t kOffK = 65536;                       // kRing x [hi 16 KB, lo 16 KB]
constexpr uint32_t kOffV = kOffK + kRing * 32768;       // kRing x 16 KB
constexpr uint32_t kOffT64 = kOffV + kRing * 16384;     // 64 rows x 272 B
constexpr uint32_t kOffTB = kOffT64 + 64 * kT64Stride;  // bases x 256 B

// TMEM columns of query tile x: S at 256x, P at 256x+128, O at 256x+192
constexpr uint32_t kTmemCols = 512;

struct Barriers {
  uint64_t q_full;
  uint64_t raw_full[kRing];  // TMA: key and value tile landed
  uint64_t kt_full[kRing];   // key tile rotated
  uint64_t k_empty[kRing];   // S MMAs of the tile done (both issuers commit)
  uint64_t v_empty[kRing];   // P.V MMAs of the tile done (both issuers commit)
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_done[2];
  uint64_t fin[2];
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
// (dims 16*half.. and 32+16*half..), angles from the shared tables t64r (row
// offset) and tbr (tile base), composed by the angle-sum identity.  The raw
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
  int kt0;       // first key of tile 0
  int ntiles;    // tiles walked by the CTA
  int begin[2];  // first tile of query tile A / B
  int end[2];    // one past the last tile of A / B (end <= begin: tile absent)
  int q0[2];     // first query of A / B
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

// Issuer of query tile x.  Walks every key tile so that the per-slot
// "empty" barriers (two arrivals: one per issuer) pair up tile by tile.
__device__ void role_issue(const TileRange &tr, Barriers &bar, int x, uint32_t tmem,
                           uint32_t base, int *err) {
  const uint32_t id_qk = tc::idesc_bf16(128, kKT, 0);
  const uint32_t id_pv = tc::idesc_bf16(128, kD, 1);
  const uint32_t s_col = tmem + 256 * x, p_col = s_col + 128, o_col = s_col + 192;
  const uint32_t qh = base + kOffQ + x * 32768, ql = qh + 16384;
  const uint64_t dqh = tc::desc_sw128(qh), dql = tc::desc_sw128(ql);
  if (!tc::mbar_wait(&bar.q_full, 0, err)) return;
  FS_TR(1 + x, 0);
  for (int t = 0; t <= tr.ntiles; ++t) {
    if (t < tr.ntiles && !tc::mbar_wait(&bar.kt_full[t % kRing], (t / kRing) & 1, err)) return;
    tc::fence_after_sync();
    if (t > 0) {
      if (uses(tr, x, t - 1)) {  // P.V of the previous key tile
        const int i = t - 1 - tr.begin[x];
        if (!tc::mbar_wait(&bar.p_full[x], i & 1, err)) return;
        tc::fence_after_sync();
        const uint64_t dv = tc::desc_sw128(base + kOffV + ((t - 1) % kRing) * 16384);
#pragma unroll
        for (int k = 0; k < kKT / 16; ++k)
          tc::mma_ts(o_col, p_col + 8 * k, dv + (uint64_t)(k * 128), id_pv,
                     (i > 0 || k > 0) ? 1u : 0u);
        FS_TR(10 + x, t - 1);
        if (t == tr.end[x]) tc::mma_commit(&bar.o_done[x]);
      }
      tc::mma_commit(&bar.v_empty[(t - 1) % kRing]);
    }
    if (t == tr.ntiles) break;
    if (uses(tr, x, t)) {  // S = Q.K^T, three split-precision chains
      const uint32_t kh = base + kOffK + (t % kRing) * 32768;
      const uint64_t dkh = tc::desc_sw128(kh), dkl = tc::desc_sw128(kh + 16384);
#pragma unroll
      for (int part = 0; part < 3; ++part) {
        const uint64_t a = part == 2 ? dql : dqh, b = part == 1 ? dkl : dkh;
#pragma unroll
        for (int k = 0; k < kD / 16; ++k)
          tc::mma_ss(s_col, a + (uint64_t)(2 * k), b + (uint64_t)(2 * k), id_qk,
                     (part > 0 || k > 0) ? 1u : 0u);
      }
      tc::mma_commit(&bar.s_full[x]);
      FS_TR(4 + x, t);
    }
    tc::mma_commit(&bar.k_empty[t % kRing]);
  }
}

__device__ void role_tma(const TileRange &tr, Barriers &bar, unsigned char *smem,
                         const CUtensorMap *tk, const CUtensorMap *tv, int row0, int *err) {
  for (int t = 0; t < tr.ntiles; ++t) {
    const int slot = t % kRing;
    if (t >= kRing) {
      const uint32_t ph = ((t / kRing) - 1) & 1;
      if (!tc::mbar_wait(&bar.k_empty[slot], ph, err)) return;
      if (!tc::mbar_wait(&bar.v_empty[slot], ph, err)) return;
    }
    tc::mbar_arrive_expect_tx(&bar.raw_full[slot], 2 * kKT * kD * 2);
    const int y = row0 + tr.kt0 + t * kKT;
    tc::tma_load_2d(smem + kOffK + slot * 32768, tk, &bar.raw_full[slot], 0, y);
    tc::tma_load_2d(smem + kOffV + slot * 16384, tv, &bar.raw_full[slot], 0, y);
    FS_TR(3, t);
  }
}

// Base rows of the angle tables: [0, 4) query bases 0, 64, 128, 192 relative
// to tile A; 4 + 2t + u: key-tile base kt0 + 128 t + 64 u - q0[A].
__device__ void role_rotate(const TileRange &tr, Barriers &bar, unsigned char *smem,
                            const Params &p, size_t head, int r, int *err) {
  const unsigned char *t64 = smem + kOffT64;
  const float2 *tb = reinterpret_cast<const float2 *>(smem + kOffTB);
  const float2 *t64r = reinterpret_cast<const float2 *>(t64 + (r & 63) * kT64Stride);
  for (int x = 0; x < 2; ++x) {
    if (tr.end[x] <= tr.begin[x]) continue;
    unsigned char *qh = smem + kOffQ + x * 32768;
    const uint4 *src = reinterpret_cast<const uint4 *>(p.q + (head + tr.q0[x] + r) * kD);
#pragma unroll
    for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(qh + swz128(r, c)) = __ldg(src + c);
    const float2 *tbr = tb + (2 * x + (r >> 6)) * (kD / 2);
    rotate_half_row(qh, qh + 16384, r, 0, t64r, tbr);
    rotate_half_row(qh, qh + 16384, r, 1, t64r, tbr);
  }
  tc::fence_async_smem();
  tc::mbar_arrive(&bar.q_full);
  for (int t = 0; t < tr.ntiles; ++t) {
    const int slot = t % kRing;
    if (!tc::mbar_wait(&bar.raw_full[slot], (t / kRing) & 1, err)) return;
    unsigned char *kh = smem + kOffK + slot * 32768;
    const float2 *tbr = tb + (4 + 2 * t + (r >> 6)) * (kD / 2);
    rotate_half_row(kh, kh + 16384, r, 0, t64r, tbr);
    rotate_half_row(kh, kh + 16384, r, 1, t64r, tbr);
    tc::fence_async_smem();
    tc::mbar_arrive(&bar.kt_full[slot]);
    if (r == 0) FS_TR(6, t);
  }
}

// Pass 1: row maximum of the (masked) score tile, 4 chunks of 32 columns.
template <bool kMask>
__device__ __forceinline__ float row_max(uint32_t s_addr, int lo, int hi) {
  float mx = -INFINITY;
#pragma unroll
  for (int ch = 0; ch < kKT / 32; ++ch) {
    uint32_t s[32];
    tc::tmem_ld32(s_addr + 32 * ch, s);
    tc::tmem_wait_ld();
#pragma unroll
    for (int c = 0; c < 32; ++c)
      if (!kMask || (32 * ch + c >= lo && 32 * ch + c <= hi)) mx = fmaxf(mx, __uint_as_float(s[c]));
  }
  return mx;
}

// Pass 2: probabilities 2^(s*sl2 - m) written as bf16 into the P columns;
// returns the row sum of the unrounded values.
template <bool kMask>
__device__ __forceinline__ float row_exp(uint32_t s_addr, uint32_t p_addr, int lo, int hi,
                                         float sl2, float m) {
  float ls = 0.f;
#pragma unroll
  for (int ch = 0; ch < kKT / 32; ++ch) {
    uint32_t s[32], pk[16];
    tc::tmem_ld32(s_addr + 32 * ch, s);
    tc::tmem_wait_ld();
    float l0 = 0.f, l1 = 0.f;
#pragma unroll
    for (int c = 0; c < 32; c += 2) {
      const int col = 32 * ch + c;
      const float e0 = (!kMask || (col >= lo && col <= hi))
                           ? tc::ex2(fmaf(__uint_as_float(s[c]), sl2, -m)) : 0.f;
      const float e1 = (!kMask || (col + 1 >= lo && col + 1 <= hi))
                           ? tc::ex2(fmaf(__uint_as_float(s[c + 1]), sl2, -m)) : 0.f;
      l0 += e0;
      l1 += e1;
      pk[c / 2] = pack_bf16(e0, e1);
    }
    ls += l0 + l1;
    tc::tmem_st16(p_addr + 16 * ch, pk);
  }
  return ls;
}

__device__ void role_softmax(const TileRange &tr, Barriers &bar, uint32_t tmem, const Params &p,
                             size_t head, int h, int x, int r, int *err) {
  const int warp = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  const uint32_t s_addr = tmem + 256 * x + lane_base, p_addr = s_addr + 128, o_addr = s_addr + 192;
  const int n = tr.q0[x] + r;
  const float sl2 = 1.4426950408889634f * 0.125f;  // log2(e) / sqrt(64)
  float m = -INFINITY, l = 0.f;
  for (int t = tr.begin[x]; t < tr.end[x]; ++t) {
    const int i = t - tr.begin[x];
    if (!tc::mbar_wait(&bar.s_full[x], i & 1, err)) return;
    tc::fence_after_sync();
    if (r == 0) FS_TR(7 + x, t);
    const int kt = tr.kt0 + t * kKT;
    const int lo = max(0, n - p.w + 1 - kt), hi = min(kKT - 1, n - kt);
    if (__any_sync(0xffffffffu, lo <= hi)) {
      const bool full = __all_sync(0xffffffffu, lo == 0 && hi == kKT - 1);
      const float mx = full ? row_max<false>(s_addr, lo, hi) : row_max<true>(s_addr, lo, hi);
      const float mnew = fmaxf(m, mx * sl2);
      const float alpha = (mnew == m) ? 1.f : tc::ex2(m - mnew);
      const float ls = full ? row_exp<false>(s_addr, p_addr, lo, hi, sl2, mnew)
                            : row_exp<true>(s_addr, p_addr, lo, hi, sl2, mnew);
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
      }
    } else {
      uint32_t z[16];
#pragma unroll
      for (int c = 0; c < 16; ++c) z[c] = 0u;
#pragma unroll
      for (int ch = 0; ch < kKT / 32; ++ch) tc::tmem_st16(p_addr + 16 * ch, z);
    }
    tc::tmem_wait_st();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&bar.p_full[x]);
    if (r == 0) FS_TR(12 + x, t);
  }
  // epilogue: O / l (+ mix_h * o_long)
  if (!tc::mbar_wait(&bar.o_done[x], 0, err)) return;
  if (r == 0) FS_TR(14 + x, 0);
  tc::fence_after_sync();
  uint32_t o0[32], o1[32];
  tc::tmem_ld32(o_addr, o0);
  tc::tmem_ld32(o_addr + 32, o1);
  tc::tmem_wait_ld();
  const float inv = 1.f / l;
  const float mh = p.mix ? p.mix[h] : 0.f;
  float4 *dst = reinterpret_cast<float4 *>(p.out + (head + n) * kD);
  const float4 *ol =
      p.o_long ? reinterpret_cast<const float4 *>(p.o_long + (head + n) * kD) : nullptr;
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
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Barriers bar;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = blockIdx.x, bh = blockIdx.y, h = bh % p.H;
  const size_t head = (size_t)bh * p.N;
  const TileRange tr = tile_range(pair, p.nblk, p.w);
  if (threadIdx.x == 0) FS_TR(0, 0);

  if (threadIdx.x == 0) {
    tc::mbar_init(&bar.q_full, 128);
    for (int i = 0; i < kRing; ++i) {
      tc::mbar_init(&bar.raw_full[i], 1);
      tc::mbar_init(&bar.kt_full[i], 128);
      tc::mbar_init(&bar.k_empty[i], 2);
      tc::mbar_init(&bar.v_empty[i], 2);
    }
    for (int x = 0; x < 2; ++x) {
      tc::mbar_init(&bar.s_full[x], 1);
      tc::mbar_init(&bar.p_full[x], 4);
      tc::mbar_init(&bar.o_done[x], 1);
      tc::mbar_init(&bar.fin[x], 1);
    }
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
    if (tr.end[x] > tr.begin[x]) role_softmax(tr, bar, tmem, p, head, h, x, threadIdx.x & 127, p.err);
  } else if (warp == 8 || warp == 9) {
    if (lane == 0) {
      const int x = warp - 8;
      role_issue(tr, bar, x, tmem, sbase, p.err);
      tc::mma_commit(&bar.fin[x]);  // every MMA this thread issued has completed
      tc::mbar_wait(&bar.fin[x], 0, p.err);
    }
  } else if (warp == 10) {
    if (lane == 0) role_tma(tr, bar, smem, &tmap_k, &tmap_v, (int)head, p.err);
  } else {
    // rotation warps: stage the angle tables, sync among themselves, rotate
    const int r = threadIdx.x - 352;
    const float4 *rel = reinterpret_cast<const float4 *>(p.rel);
    for (int i = r; i < 64 * 16; i += 128) {
      const int row = i >> 4, part = i & 15;
      *reinterpret_cast<float4 *>(smem + kOffT64 + row * kT64Stride + part * 16) =
          __ldg(rel + (size_t)(row + p.rel_off) * 16 + part);
    }
    float4 *tb = reinterpret_cast<float4 *>(smem + kOffTB);
    for (int i = r; i < (4 + 2 * tr.ntiles) * 16; i += 128) {
      const int row = i >> 4, part = i & 15;
      const int off = row < 4 ? 64 * row : tr.kt0 + (row - 4) * 64 - tr.q0[0];
      tb[i] = __ldg(rel + (size_t)(off + p.rel_off) * 16 + part);
    }
    asm volatile("bar.sync 1, 128;\n" ::: "memory");
    role_rotate(tr, bar, smem, p, head, r, p.err);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 8) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0) FS_TR(16, 0);
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

// [rows, 64] bf16 row-major, boxes of box_rows x 64 with the 128-byte swizzle.
bool make_rows_map(CUtensorMap *map, const void *ptr, size_t rows, int box_rows) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)kD, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kD, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// key tiles a CTA walks at most, and the dynamic shared memory it needs
constexpr int max_tiles(int w) { return (w + 126 + 256) / kKT + 1; }
constexpr uint32_t smem_bytes(int w) { return kOffTB + (4 + 2 * max_tiles(w)) * 256 + 1024; }

}  // namespace

// Relative-angle table rows: offsets t in [-rel_off, 2*kBq).
int window_rel_offset(int w) { return (w + 126 + 63) / 64 * 64; }
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
  if (!make_rows_map(&mk, k, nrows, kKT) || !make_rows_map(&mv, v, nrows, kKT))
    return cudaErrorInvalidValue;
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

#ifdef FS_TRACE
extern "C" int fs_trace_set(long long *buf) {
  return (int)cudaMemcpyToSymbol(fs::g_trace, &buf, sizeof(buf));
}
#endif
