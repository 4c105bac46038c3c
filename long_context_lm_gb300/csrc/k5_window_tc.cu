// k5_window_tc.cu -- sliding-window RoPE branch on the 5th-generation tensor
// cores (tcgen05 + TMEM), with the branch mix fused into the epilogue.
//
// FreeSolo (paper.rainbus.top summary, 方法步骤详情 ② "在 w=512 窗口内做 RoPE
// 注意力" and ⑥ "与局部分支相加"; 前置知识 RoPE; ai.info summary, "Methodology
// in Plain English"):
//     o_win[n] = softmax_j((R(n) q_n . R(j) k_j) / sqrt(d)) v_j,  j in [n-w+1, n]
//     out[n]   = o_win[n] + mix_h * o_long[n].
//
// Persistent kernel: one CTA per SM walks 128-query tiles (q-tiles), each over
// the 128-key tiles covering its window.  Sixteen warps (four per SM
// sub-partition, 128 registers each) with fixed roles and mbarrier hand-offs;
// every counter runs across q-tiles so the producers start the next q-tile
// while the softmax finishes the current one:
//   warps 0-7   softmax and epilogue: warp w owns TMEM lanes / query rows
//               32*(w%4).. and key columns 64*(w/4).. of each 128-key tile;
//               the two warps of a row block exchange their row maxima
//               through shared memory (one named barrier per tile)
//   warp  8     TMEM allocation; lane 0 issues the S = Q.K^T MMAs
//   warp  9     lane 0 issues the O += P.V MMAs (a single issuing thread
//               sustains roughly one tcgen05.mma per ~100 cycles, so the two
//               products get their own issuer)
//   warp  10    lane 0: TMA producer of the key and value tiles
//   warps 12-15 rotate the queries of each q-tile and every key tile, in place
// TMEM: S double-buffered (2 x 128 columns), P (64 columns of bf16 pairs,
// the A operand of P.V), O (64 columns).  With two S buffers the MMAs of key
// tile t+1 run while the softmax works on tile t.
// RoPE is applied relative to the q-tile's first position b: q_n.k_j after
// rotations by n-b and j-b equals the absolute-position product (R is
// orthogonal and depends only on differences), and the angles stay small.
// An offset o = 64*u + r is rotated with cos/sin of o*theta_i formed by the
// angle-sum identity from two small shared tables (r*theta_i, r < 64, and
// 64*u*theta_i), both taken from an fp64-computed table.
// The rotated q and k are split into bf16 hi + lo halves; S = Q.K^T takes
// three tcgen05.mma chains (hi.hi + hi.lo + lo.hi) accumulating in TMEM, which
// keeps logits at ~2^-16 relative error (a single bf16 rounding of the
// rotated vectors exceeds the output tolerance on lognormal keys).
#include <cuda.h>

#include "fs_common.cuh"
#include "fs_internal.h"
#include "tc05.cuh"

namespace fs {
namespace {

// Pipeline timeline probe (builds with -DFS_TRACE only): clock64() stamps of
// each role's hand-offs in CTA 0, event e of global tile t at [e*64 + t].
#ifdef FS_TRACE
__device__ long long *g_trace = nullptr;
#define FS_TR(e, t)                                                  \
  do {                                                               \
    if (g_trace && blockIdx.x == 0 && (t) < 64) g_trace[(e) * 64 + (t)] = clock64(); \
  } while (0)
#else
#define FS_TR(e, t) \
  do {              \
  } while (0)
#endif

constexpr int kKT = 128;         // keys per tile
constexpr int kRing = 3;         // key / value ring depth (keys rotated in place)
constexpr int kThreads = 512;
constexpr int kRotThreads = 128;  // rotation threads: one 64-element row each
constexpr int kRotBase = 384;     // first rotation thread
constexpr int kT64Stride = 272;  // bytes per row of the r*theta table (padded: no bank conflicts)

// shared-memory layout, offsets from a 1024-byte aligned base
constexpr uint32_t kOffQ = 0;                          // [hi 16 KB, lo 16 KB]
constexpr uint32_t kOffK = 32768;                      // kRing x [hi 16 KB, lo 16 KB]
constexpr uint32_t kOffV = kOffK + kRing * 32768;      // kRing x 16 KB
constexpr uint32_t kOffT64 = kOffV + kRing * 16384;    // 64 rows x 272 B
constexpr uint32_t kOffTU = kOffT64 + 64 * kT64Stride; // rows of 64*u*theta, 256 B each

// TMEM columns
constexpr uint32_t kColS = 0, kColP = 256, kColO = 320;
constexpr uint32_t kTmemCols = 512;

struct Barriers {
  uint64_t q_full, q_empty;
  uint64_t raw_full[kRing];  // TMA: key and value tile landed
  uint64_t kt_full[kRing];   // key tile rotated
  uint64_t k_empty[kRing];   // S MMAs of the tile done
  uint64_t v_empty[kRing];   // P.V MMAs of the tile done
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, pv_done;
  uint64_t o_done, o_free;
  uint64_t fin[2];
  uint32_t tmem;
  float xmax[2][128];  // per-half row maxima of the current tile
  float xsum[2][128];  // per-half row sums at the end of a q-tile
};

struct Params {
  const __nv_bfloat16 *q;
  const float *o_long;
  const float *mix;
  const float2 *rel;  // (cos, sin) of o*theta_i, row o + rel_off
  int rel_off;
  int umin;           // smallest u of the 64*u*theta table
  int H, N, w, nblk, nitems;
  float *out;
  int *err;
};

// wait for completion number `k` (0-based) of a barrier that completes once
// per use: parity k & 1
__device__ __forceinline__ bool wait_nth(uint64_t *bar, uint32_t k, int *err) {
  return tc::mbar_wait(bar, k & 1, err);
}

struct Item {
  int bh, b0, kt0, ntiles;
};
__device__ __forceinline__ Item item_of(const Params &p, int g) {
  Item it;
  it.bh = g / p.nblk;
  it.b0 = (g % p.nblk) * kBq;
  it.kt0 = max(0, it.b0 - p.w + 1) / kKT * kKT;
  it.ntiles = (it.b0 + kBq - it.kt0) / kKT;
  return it;
}

// Rotate half of one 64-element row in place: pairs i in [16*half, 16*half+16)
// (dims 16*half.. and 32+16*half..), angles composed from rows t64r (offset
// mod 64) and tur (64*u) by the angle-sum identity.  The raw row is read from
// `hi` (chunks 2*half, 2*half+1, 4+2*half, 5+2*half) and the rotated bf16
// hi / lo halves are written back to the same chunks of `hi` and `lo`.
__device__ __forceinline__ void rotate_half_row(unsigned char *hi, unsigned char *lo, int r,
                                                int half, const float2 *t64r,
                                                const float2 *tur) {
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
      const float4 bb = *reinterpret_cast<const float4 *>(tur + i0);
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

// Rotate row r (64 elements, in place) by the relative offset o.
__device__ __forceinline__ void rotate_row(unsigned char *hi, unsigned char *lo, int r, int o,
                                           const unsigned char *smem, int umin) {
  const float2 *t64r = reinterpret_cast<const float2 *>(smem + kOffT64 + (o & 63) * kT64Stride);
  const float2 *tur =
      reinterpret_cast<const float2 *>(smem + kOffTU) + ((o >> 6) - umin) * (kD / 2);
  rotate_half_row(hi, lo, r, 0, t64r, tur);
  rotate_half_row(hi, lo, r, 1, t64r, tur);
}

// --------------------------------------------------------------------------
// roles
// --------------------------------------------------------------------------

__device__ void role_qk(const Params &p, Barriers &bar, uint32_t tmem, uint32_t base) {
  const uint32_t id_qk = tc::idesc_bf16(128, kKT, 0);
  const uint64_t dqh = tc::desc_sw128(base + kOffQ), dql = tc::desc_sw128(base + kOffQ + 16384);
  uint32_t T = 0, u = 0, i = 0;
  for (int g = blockIdx.x; g < p.nitems; g += gridDim.x, ++i) {
    const Item it = item_of(p, g);
    if (!wait_nth(&bar.q_full, i, p.err)) return;
    for (int t = 0; t < it.ntiles; ++t, ++T, ++u) {
      const int slot = T % kRing, b = u & 1;
      if (!wait_nth(&bar.kt_full[slot], T / kRing, p.err)) return;
      if (u >= 2 && !wait_nth(&bar.s_free[b], u / 2 - 1, p.err)) return;
      tc::fence_after_sync();
      const uint32_t kh = base + kOffK + slot * 32768;
      const uint64_t dkh = tc::desc_sw128(kh), dkl = tc::desc_sw128(kh + 16384);
      const uint32_t s_col = tmem + kColS + 128 * b;
#pragma unroll
      for (int part = 0; part < 3; ++part) {
        const uint64_t a = part == 2 ? dql : dqh, bd = part == 1 ? dkl : dkh;
#pragma unroll
        for (int k = 0; k < kD / 16; ++k)
          tc::mma_ss(s_col, a + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), id_qk,
                     (part > 0 || k > 0) ? 1u : 0u);
      }
      tc::mma_commit(&bar.s_full[b]);
      tc::mma_commit(&bar.k_empty[slot]);
      FS_TR(2, T);
    }
    tc::mma_commit(&bar.q_empty);
  }
}

__device__ void role_pv(const Params &p, Barriers &bar, uint32_t tmem, uint32_t base) {
  const uint32_t id_pv = tc::idesc_bf16(128, kD, 1);
  uint32_t T = 0, i = 0;
  for (int g = blockIdx.x; g < p.nitems; g += gridDim.x, ++i) {
    const Item it = item_of(p, g);
    for (int t = 0; t < it.ntiles; ++t, ++T) {
      const int slot = T % kRing;
      if (!wait_nth(&bar.p_full, T, p.err)) return;
      if (t == 0 && i > 0 && !wait_nth(&bar.o_free, i - 1, p.err)) return;
      tc::fence_after_sync();
      const uint64_t dv = tc::desc_sw128(base + kOffV + slot * 16384);
#pragma unroll
      for (int k = 0; k < kKT / 16; ++k)
        tc::mma_ts(tmem + kColO, tmem + kColP + 8 * k, dv + (uint64_t)(k * 128), id_pv,
                   (t > 0 || k > 0) ? 1u : 0u);
      tc::mma_commit(&bar.pv_done);
      tc::mma_commit(&bar.v_empty[slot]);
      if (t == it.ntiles - 1) tc::mma_commit(&bar.o_done);
      FS_TR(5, T);
    }
  }
}

__device__ void role_tma(const Params &p, Barriers &bar, unsigned char *smem,
                         const CUtensorMap *tk, const CUtensorMap *tv) {
  uint32_t T = 0;
  for (int g = blockIdx.x; g < p.nitems; g += gridDim.x) {
    const Item it = item_of(p, g);
    for (int t = 0; t < it.ntiles; ++t, ++T) {
      const int slot = T % kRing;
      if (T >= kRing) {
        if (!wait_nth(&bar.k_empty[slot], T / kRing - 1, p.err)) return;
        if (!wait_nth(&bar.v_empty[slot], T / kRing - 1, p.err)) return;
      }
      tc::mbar_arrive_expect_tx(&bar.raw_full[slot], 2 * kKT * kD * 2);
      const int y = it.bh * p.N + it.kt0 + t * kKT;
      tc::tma_load_2d(smem + kOffK + slot * 32768, tk, &bar.raw_full[slot], 0, y);
      tc::tma_load_2d(smem + kOffV + slot * 16384, tv, &bar.raw_full[slot], 0, y);
      FS_TR(0, T);
    }
  }
}

__device__ void role_rotate(const Params &p, Barriers &bar, unsigned char *smem, int r) {
  uint32_t T = 0, i = 0;
  for (int g = blockIdx.x; g < p.nitems; g += gridDim.x, ++i) {
    const Item it = item_of(p, g);
    // query row r: fetch the raw row first, then wait until the previous
    // q-tile's S MMAs no longer read the query tile
    const uint4 *src = reinterpret_cast<const uint4 *>(p.q + ((size_t)it.bh * p.N + it.b0 + r) * kD);
    uint4 raw[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) raw[c] = __ldg(src + c);
    if (i > 0 && !wait_nth(&bar.q_empty, i - 1, p.err)) return;
    unsigned char *qh = smem + kOffQ;
#pragma unroll
    for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(qh + swz128(r, c)) = raw[c];
    rotate_row(qh, qh + 16384, r, r, smem, p.umin);
    tc::fence_async_smem();
    tc::mbar_arrive(&bar.q_full);
    for (int t = 0; t < it.ntiles; ++t, ++T) {
      const int slot = T % kRing;
      if (!wait_nth(&bar.raw_full[slot], T / kRing, p.err)) return;
      unsigned char *kh = smem + kOffK + slot * 32768;
      rotate_row(kh, kh + 16384, r, it.kt0 + t * kKT + r - it.b0, smem, p.umin);
      tc::fence_async_smem();
      tc::mbar_arrive(&bar.kt_full[slot]);
      if (r == 0) FS_TR(1, T);
    }
  }
}

// Half of a score row (64 columns) held in registers.  Columns outside
// [lo, hi] (the row's window, in tile columns) are set to -inf; the decision
// is made per 32-column chunk and is uniform across the warp except in the
// chunk a triangular edge crosses.
struct Half64 {
  uint32_t s[2][32];
};

__device__ __forceinline__ void load_half(uint32_t s_addr, Half64 &x) {
  tc::tmem_ld32(s_addr, x.s[0]);
  tc::tmem_ld32(s_addr + 32, x.s[1]);
  tc::tmem_wait_ld();
}

__device__ __forceinline__ void mask_half(Half64 &x, int lo, int hi, int col0) {
  constexpr uint32_t kNegInf = 0xff800000u;
#pragma unroll
  for (int ch = 0; ch < 2; ++ch) {
    const int c0 = col0 + 32 * ch;
    const bool full = lo <= c0 && hi >= c0 + 31;
    const bool empty = hi < c0 || lo > c0 + 31;
    if (__all_sync(0xffffffffu, full)) continue;
    if (__all_sync(0xffffffffu, empty)) {
#pragma unroll
      for (int c = 0; c < 32; ++c) x.s[ch][c] = kNegInf;
      continue;
    }
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const int col = c0 + c;
      if (col < lo || col > hi) x.s[ch][c] = kNegInf;
    }
  }
}

__device__ __forceinline__ float max_half(const Half64 &x) {
  float mx[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) mx[j] = __uint_as_float(x.s[j >> 2][(j & 3) * 8]);
#pragma unroll
  for (int ch = 0; ch < 2; ++ch)
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const int j = (ch * 4 + (c >> 3)) & 7;
      mx[j] = fmaxf(mx[j], __uint_as_float(x.s[ch][c]));
    }
  return fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
}

// 2^(s*sl2 - m) for the half row, written as bf16 pairs into its 32 P
// columns; returns the sum of the unrounded values (8 partial sums).
__device__ __forceinline__ float exp_half(const Half64 &x, uint32_t p_addr, float sl2, float m) {
  float part[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) part[j] = 0.f;
#pragma unroll
  for (int ch = 0; ch < 2; ++ch) {
    uint32_t pk[16];
#pragma unroll
    for (int c = 0; c < 32; c += 2) {
      const float e0 = tc::ex2(fmaf(__uint_as_float(x.s[ch][c]), sl2, -m));
      const float e1 = tc::ex2(fmaf(__uint_as_float(x.s[ch][c + 1]), sl2, -m));
      part[(c >> 2) & 7] += e0 + e1;
      pk[c / 2] = pack_bf16(e0, e1);
    }
    tc::tmem_st16(p_addr + 16 * ch, pk);
  }
  return ((part[0] + part[1]) + (part[2] + part[3])) + ((part[4] + part[5]) + (part[6] + part[7]));
}

// named barrier of the two softmax warps that share a row block
__device__ __forceinline__ void pair_sync(int quarter) {
  asm volatile("bar.sync %0, 64;\n" ::"r"(1 + quarter) : "memory");
}

__device__ void role_softmax(const Params &p, Barriers &bar, uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int r = quarter * 32 + lane;  // query row of this thread
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
  const uint32_t p_addr = tmem + kColP + 32 * half + lane_base;
  const uint32_t o_addr = tmem + kColO + 32 * half + lane_base;
  const float sl2 = 1.4426950408889634f * 0.125f;  // log2(e) / sqrt(64)
  uint32_t T = 0, i = 0;
  for (int g = blockIdx.x; g < p.nitems; g += gridDim.x, ++i) {
    const Item it = item_of(p, g);
    const int n = it.b0 + r;
    float m = -INFINITY, l = 0.f;
    for (int t = 0; t < it.ntiles; ++t, ++T) {
      const int b = T & 1;
      const uint32_t s_addr = tmem + kColS + 128 * b + 64 * half + lane_base;
      if (!wait_nth(&bar.s_full[b], T / 2, p.err)) return;
      tc::fence_after_sync();
      if (r == 0 && half == 0) FS_TR(3, T);
      const int kt = it.kt0 + t * kKT;
      const int lo = max(0, n - p.w + 1 - kt), hi = min(kKT - 1, n - kt);
      const bool any = __any_sync(0xffffffffu, lo <= hi && hi >= 64 * half && lo <= 64 * half + 63);
      Half64 x;
      float mx = -INFINITY;
      if (any) {
        load_half(s_addr, x);
        mask_half(x, lo, hi, 64 * half);
        mx = max_half(x);
      }
      // the S buffer may be refilled once both halves are in registers
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar.s_free[b]);
      bar.xmax[half][r] = mx;
      pair_sync(quarter);
      mx = fmaxf(mx, bar.xmax[half ^ 1][r]);
      pair_sync(quarter);  // the slot is rewritten next tile
      const float mnew = fmaxf(m, mx * sl2);
      const float alpha = (mnew == m) ? 1.f : tc::ex2(m - mnew);
      // P and O belong to the previous P.V until it completes
      if (T > 0 && !wait_nth(&bar.pv_done, T - 1, p.err)) return;
      tc::fence_after_sync();
      if (any) {
        const float muse = mnew == -INFINITY ? 0.f : mnew;
        l = l * alpha + exp_half(x, p_addr, sl2, muse);
      } else {
        l = l * alpha;
        uint32_t z[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) z[c] = 0u;
        tc::tmem_st16(p_addr, z);
        tc::tmem_st16(p_addr + 16, z);
      }
      m = mnew;
      if (t > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        uint32_t o[32];
        tc::tmem_ld32(o_addr, o);
        tc::tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
        tc::tmem_st32(o_addr, o);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bar.p_full);
      if (r == 0 && half == 0) FS_TR(4, T);
    }
    // epilogue: O / l (+ mix_h * o_long); each warp writes its 32 columns
    bar.xsum[half][r] = l;
    if (!wait_nth(&bar.o_done, i, p.err)) return;
    tc::fence_after_sync();
    uint32_t o[32];
    tc::tmem_ld32(o_addr, o);
    tc::tmem_wait_ld();
    tc::fence_before_sync();
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&bar.o_free);
    pair_sync(quarter);
    const float inv = 1.f / (l + bar.xsum[half ^ 1][r]);
    pair_sync(quarter);
    const size_t row = (size_t)it.bh * p.N + n;
    const float mh = p.mix ? p.mix[it.bh % p.H] : 0.f;
    float4 *dst = reinterpret_cast<float4 *>(p.out + row * kD + 32 * half);
    const float4 *ol =
        p.o_long ? reinterpret_cast<const float4 *>(p.o_long + row * kD + 32 * half) : nullptr;
#pragma unroll
    for (int c4 = 0; c4 < 8; ++c4) {
      float4 v = make_float4(__uint_as_float(o[4 * c4]) * inv, __uint_as_float(o[4 * c4 + 1]) * inv,
                             __uint_as_float(o[4 * c4 + 2]) * inv, __uint_as_float(o[4 * c4 + 3]) * inv);
      if (ol) {
        const float4 u4 = __ldg(ol + c4);
        v.x = fmaf(mh, u4.x, v.x);
        v.y = fmaf(mh, u4.y, v.y);
        v.z = fmaf(mh, u4.z, v.z);
        v.w = fmaf(mh, u4.w, v.w);
      }
      dst[c4] = v;
    }
    if (r == 0 && half == 0) FS_TR(6, i);
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

  if (threadIdx.x == 0) {
    tc::mbar_init(&bar.q_full, kRotThreads);
    tc::mbar_init(&bar.q_empty, 1);
    for (int i = 0; i < kRing; ++i) {
      tc::mbar_init(&bar.raw_full[i], 1);
      tc::mbar_init(&bar.kt_full[i], kRotThreads);
      tc::mbar_init(&bar.k_empty[i], 1);
      tc::mbar_init(&bar.v_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bar.s_full[b], 1);
      tc::mbar_init(&bar.s_free[b], 8);
      tc::mbar_init(&bar.fin[b], 1);
    }
    tc::mbar_init(&bar.p_full, 8);
    tc::mbar_init(&bar.pv_done, 1);
    tc::mbar_init(&bar.o_done, 1);
    tc::mbar_init(&bar.o_free, 8);
    tc::mbar_fence_init();
  }
  if (warp == 8) {
    tc::tmem_alloc(&bar.tmem, kTmemCols);
    tc::tmem_relinquish();
  }
  // angle tables, staged once per CTA by the rotation warps
  if (threadIdx.x >= kRotBase) {
    const int r = threadIdx.x - kRotBase;
    const float4 *rel = reinterpret_cast<const float4 *>(p.rel);
    for (int i = r; i < 64 * 16; i += kRotThreads) {
      const int row = i >> 4, part = i & 15;
      *reinterpret_cast<float4 *>(smem + kOffT64 + row * kT64Stride + part * 16) =
          __ldg(rel + (size_t)(row + p.rel_off) * 16 + part);
    }
    float4 *tu = reinterpret_cast<float4 *>(smem + kOffTU);
    const int nu = 3 - p.umin;  // u in [umin, 2]
    for (int i = r; i < nu * 16; i += kRotThreads) {
      const int row = i >> 4, part = i & 15;
      tu[i] = __ldg(rel + (size_t)(64 * (row + p.umin) + p.rel_off) * 16 + part);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bar.tmem;
  const uint32_t sbase = smem_u32(smem);

  if (warp < 8) {
    role_softmax(p, bar, tmem);
  } else if (warp == 8 || warp == 9) {
    if (lane == 0) {
      if (warp == 8)
        role_qk(p, bar, tmem, sbase);
      else
        role_pv(p, bar, tmem, sbase);
      tc::mma_commit(&bar.fin[warp - 8]);  // every MMA this thread issued has completed
      tc::mbar_wait(&bar.fin[warp - 8], 0, p.err);
    }
  } else if (warp == 10) {
    if (lane == 0) role_tma(p, bar, smem, &tmap_k, &tmap_v);
  } else if (threadIdx.x >= kRotBase) {
    role_rotate(p, bar, smem, threadIdx.x - kRotBase);
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

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

}  // namespace

// Relative-angle table rows: offsets o in [-rel_off, kBq + 64); the kernel
// needs o*theta for o = 64*u (u >= umin) and o in [0, 64).
int window_rel_offset(int w) { return (w + 127 + 63) / 64 * 64; }
size_t window_table_bytes(int w) {
  return (size_t)(window_rel_offset(w) + kBq + 64) * (kD / 2) * sizeof(float2);
}

cudaError_t launch_window_tc(const void *q, const void *k, const void *v, const float *o_long,
                             const float *mix, void *table, const Shape &sh, int w, float base,
                             float *out, int *err, cudaStream_t st) {
  const int off = window_rel_offset(w);
  const int rows = off + kBq + 64;
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
  p.umin = -(off / 64);
  p.H = sh.H;
  p.N = sh.N;
  p.w = w;
  p.nblk = sh.nblk();
  p.nitems = sh.BH() * sh.nblk();
  p.out = out;
  p.err = err;
  const uint32_t smem = kOffTU + (3 - p.umin) * 256 + 1024;
  cudaError_t e = cudaFuncSetAttribute(k5_window_tc_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = p.nitems < sm_count() ? p.nitems : sm_count();
  k5_window_tc_kernel<<<grid, kThreads, smem, st>>>(mk, mv, p);
  return cudaGetLastError();
}

}  // namespace fs

#ifdef FS_TRACE
extern "C" int fs_trace_set(long long *buf) {
  return (int)cudaMemcpyToSymbol(fs::g_trace, &buf, sizeof(buf));
}
#endif
