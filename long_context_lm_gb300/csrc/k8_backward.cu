// k8_backward.cu -- gradients of the FS-L attention forward.
//
// FreeSolo (paper.rainbus.top summary, 方法步骤详情: training in two stages;
// "hard top-P / top-K indices carry no gradient"; 局限与改进: sigma_h and
// lambda_h fixed; ai.info summary, "Methodology in Plain English", training
// paragraph).  With the pools and selections held fixed, L = sum(g * out),
// out = o_win + m_h * RMSNorm(o_long):
//   window (rotated space, scale 1/8):  p = softmax(q~ . k~ / 8) over the band,
//     dv_j += p_j g,  ds_j = p_j (g . v_j - g . o_win) / 8,
//     dq~ += ds_j k~_j,  dk~_j += ds_j q~,  then dq = R(n)^T dq~, dk = R(j)^T dk~;
//   long (NoPE): o = sum p_t v_t over the selected tokens, rho = (mean(o^2) +
//     eps)^(-1/2), o^ = rho o;  dm_h += g . o^;  do = rho m_h g - rho^3 (o .
//     m_h g) o / d;  dv_t += p_t do,  ds_t = p_t (do . v_t - do . o) / 8,
//     dq += ds_t k_t,  dk_t += ds_t q.
// After the forward's own selection (cell summaries, pools, scores and top-K
// recomputed with the forward's kernels):
//   k8_split     rotated q~, k~ and g as bf16 hi | lo rows (tensor-core operands);
//   k8_win_q_tc  one CTA per 128-query tile, tcgen05: the window softmax
//                statistics (pass 1), then dS and dq~ (pass 2); writes dq
//                (rotated back), the row's log-sum-exp and g . o_win;
//   k8_win_kv_tc one CTA per 128-key tile, tcgen05: every query tile that
//                sees the tile, from the saved row statistics; writes dk
//                (rotated back) and dv;
//   k8_long_tc   one CTA per 128-query tile, tcgen05: the union of the
//                tile's selected cells in long tiles of four cells; each
//                row's softmax, RMSNorm and their backward give dq (added to
//                the window's), dm_h, and per long tile the dk, dv
//                contributions of the tile's rows, added into dk, dv.
#include "fs_common.cuh"
#include "fs_internal.h"
#include "tc05.cuh"

namespace fs {
namespace {

// ---------------------------------------------------------------------------
// window branch on the tensor cores (tcgen05, TMEM accumulators)
// ---------------------------------------------------------------------------
// Operands, prepared once per call by k8_split_kernel: for every row the
// rotated q~ and k~ and the upstream gradient g, each as bf16 hi | lo (256 B
// a row: hi = bf16(x), lo = bf16(x - hi)).  A product of two split operands
// is taken as hi.hi + hi.lo + lo.hi (three MMA chains accumulating in fp32):
// about 2^-16 relative error per product, where one bf16 chain gives 2^-8.
// v is exact in bf16 (one term).  P and dS are split the same way when they
// are written back to TMEM as the A operand of the second products.
//
// Both kernels take one 128-row tile per CTA with 8 warps: thread t and
// t + 128 own TMEM lane t = the tile's row t, and the tile's columns 0..63
// and 64..127 (two warps per SM sub-partition for the element-wise work).  Tiles sit in shared memory as 128-byte rows with the
// hardware's 128-byte swizzle; the same bytes serve as a K-major operand
// (contraction over d) and as an MN-major B operand (contraction over rows).
// TMEM: S (128 columns), dP (128), then the accumulators; P (dS) is written
// in place of S (dP): chunk c of 32 columns keeps its bf16 hi pairs in
// columns 32c..32c+15 and its lo pairs in 32c+16..32c+31.
constexpr int kT = 128;                    // rows of a tile (queries or keys)
constexpr uint32_t kTileB = kT * 128;      // one bf16 tile of 64 columns
constexpr uint32_t kColSt = 0, kColDp = 128, kColA0 = 256, kColA1 = 320;
constexpr uint32_t kBwdTmem = 512;
// shared memory: [hi | lo] of the CTA's own operand pair, v, then the
// streamed tiles and the per-row statistics of the streamed rows
constexpr uint32_t kOffA = 0;              // own q~ (or k~) hi, lo
constexpr uint32_t kOffB = 2 * kTileB;     // own g (q side) or v (key side)
constexpr uint32_t kOffC = 4 * kTileB;     // streamed k~ (q side) / q~ (key side) hi, lo
constexpr uint32_t kOffD = 6 * kTileB;     // streamed v (q side) / g hi, lo (key side)
constexpr uint32_t kOffStat = 8 * kTileB;  // lse2, gdo of the streamed queries
constexpr uint32_t kBwdSmem = kOffStat + 2 * kT * 4 + 1024;

__device__ __forceinline__ uint32_t p_chunk_col(int ks) {  // A operand, K step ks (16 rows)
  return 32 * (ks >> 1) + 8 * (ks & 1);
}

// 128 rows of `src` (row stride `ld` bytes, 128 bytes taken at byte `off`)
// into a swizzled tile, by 16-byte asynchronous copies of all 128 threads
__device__ __forceinline__ void load_tile(unsigned char *dst, const unsigned char *src,
                                          size_t ld, int off) {
  for (int e = threadIdx.x; e < kT * 8; e += blockDim.x) {
    const int r = e >> 3, ch = e & 7;
    cp_async16(dst + swz128(r, ch), src + (size_t)r * ld + off + 16 * ch);
  }
}

// hi/lo split of 32 fp32 values into packed bf16 pairs
__device__ __forceinline__ void split32(const float (&x)[32], uint32_t (&hi)[16],
                                        uint32_t (&lo)[16]) {
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    hi[e] = pack_bf16(x[2 * e], x[2 * e + 1]);
    lo[e] = pack_bf16(x[2 * e] - bf16_lo(hi[e]), x[2 * e + 1] - bf16_hi(hi[e]));
  }
}

// (hi, lo) A operand chunk of 32 columns written in place of what was read
__device__ __forceinline__ void store_split(uint32_t taddr, const float (&x)[32]) {
  uint32_t hi[16], lo[16];
  split32(x, hi, lo);
  tc::tmem_st16(taddr, hi);
  tc::tmem_st16(taddr + 16, lo);
}

// y = R(n)^T y~ for a whole row (pairs (i, i + 32))
__device__ __forceinline__ void rotate_back_row(float (&y)[64], int n, const float2 *tab) {
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float2 a = __ldg(tab + (size_t)(n & 63) * (kD / 2) + i);
    const float2 b = __ldg(tab + (size_t)(64 + (n >> 6)) * (kD / 2) + i);
    const float c = fmaf(b.x, a.x, -b.y * a.y), s = fmaf(b.y, a.x, b.x * a.y);
    const float y0 = y[i], y1 = y[i + 32];
    y[i] = fmaf(y0, c, y1 * s);
    y[i + 32] = fmaf(-y0, s, y1 * c);
  }
}

// Four threads per row: thread part p rotates pairs 8p .. 8p+7 of q and k
// (dims 8p.. and 32+8p..) and splits them and the same dims of g.
__global__ void __launch_bounds__(256) k8_split_kernel(const uint16_t *__restrict__ q,
                                                       const uint16_t *__restrict__ k,
                                                       const float *__restrict__ g,
                                                       const float2 *__restrict__ tab, int N,
                                                       size_t rows, uint4 *__restrict__ qs,
                                                       uint4 *__restrict__ ks,
                                                       uint4 *__restrict__ gs) {
  const size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= rows * 4) return;
  const size_t row = t >> 2;
  const int part = (int)(t & 3), n = (int)(row % N);
  float c[8], s[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float2 a = __ldg(tab + (size_t)(n & 63) * (kD / 2) + 8 * part + e);
    const float2 b = __ldg(tab + (size_t)(64 + (n >> 6)) * (kD / 2) + 8 * part + e);
    c[e] = fmaf(b.x, a.x, -b.y * a.y);
    s[e] = fmaf(b.y, a.x, b.x * a.y);
  }
  // 16-byte chunk j of a split row: hi dims 8j.. at chunk j, lo at chunk 8 + j
  auto emit = [&](uint4 *dst, const float (&x0)[8], const float (&x1)[8]) {
    uint32_t h0[4], l0[4], h1[4], l1[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      h0[e] = pack_bf16(x0[2 * e], x0[2 * e + 1]);
      l0[e] = pack_bf16(x0[2 * e] - bf16_lo(h0[e]), x0[2 * e + 1] - bf16_hi(h0[e]));
      h1[e] = pack_bf16(x1[2 * e], x1[2 * e + 1]);
      l1[e] = pack_bf16(x1[2 * e] - bf16_lo(h1[e]), x1[2 * e + 1] - bf16_hi(h1[e]));
    }
    uint4 *o = dst + row * 16;
    o[part] = make_uint4(h0[0], h0[1], h0[2], h0[3]);
    o[4 + part] = make_uint4(h1[0], h1[1], h1[2], h1[3]);
    o[8 + part] = make_uint4(l0[0], l0[1], l0[2], l0[3]);
    o[12 + part] = make_uint4(l1[0], l1[1], l1[2], l1[3]);
  };
  auto rotate = [&](const uint16_t *x, uint4 *dst) {
    const uint4 wa = __ldg(reinterpret_cast<const uint4 *>(x + row * kD) + part);
    const uint4 wb = __ldg(reinterpret_cast<const uint4 *>(x + row * kD + kD / 2) + part);
    const uint32_t a4[4] = {wa.x, wa.y, wa.z, wa.w}, b4[4] = {wb.x, wb.y, wb.z, wb.w};
    float y0[8], y1[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float x0 = (e & 1) ? bf16_hi(a4[e >> 1]) : bf16_lo(a4[e >> 1]);
      const float x1 = (e & 1) ? bf16_hi(b4[e >> 1]) : bf16_lo(b4[e >> 1]);
      y0[e] = fmaf(x0, c[e], -x1 * s[e]);
      y1[e] = fmaf(x0, s[e], x1 * c[e]);
    }
    emit(dst, y0, y1);
  };
  rotate(q, qs);
  rotate(k, ks);
  const float4 *gr = reinterpret_cast<const float4 *>(g + row * kD);
  float g0[8], g1[8];
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const float4 u = __ldg(gr + 2 * part + e), v = __ldg(gr + 8 + 2 * part + e);
    g0[4 * e] = u.x; g0[4 * e + 1] = u.y; g0[4 * e + 2] = u.z; g0[4 * e + 3] = u.w;
    g1[4 * e] = v.x; g1[4 * e + 1] = v.y; g1[4 * e + 2] = v.z; g1[4 * e + 3] = v.w;
  }
  emit(gs, g0, g1);
}

struct WinBwd {
  const unsigned char *qs, *ks, *gs;  // split rows, 256 B each
  const unsigned char *v;             // bf16 rows, 128 B each
  const float2 *tab;
  float *lse2, *gdo;  // per query row: log-sum-exp of s/8 in log2 units; g . o_win
  float *dq, *dk, *dv;
  int N, w;
  int *err;
};

// D (+)= A . B^T over d = 64 (four K steps of 32 bytes), A and B K-major
__device__ __forceinline__ void mma_d64(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                        bool acc) {
#pragma unroll
  for (int k = 0; k < kD / 16; ++k)
    tc::mma_ss(d, a + (uint64_t)(2 * k), b + (uint64_t)(2 * k), id, (acc || k > 0) ? 1u : 0u);
}
// D (+)= A . B over 128 rows: A in TMEM (one split half, packed pairs), B
// MN-major in shared memory (a K step of 16 rows is 2048 bytes)
__device__ __forceinline__ void mma_r128(uint32_t d, uint32_t a, uint64_t b, uint32_t id,
                                         bool acc) {
#pragma unroll 1
  for (int ks = 0; ks < kT / 16; ++ks)
    tc::mma_ts(d, a + p_chunk_col(ks), b + (uint64_t)(ks * 128), id, (acc || ks > 0) ? 1u : 0u);
}
// hi.hi + hi.lo + lo.hi of a split A in TMEM against a split B
__device__ __forceinline__ void mma_r128_split(uint32_t d, uint32_t a, uint64_t bh, uint64_t bl,
                                               uint32_t id, bool acc) {
  mma_r128(d, a, bh, id, acc);
  mma_r128(d, a, bl, id, true);
  mma_r128(d, a + 16, bh, id, true);
}

__device__ __forceinline__ void load_split(unsigned char *dst, const unsigned char *rows) {
  load_tile(dst, rows, 256, 0);
  load_tile(dst + kTileB, rows, 256, 128);
}

// The CTA's loads have landed and its TMEM reads are done; every thread
// learns whether every other one is still on track.
__device__ __forceinline__ bool cta_sync_ok(bool ok) {
  tc::tmem_wait_ld();
  tc::fence_async_smem();
  tc::fence_before_sync();
  ok = __syncthreads_and(ok) != 0;
  tc::fence_after_sync();
  return ok;
}

// Query side: one CTA per (head, 128-query tile).  Pass 1 over the window's
// key tiles: S = q~ k~^T and dP = g v^T, the row's online log-sum-exp and
// gdo = sum_j p_j dP_j (= g . o_win).  Pass 2: S and dP again, dS = P (dP -
// gdo) / 8, dq~ += dS k~.  Writes lse2 and gdo (for the key side) and dq.
__global__ void __launch_bounds__(2 * kT, 1) k8_win_q_tc_kernel(const WinBwd p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ uint32_t s_tmem;
  __shared__ float s_mla[3][kT];  // the second half's pass-0 partials
  __shared__ float s_st[2][kT];   // the merged row statistics
  // 8 warps: warps w and w + 4 share TMEM lanes 32 (w % 4).. (query rows) and
  // take each key tile's columns 0..63 and 64..127
  const int tid = threadIdx.x, warp = tid >> 5, row = tid & (kT - 1), half = tid >> 7;
  const int nblk = p.N / kT;
  const int bh = blockIdx.x / nblk, b0 = (blockIdx.x % nblk) * kT;
  const int n = b0 + row;
  const size_t head = (size_t)bh * p.N;
  const uint32_t sb = smem_u32(smem);
  if (warp == 0) {
    tc::tmem_alloc(&s_tmem, kBwdTmem);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(&bar[0], 1);
    tc::mbar_init(&bar[1], 1);
    tc::mbar_fence_init();
  }
  load_split(smem + kOffA, p.qs + (head + b0) * 256);
  load_split(smem + kOffB, p.gs + (head + b0) * 256);
  cp_async_commit();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem, lane_base = (uint32_t)((warp & 3) * 32) << 16;
  const uint32_t id_s = tc::idesc_bf16(kT, kT, 0), id_dq = tc::idesc_bf16(kT, kD, 1);
  const uint64_t dqh = tc::desc_sw128(sb + kOffA), dql = tc::desc_sw128(sb + kOffA + kTileB);
  const uint64_t dgh = tc::desc_sw128(sb + kOffB), dgl = tc::desc_sw128(sb + kOffB + kTileB);
  const uint64_t dkh = tc::desc_sw128(sb + kOffC), dkl = tc::desc_sw128(sb + kOffC + kTileB);
  const uint64_t dvv = tc::desc_sw128(sb + kOffD);
  const float sl2 = 1.4426950408889634f * 0.125f;
  const int kt0 = max(0, b0 - p.w + 1) / kT * kT;
  uint32_t ph0 = 0, ph1 = 0;
  bool ok = true;
  float m = -INFINITY, l = 0.f, a = 0.f, lse2 = 0.f, gdo = 0.f;
  for (int pass = 0; pass < 2; ++pass) {
    for (int j0 = kt0; j0 <= b0; j0 += kT) {
      // the previous tile's MMAs have completed (waited below): its operand
      // tiles and TMEM columns are free
      load_split(smem + kOffC, p.ks + (head + j0) * 256);
      load_tile(smem + kOffD, p.v + (head + j0) * 128, 128, 0);
      cp_async_commit();
      cp_async_wait<0>();
      ok = cta_sync_ok(ok);
      if (!ok) break;
      if (tid == 0) {
        mma_d64(tmem + kColSt, dqh, dkh, id_s, false);
        mma_d64(tmem + kColSt, dqh, dkl, id_s, true);
        mma_d64(tmem + kColSt, dql, dkh, id_s, true);
        mma_d64(tmem + kColDp, dgh, dvv, id_s, false);
        mma_d64(tmem + kColDp, dgl, dvv, id_s, true);
        tc::mma_commit(&bar[0]);
      }
      ok = tc::mbar_wait(&bar[0], ph0, p.err) && ok;
      ph0 ^= 1;
      tc::fence_after_sync();
#pragma unroll 1
      for (int c0 = 64 * half; c0 < 64 * half + 64; c0 += 32) {
        uint32_t xs[32], xd[32];
        tc::tmem_ld32(tmem + kColSt + c0 + lane_base, xs);
        tc::tmem_ld32(tmem + kColDp + c0 + lane_base, xd);
        tc::tmem_wait_ld();
        float x[32];
        if (pass == 0) {  // online: maximum, sum of 2^(s - m), sum of 2^(s - m) dP
          float cm = -INFINITY;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int j = j0 + c0 + e;
            const bool vis = j <= n && j >= n - p.w + 1;
            x[e] = vis ? __uint_as_float(xs[e]) * sl2 : -INFINITY;
            cm = fmaxf(cm, x[e]);
          }
          if (cm > m) {
            const float alpha = tc::ex2(m - cm);  // 0 while m is -inf
            l *= alpha;
            a *= alpha;
            m = cm;
          }
          if (m != -INFINITY) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const float pe = tc::ex2(x[e] - m);
              l += pe;
              a = fmaf(pe, __uint_as_float(xd[e]), a);
            }
          }
        } else {  // dS = P (dP - gdo) / 8, split in place of S
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int j = j0 + c0 + e;
            const bool vis = j <= n && j >= n - p.w + 1;
            const float pe = vis ? tc::ex2(fmaf(__uint_as_float(xs[e]), sl2, -lse2)) : 0.f;
            x[e] = pe * (__uint_as_float(xd[e]) - gdo) * 0.125f;
          }
          store_split(tmem + kColSt + c0 + lane_base, x);
        }
      }
      if (pass == 1) {
        tc::tmem_wait_st();
        ok = cta_sync_ok(ok);
        if (!ok) break;
        if (tid == 0) {
          mma_r128_split(tmem + kColA0, tmem + kColSt, dkh, dkl, id_dq, j0 != kt0);
          tc::mma_commit(&bar[1]);
        }
        ok = tc::mbar_wait(&bar[1], ph1, p.err) && ok;
        ph1 ^= 1;
        tc::fence_after_sync();
      }
    }
    ok = cta_sync_ok(ok);
    if (!ok) break;
    if (pass == 0) {  // merge the halves' partials (a half may have seen no key: m = -inf)
      if (half) {
        s_mla[0][row] = m;
        s_mla[1][row] = l;
        s_mla[2][row] = a;
      }
      __syncthreads();
      if (!half) {
        const float m1 = s_mla[0][row], mm = fmaxf(m, m1);
        const float f0 = tc::ex2(m - mm), f1 = tc::ex2(m1 - mm);
        const float lt = l * f0 + s_mla[1][row] * f1, at = a * f0 + s_mla[2][row] * f1;
        lse2 = mm + __log2f(lt);  // lt >= 1: the row sees itself
        gdo = at / lt;
        p.lse2[head + n] = lse2;
        p.gdo[head + n] = gdo;
        s_st[0][row] = lse2;
        s_st[1][row] = gdo;
      }
      __syncthreads();
      lse2 = s_st[0][row];
      gdo = s_st[1][row];
    }
  }
  ok = cta_sync_ok(ok);
  if (ok && !half) {  // warps 0-3 (warp-uniform)
    uint32_t r0[32], r1[32];
    tc::tmem_ld32(tmem + kColA0 + lane_base, r0);
    tc::tmem_ld32(tmem + kColA0 + 32 + lane_base, r1);
    tc::tmem_wait_ld();
    float y[64];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      y[e] = __uint_as_float(r0[e]);
      y[32 + e] = __uint_as_float(r1[e]);
    }
    rotate_back_row(y, n, p.tab);
    float4 *o = reinterpret_cast<float4 *>(p.dq + (head + n) * kD);
#pragma unroll
    for (int e = 0; e < 16; ++e) o[e] = make_float4(y[4 * e], y[4 * e + 1], y[4 * e + 2], y[4 * e + 3]);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kBwdTmem);
  }
}

// Key side: one CTA per (head, 128-key tile), over the query tiles whose
// windows reach it.  S^T = k~ q~^T and dP^T = v g^T, P^T and dS^T from the
// query side's row statistics, then dv += P^T g and dk~ += dS^T q~.
__global__ void __launch_bounds__(2 * kT, 1) k8_win_kv_tc_kernel(const WinBwd p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ uint32_t s_tmem;
  // 8 warps: warps w and w + 4 share TMEM lanes 32 (w % 4).. (key rows) and
  // take the tile's columns 0..63 and 64..127
  const int tid = threadIdx.x, warp = tid >> 5, row = tid & (kT - 1), half = tid >> 7;
  const int nblk = p.N / kT;
  const int bh = blockIdx.x / nblk, j0 = (blockIdx.x % nblk) * kT;
  const int j = j0 + row;
  const size_t head = (size_t)bh * p.N;
  const uint32_t sb = smem_u32(smem);
  float *s_lse2 = reinterpret_cast<float *>(smem + kOffStat);
  float *s_gdo = s_lse2 + kT;
  if (warp == 0) {
    tc::tmem_alloc(&s_tmem, kBwdTmem);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(&bar[0], 1);
    tc::mbar_init(&bar[1], 1);
    tc::mbar_fence_init();
  }
  load_split(smem + kOffA, p.ks + (head + j0) * 256);
  load_tile(smem + kOffB, p.v + (head + j0) * 128, 128, 0);
  cp_async_commit();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem, lane_base = (uint32_t)((warp & 3) * 32) << 16;
  const uint32_t id_s = tc::idesc_bf16(kT, kT, 0), id_kv = tc::idesc_bf16(kT, kD, 1);
  const uint64_t dkh = tc::desc_sw128(sb + kOffA), dkl = tc::desc_sw128(sb + kOffA + kTileB);
  const uint64_t dvv = tc::desc_sw128(sb + kOffB);
  const uint64_t dqh = tc::desc_sw128(sb + kOffC), dql = tc::desc_sw128(sb + kOffC + kTileB);
  const uint64_t dgh = tc::desc_sw128(sb + kOffD), dgl = tc::desc_sw128(sb + kOffD + kTileB);
  const float sl2 = 1.4426950408889634f * 0.125f;
  // queries that see a key of the tile: [j0, j0 + 127 + w - 1]
  const int nlast = min(p.N - kT, (j0 + kT - 1 + p.w - 1) / kT * kT);
  uint32_t ph0 = 0, ph1 = 0;
  bool ok = true;
  for (int n0 = j0; n0 <= nlast; n0 += kT) {
    load_split(smem + kOffC, p.qs + (head + n0) * 256);
    load_split(smem + kOffD, p.gs + (head + n0) * 256);
    if (half == 0) s_lse2[row] = p.lse2[head + n0 + row];
    else s_gdo[row] = p.gdo[head + n0 + row];
    cp_async_commit();
    cp_async_wait<0>();
    ok = cta_sync_ok(ok);
    if (!ok) break;
    if (tid == 0) {
      mma_d64(tmem + kColSt, dkh, dqh, id_s, false);
      mma_d64(tmem + kColSt, dkh, dql, id_s, true);
      mma_d64(tmem + kColSt, dkl, dqh, id_s, true);
      mma_d64(tmem + kColDp, dvv, dgh, id_s, false);
      mma_d64(tmem + kColDp, dvv, dgl, id_s, true);
      tc::mma_commit(&bar[0]);
    }
    ok = tc::mbar_wait(&bar[0], ph0, p.err) && ok;
    ph0 ^= 1;
    tc::fence_after_sync();
#pragma unroll 1
    for (int c0 = 64 * half; c0 < 64 * half + 64; c0 += 32) {
      uint32_t xs[32], xd[32];
      tc::tmem_ld32(tmem + kColSt + c0 + lane_base, xs);
      tc::tmem_ld32(tmem + kColDp + c0 + lane_base, xd);
      tc::tmem_wait_ld();
      float pe[32], ds[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int nn = n0 + c0 + e;
        const bool vis = nn >= j && nn <= j + p.w - 1;
        pe[e] = vis ? tc::ex2(fmaf(__uint_as_float(xs[e]), sl2, -s_lse2[c0 + e])) : 0.f;
        ds[e] = pe[e] * (__uint_as_float(xd[e]) - s_gdo[c0 + e]) * 0.125f;
      }
      store_split(tmem + kColSt + c0 + lane_base, pe);
      store_split(tmem + kColDp + c0 + lane_base, ds);
    }
    tc::tmem_wait_st();
    ok = cta_sync_ok(ok);
    if (!ok) break;
    if (tid == 0) {
      mma_r128_split(tmem + kColA0, tmem + kColSt, dgh, dgl, id_kv, n0 != j0);
      mma_r128_split(tmem + kColA1, tmem + kColDp, dqh, dql, id_kv, n0 != j0);
      tc::mma_commit(&bar[1]);
    }
    ok = tc::mbar_wait(&bar[1], ph1, p.err) && ok;
    ph1 ^= 1;
    tc::fence_after_sync();
  }
  ok = cta_sync_ok(ok);
  if (ok) {  // warps 0-3: dv; warps 4-7: dk~, rotated back
    uint32_t r0[32], r1[32];
    const uint32_t col = half ? kColA1 : kColA0;
    tc::tmem_ld32(tmem + col + lane_base, r0);
    tc::tmem_ld32(tmem + col + 32 + lane_base, r1);
    tc::tmem_wait_ld();
    float y[64];
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      y[e] = __uint_as_float(r0[e]);
      y[32 + e] = __uint_as_float(r1[e]);
    }
    if (half) rotate_back_row(y, j, p.tab);
    float4 *o = reinterpret_cast<float4 *>((half ? p.dk : p.dv) + (head + j) * kD);
#pragma unroll
    for (int e = 0; e < 16; ++e) o[e] = make_float4(y[4 * e], y[4 * e + 1], y[4 * e + 2], y[4 * e + 3]);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kBwdTmem);
  }
}

// ---------------------------------------------------------------------------
// long branch on the tensor cores
// ---------------------------------------------------------------------------
// One CTA per (head, 128-query tile), 8 warps: threads r and r + 128 own TMEM
// lane r = query row r (token r of the transposed tile) and a tile's columns
// 0..63 and 64..127; the rows' maxima and sums are merged across the halves.
// The union of the tile's selected cells (ascending) is cut into long tiles
// of four cells (128 tokens, raw bf16 k and v gathered into shared memory);
// a row reads only the cells it picked, the other columns of a tile are
// masked.  q and k are exact in bf16, so S = q k^T is one MMA chain; the
// forward's P, the gradient do and dS are split hi | lo like the window's.
//   pass A  S per tile: the row maximum;
//   pass B  S again, P = 2^(s/8 - m), l, o += P v: o, RMSNorm, dm_h, do, lse;
//   pass C  S and dP = do v^T: dS = P (dP - do.o) / 8, dq += dS k; then the
//           tile transposed (tokens in the lanes): S^T, dP^T, P^T, dS^T from
//           the rows' statistics, dv_t = P^T do and dk_t = dS^T q, added to
//           the cells' rows with fp32 atomics (other query tiles read the
//           same cells).
constexpr uint32_t kLOffQ = 0;                  // q tile (bf16)
constexpr uint32_t kLOffDo = kTileB;            // do hi, lo
constexpr uint32_t kLOffK = 3 * kTileB;         // gathered keys
constexpr uint32_t kLOffV = 4 * kTileB;         // gathered values
constexpr uint32_t kLOffStat = 5 * kTileB;      // lse2[128], dodo[128], rmask[128]
constexpr uint32_t kLOffUl = kLOffStat + 3 * kT * 4;  // union list (<= 128 K ids)
constexpr uint32_t kLOffBm = kLOffUl + kT * kMaxK * 4;  // bitmap words, then word ranks
constexpr uint32_t kColO = 256, kColDv = 320, kColDk = 384;

__host__ __device__ inline uint32_t long_bwd_smem(int N) {
  const uint32_t nwd = (uint32_t)((N / kS + 31) / 32);
  return kLOffBm + nwd * 4 + (nwd * 2 + 15) / 16 * 16 + 1024;
}

struct LongBwd {
  const unsigned char *q, *k, *v;  // bf16 rows, 128 B each
  const float *g;
  const int32_t *sel;
  const float *mix;
  float *dq, *dk, *dv, *dmix;
  int H, N, K;
  float rms_eps;
  int *err;
};

// 128 token rows of a long tile: row i is token i % 32 of union cell
// slot 4t + i / 32; rows past the union are zeros
__device__ __forceinline__ void load_cells(unsigned char *dst, const unsigned char *x,
                                           size_t head, const int *ul, int slot0, int nu) {
  for (int e = threadIdx.x; e < kT * 8; e += blockDim.x) {
    const int i = e >> 3, ch = e & 7, sl = slot0 + (i >> 5);
    unsigned char *d = dst + swz128(i, ch);
    if (sl < nu)
      cp_async16(d, x + (head + (size_t)ul[sl] * kS + (i & 31)) * 128 + 16 * ch);
    else
      *reinterpret_cast<uint4 *>(d) = make_uint4(0u, 0u, 0u, 0u);
  }
}

// D (+)= A(tmem, packed pairs; hi at +0, lo at +16 per chunk) . B over 128
// rows, the A halves given by `parts` (1: hi; 2: hi, lo)
__device__ __forceinline__ void mma_r128_parts(uint32_t d, uint32_t a, uint64_t b, uint32_t id,
                                               bool acc, int parts) {
  for (int part = 0; part < parts; ++part) mma_r128(d, a + 16u * part, b, id, acc || part > 0);
}

__global__ void __launch_bounds__(2 * kT, 1) k8_long_tc_kernel(const LongBwd p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ uint32_t s_tmem;
  __shared__ int s_nu;
  __shared__ float s_red[4];
  __shared__ float s_half[2][kT];  // the halves' partial row maxima, then row sums
  // 8 warps: warps w and w + 4 share TMEM lanes 32 (w % 4).. (rows, or tokens
  // in the transposed tile) and take columns 0..63 and 64..127 of a tile
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = tid & (kT - 1), half = tid >> 7;
  const int nblk = p.N / kT;
  const int bh = blockIdx.x / nblk, b0 = (blockIdx.x % nblk) * kT, h = bh % p.H;
  const int n = b0 + row;
  const size_t head = (size_t)bh * p.N;
  const int A = b0 / kS;  // cells available to the tile
  if (A == 0) return;     // the first block has no long branch: nothing to add
  const uint32_t sb = smem_u32(smem);
  float *s_lse2 = reinterpret_cast<float *>(smem + kLOffStat);
  float *s_dodo = s_lse2 + kT;
  int *s_rmask = reinterpret_cast<int *>(s_dodo + kT);
  int *ul = reinterpret_cast<int *>(smem + kLOffUl);
  const int nwd = (A + 31) / 32;
  uint32_t *bm = reinterpret_cast<uint32_t *>(smem + kLOffBm);
  uint16_t *pw = reinterpret_cast<uint16_t *>(bm + nwd);
  if (warp == 0) {
    tc::tmem_alloc(&s_tmem, kBwdTmem);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(&bar[0], 1);
    tc::mbar_init(&bar[1], 1);
    tc::mbar_fence_init();
  }
  load_tile(smem + kLOffQ, p.q + (head + b0) * 128, 128, 0);
  cp_async_commit();
  for (int w = tid; w < nwd; w += blockDim.x) bm[w] = 0u;
  __syncthreads();
  // union: mark, rank the words (warp 0), then each pick's slot
  int pick[kMaxK];
#pragma unroll
  for (int k = 0; k < kMaxK; ++k) {
    const int c = k < p.K ? p.sel[(head + n) * p.K + k] : -1;
    pick[k] = (c >= 0 && c < A) ? c : -1;
    if (!half && pick[k] >= 0) atomicOr(bm + (pick[k] >> 5), 1u << (pick[k] & 31));
  }
  __syncthreads();
  if (warp == 0) {
    int nu = 0;
    for (int w0 = 0; w0 < nwd; w0 += 32) {
      const int w = w0 + lane;
      uint32_t bits = w < nwd ? bm[w] : 0u;
      const int cnt = __popc(bits);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      int kk = nu + incl - cnt;
      if (w < nwd) pw[w] = (uint16_t)kk;
      while (bits) {
        ul[kk++] = 32 * w + (__ffs(bits) - 1);
        bits &= bits - 1;
      }
      nu += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_nu = nu;
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const int nu = s_nu, nt = (nu + 3) / 4;
  int slot[kMaxK];
#pragma unroll
  for (int k = 0; k < kMaxK; ++k) {
    const int c = pick[k];
    slot[k] = c < 0 ? -1 : pw[c >> 5] + __popc(bm[c >> 5] & ((1u << (c & 31)) - 1u));
  }
  const uint32_t tmem = s_tmem, lane_base = (uint32_t)((warp & 3) * 32) << 16;
  const uint32_t id_s = tc::idesc_bf16(kT, kT, 0), id_o = tc::idesc_bf16(kT, kD, 1);
  const uint64_t dq_ = tc::desc_sw128(sb + kLOffQ);
  const uint64_t ddh = tc::desc_sw128(sb + kLOffDo), ddl = tc::desc_sw128(sb + kLOffDo + kTileB);
  const uint64_t dk_ = tc::desc_sw128(sb + kLOffK), dv_ = tc::desc_sw128(sb + kLOffV);
  const float sl2 = 1.4426950408889634f * 0.125f;
  uint32_t ph0 = 0, ph1 = 0;
  bool ok = true;
  float m = -INFINITY, l = 0.f;
  // which of tile t's four cells this row reads (bit c)
  auto row_mask = [&](int t) {
    int mk = 0;
#pragma unroll
    for (int k = 0; k < kMaxK; ++k)
      if (slot[k] >= 4 * t && slot[k] < 4 * t + 4) mk |= 1 << (slot[k] - 4 * t);
    return mk;
  };
  // ---- pass A: row maxima
  for (int t = 0; t < nt; ++t) {
    load_cells(smem + kLOffK, p.k, head, ul, 4 * t, nu);
    cp_async_commit();
    cp_async_wait<0>();
    ok = cta_sync_ok(ok);
    if (!ok) break;
    if (tid == 0) {
      mma_d64(tmem + kColSt, dq_, dk_, id_s, false);
      tc::mma_commit(&bar[0]);
    }
    ok = tc::mbar_wait(&bar[0], ph0, p.err) && ok;
    ph0 ^= 1;
    tc::fence_after_sync();
    const int mk = row_mask(t);
#pragma unroll 1
    for (int ch = 2 * half; ch < 2 * half + 2; ++ch) {
      if (!__any_sync(0xffffffffu, (mk >> ch) & 1)) continue;  // warp-uniform
      uint32_t xs[32];
      tc::tmem_ld32(tmem + kColSt + 32 * ch + lane_base, xs);
      tc::tmem_wait_ld();
      if ((mk >> ch) & 1) {
        float cm = __uint_as_float(xs[0]);
#pragma unroll
        for (int e = 1; e < 32; ++e) cm = fmaxf(cm, __uint_as_float(xs[e]));
        m = fmaxf(m, cm * sl2);
      }
    }
  }
  // ---- pass B: P, l and o += P v
  s_half[half][row] = m;  // the row maximum over both halves
  ok = cta_sync_ok(ok);
  m = fmaxf(s_half[0][row], s_half[1][row]);
  for (int t = 0; t < nt; ++t) {
    load_cells(smem + kLOffK, p.k, head, ul, 4 * t, nu);
    load_cells(smem + kLOffV, p.v, head, ul, 4 * t, nu);
    cp_async_commit();
    cp_async_wait<0>();
    ok = cta_sync_ok(ok);
    if (!ok) break;
    if (tid == 0) {
      mma_d64(tmem + kColSt, dq_, dk_, id_s, false);
      tc::mma_commit(&bar[0]);
    }
    ok = tc::mbar_wait(&bar[0], ph0, p.err) && ok;
    ph0 ^= 1;
    tc::fence_after_sync();
    const int mk = row_mask(t);
#pragma unroll 1
    for (int ch = 2 * half; ch < 2 * half + 2; ++ch) {
      uint32_t xs[32];
      tc::tmem_ld32(tmem + kColSt + 32 * ch + lane_base, xs);
      tc::tmem_wait_ld();
      const bool vis = (mk >> ch) & 1;
      float x[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        x[e] = vis ? tc::ex2(fmaf(__uint_as_float(xs[e]), sl2, -m)) : 0.f;
        l += x[e];
      }
      store_split(tmem + kColSt + 32 * ch + lane_base, x);
    }
    tc::tmem_wait_st();
    ok = cta_sync_ok(ok);
    if (!ok) break;
    if (tid == 0) {
      mma_r128_parts(tmem + kColO, tmem + kColSt, dv_, id_o, t > 0, 2);
      tc::mma_commit(&bar[1]);
    }
    ok = tc::mbar_wait(&bar[1], ph1, p.err) && ok;
    ph1 ^= 1;
    tc::fence_after_sync();
  }
  s_half[half][row] = l;  // the row sum over both halves
  ok = cta_sync_ok(ok);
  l = s_half[0][row] + s_half[1][row];
  // ---- the row's RMSNorm, dm_h, do, lse (warps 0-3)
  const bool has = l > 0.f;
  float lse2 = 0.f, dodo = 0.f, dmx = 0.f;
  if (ok && !half) {
    float o[64];
    {
      uint32_t r0[32], r1[32];
      tc::tmem_ld32(tmem + kColO + lane_base, r0);
      tc::tmem_ld32(tmem + kColO + 32 + lane_base, r1);
      tc::tmem_wait_ld();
      const float il = has ? 1.f / l : 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        // (selects, not products: with no long tile the columns were never written)
        o[e] = has ? __uint_as_float(r0[e]) * il : 0.f;
        o[32 + e] = has ? __uint_as_float(r1[e]) * il : 0.f;
      }
    }
    const float mh = p.mix[h];
    const float4 *gr = reinterpret_cast<const float4 *>(p.g + (head + n) * kD);
    float ss = 0.f, og = 0.f;
#pragma unroll
    for (int e4 = 0; e4 < 16; ++e4) {
      const float4 g4 = __ldg(gr + e4);
      const float ge[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float oe = o[4 * e4 + u];
        ss = fmaf(oe, oe, ss);
        og = fmaf(oe, mh * ge[u], og);
        dmx = fmaf(ge[u], oe, dmx);
      }
    }
    const float rho = has ? rsqrtf(ss / kD + p.rms_eps) : 0.f;
    dmx *= rho;
    const float c3 = rho * rho * rho * og / kD;
    // do = rho m_h g - rho^3 (o . m_h g) o / d, written split into shared memory
    unsigned char *dh = smem + kLOffDo, *dl = smem + kLOffDo + kTileB;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      const float4 ga = __ldg(gr + 2 * ch), gb = __ldg(gr + 2 * ch + 1);
      const float ge[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
      float dv8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        dv8[u] = has ? rho * mh * ge[u] - c3 * o[8 * ch + u] : 0.f;
        dodo = fmaf(dv8[u], o[8 * ch + u], dodo);
      }
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        hi[u] = pack_bf16(dv8[2 * u], dv8[2 * u + 1]);
        lo[u] = pack_bf16(dv8[2 * u] - bf16_lo(hi[u]), dv8[2 * u + 1] - bf16_hi(hi[u]));
      }
      *reinterpret_cast<uint4 *>(dh + swz128(row, ch)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4 *>(dl + swz128(row, ch)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    lse2 = has ? m + __log2f(l) : 0.f;
  }
  if (!half) {
    s_lse2[row] = lse2;
    s_dodo[row] = dodo;
  }
  dmx = warp_sum(dmx);
  if (lane == 0 && !half) s_red[warp] = dmx;
  ok = cta_sync_ok(ok);
  lse2 = s_lse2[row];  // the row's statistics, for both halves
  dodo = s_dodo[row];
  if (tid == 0 && ok) atomicAdd(p.dmix + h, (s_red[0] + s_red[1]) + (s_red[2] + s_red[3]));
  // ---- pass C: dq from the rows' side, then dk, dv from the tokens' side
  for (int t = 0; t < nt; ++t) {
    load_cells(smem + kLOffK, p.k, head, ul, 4 * t, nu);
    load_cells(smem + kLOffV, p.v, head, ul, 4 * t, nu);
    cp_async_commit();
    cp_async_wait<0>();
    ok = cta_sync_ok(ok);  // also publishes do (generic stores) to the tensor core
    if (!ok) break;
    if (tid == 0) {
      mma_d64(tmem + kColSt, dq_, dk_, id_s, false);
      mma_d64(tmem + kColDp, ddh, dv_, id_s, false);
      mma_d64(tmem + kColDp, ddl, dv_, id_s, true);
      tc::mma_commit(&bar[0]);
    }
    ok = tc::mbar_wait(&bar[0], ph0, p.err) && ok;
    ph0 ^= 1;
    tc::fence_after_sync();
    const int mk = row_mask(t);
    s_rmask[row] = mk;
#pragma unroll 1
    for (int ch = 2 * half; ch < 2 * half + 2; ++ch) {
      uint32_t xs[32], xd[32];
      tc::tmem_ld32(tmem + kColSt + 32 * ch + lane_base, xs);
      tc::tmem_ld32(tmem + kColDp + 32 * ch + lane_base, xd);
      tc::tmem_wait_ld();
      const bool vis = (mk >> ch) & 1;
      float x[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const float pe = vis ? tc::ex2(fmaf(__uint_as_float(xs[e]), sl2, -lse2)) : 0.f;
        x[e] = pe * (__uint_as_float(xd[e]) - dodo) * 0.125f;
      }
      store_split(tmem + kColSt + 32 * ch + lane_base, x);
    }
    tc::tmem_wait_st();
    ok = cta_sync_ok(ok);
    if (!ok) break;
    if (tid == 0) {
      mma_r128_parts(tmem + kColO, tmem + kColSt, dk_, id_o, t > 0, 2);  // dq += dS k
      tc::mma_commit(&bar[1]);
    }
    ok = tc::mbar_wait(&bar[1], ph1, p.err) && ok;
    ph1 ^= 1;
    tc::fence_after_sync();
    if (tid == 0 && ok) {  // the tile transposed: S^T = k q^T, dP^T = v do^T
      mma_d64(tmem + kColSt, dk_, dq_, id_s, false);
      mma_d64(tmem + kColDp, dv_, ddh, id_s, false);
      mma_d64(tmem + kColDp, dv_, ddl, id_s, true);
      tc::mma_commit(&bar[0]);
    }
    ok = cta_sync_ok(ok);
    if (!ok) break;
    ok = tc::mbar_wait(&bar[0], ph0, p.err) && ok;
    ph0 ^= 1;
    tc::fence_after_sync();
    const int cell = row >> 5;  // this thread's token is token row % 32 of cell slot 4t + cell
#pragma unroll 1
    for (int ch = 2 * half; ch < 2 * half + 2; ++ch) {
      uint32_t xs[32], xd[32];
      tc::tmem_ld32(tmem + kColSt + 32 * ch + lane_base, xs);
      tc::tmem_ld32(tmem + kColDp + 32 * ch + lane_base, xd);
      tc::tmem_wait_ld();
      float pe[32], ds[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        const int r = 32 * ch + e;
        const bool vis = (s_rmask[r] >> cell) & 1;
        pe[e] = vis ? tc::ex2(fmaf(__uint_as_float(xs[e]), sl2, -s_lse2[r])) : 0.f;
        ds[e] = pe[e] * (__uint_as_float(xd[e]) - s_dodo[r]) * 0.125f;
      }
      store_split(tmem + kColSt + 32 * ch + lane_base, pe);
      store_split(tmem + kColDp + 32 * ch + lane_base, ds);
    }
    tc::tmem_wait_st();
    ok = cta_sync_ok(ok);
    if (!ok) break;
    if (tid == 0) {
      mma_r128_split(tmem + kColDv, tmem + kColSt, ddh, ddl, id_o, false);  // dv = P^T do
      mma_r128_parts(tmem + kColDk, tmem + kColDp, dq_, id_o, false, 2);   // dk = dS^T q
      tc::mma_commit(&bar[1]);
    }
    ok = tc::mbar_wait(&bar[1], ph1, p.err) && ok;
    ph1 ^= 1;
    ok = cta_sync_ok(ok);
    if (!ok) break;
    const int sl = 4 * t + cell;
    if (sl < nu) {  // warps 0-3: dv, warps 4-7: dk (sl is warp-uniform)
      const size_t trow = head + (size_t)ul[sl] * kS + (row & 31);
      uint32_t r0[32], r1[32];
      const uint32_t col = half ? kColDk : kColDv;
      float4 *d4 = reinterpret_cast<float4 *>((half ? p.dk : p.dv) + trow * kD);
      tc::tmem_ld32(tmem + col + lane_base, r0);
      tc::tmem_ld32(tmem + col + 32 + lane_base, r1);
      tc::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        atomicAdd(d4 + e, make_float4(__uint_as_float(r0[4 * e]), __uint_as_float(r0[4 * e + 1]),
                                      __uint_as_float(r0[4 * e + 2]), __uint_as_float(r0[4 * e + 3])));
        atomicAdd(d4 + 8 + e,
                  make_float4(__uint_as_float(r1[4 * e]), __uint_as_float(r1[4 * e + 1]),
                              __uint_as_float(r1[4 * e + 2]), __uint_as_float(r1[4 * e + 3])));
      }
    }
  }
  ok = cta_sync_ok(ok);
  if (ok && nt > 0 && !half) {  // dq of the long branch, added to the window's
    uint32_t r0[32], r1[32];
    tc::tmem_ld32(tmem + kColO + lane_base, r0);
    tc::tmem_ld32(tmem + kColO + 32 + lane_base, r1);
    tc::tmem_wait_ld();
    float4 *o = reinterpret_cast<float4 *>(p.dq + (head + n) * kD);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      float4 a = o[e], b = o[8 + e];
      a.x += __uint_as_float(r0[4 * e]); a.y += __uint_as_float(r0[4 * e + 1]);
      a.z += __uint_as_float(r0[4 * e + 2]); a.w += __uint_as_float(r0[4 * e + 3]);
      b.x += __uint_as_float(r1[4 * e]); b.y += __uint_as_float(r1[4 * e + 1]);
      b.z += __uint_as_float(r1[4 * e + 2]); b.w += __uint_as_float(r1[4 * e + 3]);
      o[e] = a;
      o[8 + e] = b;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kBwdTmem);
  }
}

}  // namespace

// angle table, split q~ / k~ / g rows (256 B each), window row statistics
size_t backward_workspace_bytes(const Shape &sh) {
  const size_t rows = (size_t)sh.BH() * sh.N;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  return up(rope_table_bytes(sh.N)) + 3 * up(rows * 256) + 2 * up(rows * 4);
}

cudaError_t launch_backward(const BwdArgs &a, cudaStream_t st) {
  const Shape &sh = a.sh;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = (size_t)sh.BH() * sh.N;
  unsigned char *ws = static_cast<unsigned char *>(a.ws);
  void *tab = ws;
  unsigned char *qs = ws + up(rope_table_bytes(sh.N));
  unsigned char *ks = qs + up(rows * 256);
  unsigned char *gs = ks + up(rows * 256);
  float *lse2 = reinterpret_cast<float *>(gs + up(rows * 256));
  float *gdo = lse2 + up(rows * 4) / 4;
  cudaError_t e = launch_rope_table(tab, sh.N, a.rope_base, st);
  if (e != cudaSuccess) return e;
  k8_split_kernel<<<(unsigned)((rows * 4 + 255) / 256), 256, 0, st>>>(
      static_cast<const uint16_t *>(a.q), static_cast<const uint16_t *>(a.k), a.g,
      static_cast<const float2 *>(tab), sh.N, rows, reinterpret_cast<uint4 *>(qs),
      reinterpret_cast<uint4 *>(ks), reinterpret_cast<uint4 *>(gs));
  if ((e = cudaMemsetAsync(a.dmix, 0, sizeof(float) * sh.H, st)) != cudaSuccess) return e;
  WinBwd w;
  w.qs = qs;
  w.ks = ks;
  w.gs = gs;
  w.v = static_cast<const unsigned char *>(a.v);
  w.tab = static_cast<const float2 *>(tab);
  w.lse2 = lse2;
  w.gdo = gdo;
  w.dq = a.dq;
  w.dk = a.dk;
  w.dv = a.dv;
  w.N = sh.N;
  w.w = a.w;
  w.err = a.err;
  const unsigned ntile = (unsigned)(sh.BH() * (sh.N / kT));
  for (auto kern : {k8_win_q_tc_kernel, k8_win_kv_tc_kernel})
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kBwdSmem)) != cudaSuccess)
      return e;
  k8_win_q_tc_kernel<<<ntile, 2 * kT, kBwdSmem, st>>>(w);
  k8_win_kv_tc_kernel<<<ntile, 2 * kT, kBwdSmem, st>>>(w);
  LongBwd lp;
  lp.q = static_cast<const unsigned char *>(a.q);
  lp.k = static_cast<const unsigned char *>(a.k);
  lp.v = static_cast<const unsigned char *>(a.v);
  lp.g = a.g;
  lp.sel = a.sel;
  lp.mix = a.mix;
  lp.dq = a.dq;
  lp.dk = a.dk;
  lp.dv = a.dv;
  lp.dmix = a.dmix;
  lp.H = sh.H;
  lp.N = sh.N;
  lp.K = a.K;
  lp.rms_eps = a.rms_eps;
  lp.err = a.err;
  const uint32_t lsm = long_bwd_smem(sh.N);
  if ((e = cudaFuncSetAttribute(k8_long_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)lsm)) != cudaSuccess)
    return e;
  k8_long_tc_kernel<<<ntile, 2 * kT, lsm, st>>>(lp);
  return cudaGetLastError();
}

}  // namespace fs
