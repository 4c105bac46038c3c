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
//   k8_long      one CTA per 128-query tile (CUDA cores, fp32): the union of
//                the tile's selected cells is staged cell by cell; each row's
//                softmax, RMSNorm and their backward give dq (added), dm_h,
//                and per cell the dk, dv contributions of the tile's rows,
//                added into dk, dv.
#include "fs_common.cuh"
#include "fs_internal.h"
#include "tc05.cuh"

namespace fs {
namespace {

constexpr int kQT = 128;  // query tile
constexpr float kScale = 0.125f;  // 1 / sqrt(64)
// shared-memory rows of 64 floats keep dims 32..63 four words further (column
// c at c + 4 * (c / 32)): the two threads of a row read the same element
// index of their halves at the same time, which then sit in different banks,
// and both halves stay 16-byte aligned for vector loads
constexpr int kRow = kD + 4;
constexpr int kH1 = 36;  // first column of the second half
__device__ __forceinline__ int col(int c) { return c + 4 * (c >> 5); }

// dot of 32 register values with 32 consecutive shared floats (16-byte
// aligned), four independent partial sums
__device__ __forceinline__ float dot32(const float (&a)[32], const float *s) {
  float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    const float4 b = *reinterpret_cast<const float4 *>(s + e);
    p0 = fmaf(a[e], b.x, p0);
    p1 = fmaf(a[e + 1], b.y, p1);
    p2 = fmaf(a[e + 2], b.z, p2);
    p3 = fmaf(a[e + 3], b.w, p3);
  }
  return (p0 + p1) + (p2 + p3);
}
// acc += f * s[0..32)
__device__ __forceinline__ void axpy32(float (&acc)[32], float f, const float *s) {
#pragma unroll
  for (int e = 0; e < 32; e += 4) {
    const float4 b = *reinterpret_cast<const float4 *>(s + e);
    acc[e] = fmaf(f, b.x, acc[e]);
    acc[e + 1] = fmaf(f, b.y, acc[e + 1]);
    acc[e + 2] = fmaf(f, b.z, acc[e + 2]);
    acc[e + 3] = fmaf(f, b.w, acc[e + 3]);
  }
}

__device__ __forceinline__ float bf(uint16_t x) { return __uint_as_float((uint32_t)x << 16); }

struct BwdParams {
  const uint16_t *q, *k, *v;       // [BH, N, 64] bf16
  const float *g;                  // upstream gradient [BH, N, 64]
  const int32_t *sel;              // [BH, N, K]
  const float *mix;
  float *dq, *dk, *dv, *dmix;      // outputs
  int H, N, K;
  float rms_eps;
};

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
// Both kernels take one 128-row tile per CTA, 4 warps, thread t = TMEM lane
// t = the tile's row t.  Tiles sit in shared memory as 128-byte rows with the
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
  for (int e = threadIdx.x; e < kT * 8; e += kT) {
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
__global__ void __launch_bounds__(kT, 1) k8_win_q_tc_kernel(const WinBwd p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ uint32_t s_tmem;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int nblk = p.N / kT;
  const int bh = blockIdx.x / nblk, b0 = (blockIdx.x % nblk) * kT;
  const int n = b0 + tid;
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
  const uint32_t tmem = s_tmem, lane_base = (uint32_t)(warp * 32) << 16;
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
      for (int c0 = 0; c0 < kT; c0 += 32) {
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
    if (pass == 0) {
      lse2 = m + __log2f(l);  // l >= 1: the row sees itself
      gdo = a / l;
      p.lse2[head + n] = lse2;
      p.gdo[head + n] = gdo;
    }
  }
  ok = cta_sync_ok(ok);
  if (ok) {
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
__global__ void __launch_bounds__(kT, 1) k8_win_kv_tc_kernel(const WinBwd p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t bar[2];
  __shared__ uint32_t s_tmem;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int nblk = p.N / kT;
  const int bh = blockIdx.x / nblk, j0 = (blockIdx.x % nblk) * kT;
  const int j = j0 + tid;
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
  const uint32_t tmem = s_tmem, lane_base = (uint32_t)(warp * 32) << 16;
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
    s_lse2[tid] = p.lse2[head + n0 + tid];
    s_gdo[tid] = p.gdo[head + n0 + tid];
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
    for (int c0 = 0; c0 < kT; c0 += 32) {
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
  if (ok) {
    uint32_t r0[32], r1[32];
    float y[64];
    tc::tmem_ld32(tmem + kColA0 + lane_base, r0);  // dv
    tc::tmem_ld32(tmem + kColA0 + 32 + lane_base, r1);
    tc::tmem_wait_ld();
    float4 *o = reinterpret_cast<float4 *>(p.dv + (head + j) * kD);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      o[e] = make_float4(__uint_as_float(r0[4 * e]), __uint_as_float(r0[4 * e + 1]),
                         __uint_as_float(r0[4 * e + 2]), __uint_as_float(r0[4 * e + 3]));
      o[8 + e] = make_float4(__uint_as_float(r1[4 * e]), __uint_as_float(r1[4 * e + 1]),
                             __uint_as_float(r1[4 * e + 2]), __uint_as_float(r1[4 * e + 3]));
    }
    tc::tmem_ld32(tmem + kColA1 + lane_base, r0);  // dk~
    tc::tmem_ld32(tmem + kColA1 + 32 + lane_base, r1);
    tc::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      y[e] = __uint_as_float(r0[e]);
      y[32 + e] = __uint_as_float(r1[e]);
    }
    rotate_back_row(y, j, p.tab);
    o = reinterpret_cast<float4 *>(p.dk + (head + j) * kD);
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
// long branch
// ---------------------------------------------------------------------------
constexpr int kMaxU = kBq * kMaxK;

__global__ void __launch_bounds__(256) k8_long_kernel(const BwdParams p) {
  __shared__ __align__(16) float s_k[kS][kRow];
  __shared__ __align__(16) float s_v[kS][kRow];
  __shared__ int s_ul[kMaxU];
  __shared__ int s_nu;
  __shared__ float s_red[8];
  __shared__ int s_pick[kQT][kMaxK];  // the tile's rows' selected cells
  extern __shared__ float dyn[];  // per row: q (64), do (64), lse, do.o
  const int tid = threadIdx.x, half = tid & 1, r = tid >> 1;
  const int nblk = p.N / kQT;
  const int bh = blockIdx.x / nblk, b0 = (blockIdx.x % nblk) * kQT, h = bh % p.H;
  const int n = b0 + r;
  const size_t row = (size_t)bh * p.N + n;
  const int A = b0 / kS;
  // union of the tile's selected cells, ascending (repeated minimum, warp 0)
  if (tid < 32) {
    int cnt = 0, last = -1;
    while (true) {
      int mn = 0x7fffffff;
      for (int e = tid; e < kQT * p.K; e += 32) {
        const int c = p.sel[((size_t)bh * p.N + b0) * p.K + e];
        if (c >= 0 && c < A && c > last) mn = min(mn, c);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
      if (mn == 0x7fffffff) break;
      if (tid == 0) s_ul[cnt] = mn;
      ++cnt;
      last = mn;
    }
    if (tid == 0) s_nu = cnt;
  }
  for (int e = tid; e < kQT * kMaxK; e += 256) {
    const int rr = e / kMaxK, k = e % kMaxK;
    s_pick[rr][k] = k < p.K ? p.sel[((size_t)bh * p.N + b0 + rr) * p.K + k] : -1;
  }
  __syncthreads();
  const int nu = s_nu;
  int pick[kMaxK];
#pragma unroll
  for (int k = 0; k < kMaxK; ++k) pick[k] = k < p.K ? p.sel[row * p.K + k] : -1;
  float qh[32], acc[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    qh[e] = bf(p.q[row * kD + 32 * half + e]) * kScale;
    acc[e] = 0.f;
  }
  float m = -INFINITY, l = 0.f;
  // pass 1: softmax over the row's selected tokens (union order) and o
  for (int u = 0; u < nu; ++u) {
    const int c = s_ul[u];
    __syncthreads();
    for (int e = tid; e < kS * kD; e += 256) {
      const size_t src = ((size_t)bh * p.N + (size_t)c * kS + e / kD) * kD + e % kD;
      s_k[e / kD][col(e % kD)] = bf(p.k[src]);
      s_v[e / kD][col(e % kD)] = bf(p.v[src]);
    }
    __syncthreads();
    bool mine = false;
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) mine |= pick[k] == c;
    if (!mine) continue;  // both threads of the row agree
    for (int t = 0; t < kS; ++t) {
      const float part = dot32(qh, &s_k[t][kH1 * half]);
      const float sc = part + __shfl_xor_sync(0x3u << (tid & 30), part, 1);
      if (sc > m) {
        const float f = __expf(m - sc);
        l *= f;
#pragma unroll
        for (int e = 0; e < 32; ++e) acc[e] *= f;
        m = sc;
      }
      const float pe = __expf(sc - m);
      l += pe;
      axpy32(acc, pe, &s_v[t][kH1 * half]);
    }
  }
  const bool has = l > 0.f;
  // RMSNorm, mix weight, and do
  float gh[32], doh[32];
  float ss = 0.f, og = 0.f, dmx = 0.f;
  const float mh = p.mix[h];
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    acc[e] = has ? acc[e] / l : 0.f;
    gh[e] = p.g[row * kD + 32 * half + e];
    ss = fmaf(acc[e], acc[e], ss);
    og = fmaf(acc[e], mh * gh[e], og);
  }
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  og += __shfl_xor_sync(0xffffffffu, og, 1);
  const float rho = has ? rsqrtf(ss / kD + p.rms_eps) : 0.f;
  float dodo = 0.f;
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    dmx = fmaf(gh[e], acc[e] * rho, dmx);
    doh[e] = rho * mh * gh[e] - rho * rho * rho * og * acc[e] / kD;
    dodo = fmaf(doh[e], acc[e], dodo);
  }
  dodo += __shfl_xor_sync(0xffffffffu, dodo, 1);
  const float lse = m + __logf(l);
  // dm_h: the tile's sum, one atomic per CTA
  const float dmx2 = dmx + __shfl_xor_sync(0xffffffffu, dmx, 1);
  const float bs = warp_sum(half == 0 ? dmx2 : 0.f);
  if ((tid & 31) == 0) s_red[tid >> 5] = bs;
  // per-row values the scatter pass reads
  float *rq = dyn + (size_t)r * (2 * kD + 2);
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    rq[32 * half + e] = qh[e];
    rq[kD + 32 * half + e] = has ? doh[e] : 0.f;
  }
  if (half == 0) {
    rq[2 * kD] = lse;
    rq[2 * kD + 1] = dodo;
  }
  __syncthreads();
  if (tid == 0) {
    float t = 0.f;
    for (int i = 0; i < 8; ++i) t += s_red[i];
    atomicAdd(p.dmix + h, t);
  }
  // pass 2: dq from the selected tokens
#pragma unroll
  for (int e = 0; e < 32; ++e) acc[e] = 0.f;
  for (int u = 0; u < nu; ++u) {
    const int c = s_ul[u];
    __syncthreads();
    for (int e = tid; e < kS * kD; e += 256) {
      const size_t src = ((size_t)bh * p.N + (size_t)c * kS + e / kD) * kD + e % kD;
      s_k[e / kD][col(e % kD)] = bf(p.k[src]);
      s_v[e / kD][col(e % kD)] = bf(p.v[src]);
    }
    __syncthreads();
    bool mine = false;
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) mine |= pick[k] == c;
    if (mine) {
      for (int t = 0; t < kS; ++t) {
        const float ps = dot32(qh, &s_k[t][kH1 * half]);
        const float pd = dot32(doh, &s_v[t][kH1 * half]);
        const float sc = ps + __shfl_xor_sync(0x3u << (tid & 30), ps, 1);
        const float dp = pd + __shfl_xor_sync(0x3u << (tid & 30), pd, 1);
        const float ds = __expf(sc - lse) * (dp - dodo) * kScale;
        axpy32(acc, ds, &s_k[t][kH1 * half]);
      }
    }
    // scatter: dk, dv of cell c from the tile's rows that picked it; thread
    // (token t = tid / 8, dims 8*(tid % 8) ..) sums over those rows
    const int t = tid >> 3, d0 = 8 * (tid & 7);
    float kt[8], vt[8], dk8[8], dv8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      kt[e] = s_k[t][col(d0 + e)];
      vt[e] = s_v[t][col(d0 + e)];
      dk8[e] = 0.f;
      dv8[e] = 0.f;
    }
    for (int rr = 0; rr < kQT; ++rr) {
      bool picked = false;
#pragma unroll
      for (int k = 0; k < kMaxK; ++k) picked |= s_pick[rr][k] == c;
      if (!picked) continue;  // the same for every thread
      const float *rq2 = dyn + (size_t)rr * (2 * kD + 2);
      float ps = 0.f, pd = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        ps = fmaf(rq2[d0 + e], kt[e], ps);
        pd = fmaf(rq2[kD + d0 + e], vt[e], pd);
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        ps += __shfl_xor_sync(0xffffffffu, ps, o);
        pd += __shfl_xor_sync(0xffffffffu, pd, o);
      }
      const float pr = __expf(ps - rq2[2 * kD]);
      const float ds = pr * (pd - rq2[2 * kD + 1]);  // the 1/8 is in the stored q
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        dv8[e] = fmaf(pr, rq2[kD + d0 + e], dv8[e]);
        dk8[e] = fmaf(ds, rq2[d0 + e], dk8[e]);
      }
    }
    const size_t trow = (size_t)bh * p.N + (size_t)c * kS + t;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      atomicAdd(p.dk + trow * kD + d0 + e, dk8[e]);
      atomicAdd(p.dv + trow * kD + d0 + e, dv8[e]);
    }
  }
  // dq of the long branch added to the window's (scale 1/8 applied here: the
  // stored q was prescaled, k was not)
#pragma unroll
  for (int e = 0; e < 32; ++e) p.dq[row * kD + 32 * half + e] += acc[e];
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
  k8_win_q_tc_kernel<<<ntile, kT, kBwdSmem, st>>>(w);
  k8_win_kv_tc_kernel<<<ntile, kT, kBwdSmem, st>>>(w);
  BwdParams p;
  p.q = static_cast<const uint16_t *>(a.q);
  p.k = static_cast<const uint16_t *>(a.k);
  p.v = static_cast<const uint16_t *>(a.v);
  p.g = a.g;
  p.sel = a.sel;
  p.mix = a.mix;
  p.dq = a.dq;
  p.dk = a.dk;
  p.dv = a.dv;
  p.dmix = a.dmix;
  p.H = sh.H;
  p.N = sh.N;
  p.K = a.K;
  p.rms_eps = a.rms_eps;
  const unsigned nq = (unsigned)(sh.BH() * (sh.N / kQT));
  const int dyn = kQT * (2 * kD + 2) * 4;
  if ((e = cudaFuncSetAttribute(k8_long_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                dyn)) != cudaSuccess)
    return e;
  k8_long_kernel<<<nq, 256, dyn, st>>>(p);
  return cudaGetLastError();
}

}  // namespace fs
