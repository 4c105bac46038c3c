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
// Three kernels after the forward's own selection (cell summaries, pools,
// scores and top-K recomputed with the forward's kernels):
//   k8_win_q    one CTA per 128-query tile, two threads per row (32 dims
//               each): the window softmax again (online), then dq~; writes dq
//               (rotated back), the row's log-sum-exp and g . o_win;
//   k8_win_kv   one CTA per 64-key tile, two threads per key: every query
//               that sees the tile, from the saved row statistics; writes dk
//               (rotated back) and dv;
//   k8_long     one CTA per 128-query tile: the union of the tile's selected
//               cells is staged cell by cell; each row's softmax, RMSNorm and
//               their backward give dq (added), dm_h, and per cell the dk, dv
//               contributions of the tile's rows, added into dk, dv.
// fp32 arithmetic throughout (CUDA cores); rotated q and k in fp32 from the
// angle table.
#include "fs_common.cuh"
#include "fs_internal.h"
#include "tc05.cuh"

namespace fs {
namespace {

constexpr int kQT = 128;  // query tile
constexpr int kKT = 64;   // key tile
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

// x~ = R(n) x in fp32 for rows of bf16 x: one thread per (row, pair i), the
// angle n*theta_i composed from table rows n mod 64 and 64 * (n / 64)
__global__ void k8_rotate_kernel(const uint16_t *__restrict__ x, const float2 *__restrict__ tab,
                                 int N, size_t rows, float *__restrict__ xr) {
  const size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= rows * (kD / 2)) return;
  const size_t row = idx / (kD / 2);
  const int i = (int)(idx % (kD / 2));
  const int n = (int)(row % N);
  const float2 a = __ldg(tab + (size_t)(n & 63) * (kD / 2) + i);
  const float2 b = __ldg(tab + (size_t)(64 + (n >> 6)) * (kD / 2) + i);
  const float c = fmaf(b.x, a.x, -b.y * a.y), s = fmaf(b.y, a.x, b.x * a.y);
  const float x0 = __uint_as_float((uint32_t)x[row * kD + i] << 16);
  const float x1 = __uint_as_float((uint32_t)x[row * kD + i + kD / 2] << 16);
  xr[row * kD + i] = fmaf(x0, c, -x1 * s);
  xr[row * kD + i + kD / 2] = fmaf(x0, s, x1 * c);
}

// y = R(n)^T y~ for one thread's half of a row (pairs h*16 .. h*16+15 of dims
// (i, i + 32)): the two halves hold dims [32h, 32h+32); a pair (i, i+32) spans
// both, so the partner's values come by a shuffle.
__device__ __forceinline__ void rotate_back_pair(float (&y)[32], int n, int half,
                                                 const float2 *tab) {
  // thread half 0 holds dims 0..31 (first of each pair), half 1 dims 32..63
  float other[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) other[e] = __shfl_xor_sync(0xffffffffu, y[e], 1);
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const float2 a = __ldg(tab + (size_t)(n & 63) * (kD / 2) + e);
    const float2 b = __ldg(tab + (size_t)(64 + (n >> 6)) * (kD / 2) + e);
    const float c = fmaf(b.x, a.x, -b.y * a.y), s = fmaf(b.y, a.x, b.x * a.y);
    const float y0 = half ? other[e] : y[e], y1 = half ? y[e] : other[e];
    // transpose of [[c, -s], [s, c]]
    y[e] = half ? fmaf(-y0, s, y1 * c) : fmaf(y0, c, y1 * s);
  }
}

__device__ __forceinline__ float bf(uint16_t x) { return __uint_as_float((uint32_t)x << 16); }

struct BwdParams {
  const uint16_t *q, *k, *v;       // [BH, N, 64] bf16
  const float *qr, *kr;            // rotated q, k fp32 [BH, N, 64]
  const float *g;                  // upstream gradient [BH, N, 64]
  const float2 *tab;
  const int32_t *sel;              // [BH, N, K]
  const float *mix;
  float *dq, *dk, *dv, *dmix;      // outputs
  float *lse, *gdo;                // window row statistics [BH, N]
  int H, N, w, K;
  float rms_eps;
};

// ---------------------------------------------------------------------------
// window, query side
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k8_win_q_kernel(const BwdParams p) {
  __shared__ __align__(16) float s_k[kKT][kRow];
  __shared__ __align__(16) float s_v[kKT][kRow];
  const int tid = threadIdx.x, half = tid & 1, r = tid >> 1;
  const int nblk = p.N / kQT;
  const int bh = blockIdx.x / nblk, b0 = (blockIdx.x % nblk) * kQT;
  const int n = b0 + r;
  const size_t row = (size_t)bh * p.N + n;
  float qh[32], acc[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) qh[e] = p.qr[row * kD + 32 * half + e] * kScale;
  const int lo = max(0, n - p.w + 1);
  const int kt0 = max(0, b0 - p.w + 1) / kKT * kKT, kt1 = b0 + kQT;  // key range of the tile
  float m = -INFINITY, l = 0.f;
#pragma unroll
  for (int e = 0; e < 32; ++e) acc[e] = 0.f;
  // pass 1: online softmax and o_win
  for (int j0 = kt0; j0 < kt1; j0 += kKT) {
    __syncthreads();
    for (int e = tid; e < kKT * kD; e += 256) {
      const int jj = e / kD, dd = e % kD;
      const size_t src = ((size_t)bh * p.N + j0 + jj) * kD + dd;
      s_k[jj][col(dd)] = p.kr[src];
      s_v[jj][col(dd)] = bf(p.v[src]);
    }
    __syncthreads();
    const int ja = max(lo, j0) - j0, jb = min(n, j0 + kKT - 1) - j0;
    for (int jj = 0; jj <= 63; ++jj) {
      const float part = dot32(qh, &s_k[jj][kH1 * half]);
      const float sc = part + __shfl_xor_sync(0xffffffffu, part, 1);
      if (jj < ja || jj > jb) continue;
      if (sc > m) {
        const float f = __expf(m - sc);
        l *= f;
#pragma unroll
        for (int e = 0; e < 32; ++e) acc[e] *= f;
        m = sc;
      }
      const float pe = __expf(sc - m);
      l += pe;
      axpy32(acc, pe, &s_v[jj][kH1 * half]);
    }
  }
  float gh[32];
  float gdo = 0.f;
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    gh[e] = p.g[row * kD + 32 * half + e];
    gdo = fmaf(gh[e], acc[e] / l, gdo);
  }
  gdo += __shfl_xor_sync(0xffffffffu, gdo, 1);
  if (half == 0) {
    p.lse[row] = m + __logf(l);
    p.gdo[row] = gdo;
  }
  // pass 2: ds and dq~
  const float lse = m + __logf(l);
#pragma unroll
  for (int e = 0; e < 32; ++e) acc[e] = 0.f;
  for (int j0 = kt0; j0 < kt1; j0 += kKT) {
    __syncthreads();
    for (int e = tid; e < kKT * kD; e += 256) {
      const int jj = e / kD, dd = e % kD;
      const size_t src = ((size_t)bh * p.N + j0 + jj) * kD + dd;
      s_k[jj][col(dd)] = p.kr[src];
      s_v[jj][col(dd)] = bf(p.v[src]);
    }
    __syncthreads();
    const int ja = max(lo, j0) - j0, jb = min(n, j0 + kKT - 1) - j0;
    for (int jj = 0; jj <= 63; ++jj) {
      const float ps = dot32(qh, &s_k[jj][kH1 * half]);
      const float pd = dot32(gh, &s_v[jj][kH1 * half]);
      const float sc = ps + __shfl_xor_sync(0xffffffffu, ps, 1);
      const float dp = pd + __shfl_xor_sync(0xffffffffu, pd, 1);
      if (jj < ja || jj > jb) continue;
      const float pr = __expf(sc - lse);
      const float ds = pr * (dp - gdo) * kScale;
      axpy32(acc, ds, &s_k[jj][kH1 * half]);
    }
  }
  rotate_back_pair(acc, n, half, p.tab);
#pragma unroll
  for (int e = 0; e < 32; ++e) p.dq[row * kD + 32 * half + e] = acc[e];
}

// ---------------------------------------------------------------------------
// window, key side
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128) k8_win_kv_kernel(const BwdParams p) {
  __shared__ __align__(16) float s_q[kKT][kRow];  // rotated q / 8
  __shared__ __align__(16) float s_g[kKT][kRow];
  __shared__ float s_lse[kKT], s_gdo[kKT];
  const int tid = threadIdx.x, half = tid & 1, jr = tid >> 1;
  const int ntile = p.N / kKT;
  const int bh = blockIdx.x / ntile, j0 = (blockIdx.x % ntile) * kKT;
  const int j = j0 + jr;
  const size_t row = (size_t)bh * p.N + j;
  float kh[32], vh[32], dk[32], dv[32];
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    kh[e] = p.kr[row * kD + 32 * half + e];
    vh[e] = bf(p.v[row * kD + 32 * half + e]);
    dk[e] = 0.f;
    dv[e] = 0.f;
  }
  const int n1 = min(p.N, j0 + kKT - 1 + p.w);  // queries that see some key of the tile
  for (int n0 = j0; n0 < n1; n0 += kKT) {
    __syncthreads();
    for (int e = tid; e < kKT * kD; e += 128) {
      const int rr = e / kD, dd = e % kD;
      const int nn = n0 + rr;
      const size_t src = ((size_t)bh * p.N + min(nn, p.N - 1)) * kD + dd;
      s_q[rr][col(dd)] = p.qr[src] * kScale;
      s_g[rr][col(dd)] = p.g[src];
    }
    for (int e = tid; e < kKT; e += 128) {
      const int nn = min(n0 + e, p.N - 1);
      s_lse[e] = p.lse[(size_t)bh * p.N + nn];
      s_gdo[e] = p.gdo[(size_t)bh * p.N + nn];
    }
    __syncthreads();
    for (int rr = 0; rr < kKT; ++rr) {
      const int nn = n0 + rr;
      const float ps = dot32(kh, &s_q[rr][kH1 * half]);
      const float pd = dot32(vh, &s_g[rr][kH1 * half]);
      const float sc = ps + __shfl_xor_sync(0xffffffffu, ps, 1);
      const float dp = pd + __shfl_xor_sync(0xffffffffu, pd, 1);
      if (nn >= p.N || j > nn || j < nn - p.w + 1) continue;  // this key is not in n's window
      const float pr = __expf(sc - s_lse[rr]);
      const float ds = pr * (dp - s_gdo[rr]);  // the 1/8 is in s_q
      axpy32(dv, pr, &s_g[rr][kH1 * half]);
      axpy32(dk, ds, &s_q[rr][kH1 * half]);
    }
  }
  rotate_back_pair(dk, j, half, p.tab);
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    p.dk[row * kD + 32 * half + e] = dk[e];
    p.dv[row * kD + 32 * half + e] = dv[e];
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

size_t backward_workspace_bytes(const Shape &sh) {
  const size_t rows = (size_t)sh.BH() * sh.N;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  return up(rope_table_bytes(sh.N)) + 2 * up(rows * kD * 4) + 2 * up(rows * 4);
}

cudaError_t launch_backward(const BwdArgs &a, cudaStream_t st) {
  const Shape &sh = a.sh;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  const size_t rows = (size_t)sh.BH() * sh.N;
  unsigned char *ws = static_cast<unsigned char *>(a.ws);
  void *tab = ws;
  float *qr = reinterpret_cast<float *>(ws + up(rope_table_bytes(sh.N)));
  float *kr = qr + up(rows * kD * 4) / 4;
  float *lse = kr + up(rows * kD * 4) / 4;
  float *gdo = lse + up(rows * 4) / 4;
  cudaError_t e = launch_rope_table(tab, sh.N, a.rope_base, st);
  if (e != cudaSuccess) return e;
  const unsigned rb = (unsigned)((rows * (kD / 2) + 255) / 256);
  k8_rotate_kernel<<<rb, 256, 0, st>>>(static_cast<const uint16_t *>(a.q),
                                       static_cast<const float2 *>(tab), sh.N, rows, qr);
  k8_rotate_kernel<<<rb, 256, 0, st>>>(static_cast<const uint16_t *>(a.k),
                                       static_cast<const float2 *>(tab), sh.N, rows, kr);
  if ((e = cudaMemsetAsync(a.dmix, 0, sizeof(float) * sh.H, st)) != cudaSuccess) return e;
  BwdParams p;
  p.q = static_cast<const uint16_t *>(a.q);
  p.k = static_cast<const uint16_t *>(a.k);
  p.v = static_cast<const uint16_t *>(a.v);
  p.qr = qr;
  p.kr = kr;
  p.g = a.g;
  p.tab = static_cast<const float2 *>(tab);
  p.sel = a.sel;
  p.mix = a.mix;
  p.dq = a.dq;
  p.dk = a.dk;
  p.dv = a.dv;
  p.dmix = a.dmix;
  p.lse = lse;
  p.gdo = gdo;
  p.H = sh.H;
  p.N = sh.N;
  p.w = a.w;
  p.K = a.K;
  p.rms_eps = a.rms_eps;
  const unsigned nq = (unsigned)(sh.BH() * (sh.N / kQT));
  k8_win_q_kernel<<<nq, 256, 0, st>>>(p);
  k8_win_kv_kernel<<<(unsigned)(sh.BH() * (sh.N / kKT)), 128, 0, st>>>(p);
  const int dyn = kQT * (2 * kD + 2) * 4;
  if ((e = cudaFuncSetAttribute(k8_long_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                dyn)) != cudaSuccess)
    return e;
  k8_long_kernel<<<nq, 256, dyn, st>>>(p);
  return cudaGetLastError();
}

}  // namespace fs
