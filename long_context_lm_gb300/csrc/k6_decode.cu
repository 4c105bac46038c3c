// k6_decode.cu -- one decode step of FS-L attention against its bounded state.
//
// FreeSolo (paper.rainbus.top summary, 核心方法 (prefill linear in N, decode
// state of constant size), 方法步骤详情 ②-⑥; ai.info summary, "Methodology
// in Plain English"): at decode time a head keeps the key/value history, the
// summaries (kbar_c, a_c) of its closed cells and the pool of its current
// query block; token t is answered from the w newest keys (RoPE window) and
// the K pool cells its query selects (NoPE readout + RMSNorm), mixed by m_h.
//
// State of one (batch, head), owned by the caller:
//   k_cache, v_cache [n_cap, d] bf16   rows < t hold the history
//   kbar [n_cap/s, d], amax [n_cap/s]  cells < floor(t/s) hold their summaries
//   pool [P+W], pool_count             the pool of block floor((t-1)/Bq), laid
//                                      out as fs_prune_cells writes a block's
//                                      row (recent cells, then the older cells
//                                      by rank); for t = 0 a count of 0
// One step for token t:
//   1. writes k_t, v_t into row t of the caches;
//   2. at a block start (t % Bq == 0, t > 0) advances the pool to block
//      t/Bq: the cells that leave the W-cell recency window join the ranked
//      older list, which keeps its best P by (a_c desc, c asc) -- the top P
//      of a growing set is the top P of the old top P plus the newcomers;
//   3. scores the pool with q_t (a3), reads the K best cells out with
//      RMSNorm (a4), attends over rows [t-w+1, t] with RoPE and mixes (a5);
//   4. when row t closes a cell ((t+1) % s == 0), writes that cell's kbar
//      and a_c, bit-identical to the prefill's cell summaries.
// One CTA of 256 threads per (batch, head); a step is launch-latency bound.
//
// Angles: RoPE enters as q_t . R(j - t) k_j.  cos / sin of o*theta_i for
// o = -(64a + r) come from two per-CTA tables (r < 64, a < 16) joined by the
// angle-sum identity; the table entries are sincospi of o*theta_i/pi with
// theta_i/pi carried as a 13-bit head (exact products with o) plus a 24-bit
// tail, reduced modulo 2 exactly before the call.
#include "cell_summary.cuh"
#include "fs_common.cuh"
#include "fs_internal.h"

namespace fs {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxWin = 1024;
constexpr int kMaxPool = kMaxP + 8;  // P + W with W <= 8 in practice; checked on the host
constexpr int kMaxTok = kMaxK * kS;

struct DecodeParams {
  const uint16_t *q_t, *k_t, *v_t;  // [BH, d] bf16
  uint16_t *k_cache, *v_cache;      // [BH, n_cap, d] bf16
  float *kbar, *amax;               // [BH, n_cap/s, d], [BH, n_cap/s]
  int32_t *pool, *pool_count;       // [BH, P+W], [BH]
  const float *lambda, *sigma, *mix;
  int H, t, n_cap, P, W, K, w;
  double rope_base;
  float rms_eps;
  float *out;                       // [BH, d] f32
  int32_t *sel_out;                 // [BH, K] (nullable)
};

__device__ __forceinline__ float bf16f(uint16_t x) { return __uint_as_float((uint32_t)x << 16); }

// block-wide max / sum over 256 threads (red: 8 floats of shared scratch)
__device__ __forceinline__ float block_max(float v, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = red[0];
#pragma unroll
  for (int i = 1; i < kThreads / 32; ++i) m = fmaxf(m, red[i]);
  return m;
}
__device__ __forceinline__ float block_sum(float v, float *red) {
  v = warp_sum(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < kThreads / 32; ++i) s += red[i];
  return s;
}

// sum_i wgt[i] * v[row(i)] for i < n: warp w takes i = w, w+8, ...; lane l
// owns dims 2l, 2l+1 (one 32-bit load per row), sixteen rows in flight per
// warp; the eight warp partials go to part[w] for the caller to add up.
template <typename RowOf>
__device__ __forceinline__ void weighted_rows(const uint16_t *__restrict__ vbase, const float *wgt,
                                              int n, RowOf row_of, const float *vt_row,
                                              float2 (*part)[kD / 2]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float ax = 0.f, ay = 0.f;
  for (int i0 = warp; i0 < n; i0 += 16 * (kThreads / 32)) {
    uint32_t x[16];
    float wv[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      const int i = i0 + u * (kThreads / 32);
      wv[u] = 0.f;
      x[u] = 0u;
      if (i < n) {
        const long long r = row_of(i);
        wv[u] = wgt[i];
        if (r >= 0)
          x[u] = reinterpret_cast<const uint32_t *>(vbase + (size_t)r * kD)[lane];
        else  // the new token's row, from shared memory
          x[u] = pack_bf16(vt_row[2 * lane], vt_row[2 * lane + 1]);
      }
    }
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      ax = fmaf(wv[u], bf16_lo(x[u]), ax);
      ay = fmaf(wv[u], bf16_hi(x[u]), ay);
    }
  }
  part[warp][lane] = make_float2(ax, ay);
}

__device__ __forceinline__ bool ranks_before(float a, int c, float a2, int c2) {
  return a > a2 || (a == a2 && c < c2);
}

__global__ void __launch_bounds__(kThreads) k6_decode_kernel(const DecodeParams p) {
  __shared__ float s_q[kD], s_k[kD], s_v[kD];
  __shared__ int s_pool[kMaxPool];
  __shared__ int s_cand_c[kMaxPool];
  __shared__ float s_cand_a[kMaxPool];
  __shared__ int s_count;
  __shared__ float s_u[kMaxPool];
  __shared__ int s_sel[kMaxK];
  __shared__ float s_lg[kMaxWin];
  __shared__ float2 s_part[kThreads / 32][kD / 2];
  __shared__ float s_olong[kD];
  __shared__ float s_red[8];
  __shared__ float s_th_hi[kD / 2], s_th_lo[kD / 2];
  __shared__ float2 s_tr[64][kD / 2], s_ta[kMaxWin / 64][kD / 2];

  const int bh = blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = bh % p.H, t = p.t;
  const int C = p.n_cap / kS;
  const size_t row0 = (size_t)bh * p.n_cap;
  const int cap = p.P + p.W;

  // ---- 1. the new token: registers of the CTA, and row t of the caches
  if (tid < kD) {
    s_q[tid] = bf16f(p.q_t[(size_t)bh * kD + tid]);
    s_k[tid] = bf16f(p.k_t[(size_t)bh * kD + tid]);
    s_v[tid] = bf16f(p.v_t[(size_t)bh * kD + tid]);
  } else if (tid < kD + 8) {
    const int c = tid - kD;
    reinterpret_cast<uint4 *>(p.k_cache + (row0 + t) * kD)[c] =
        reinterpret_cast<const uint4 *>(p.k_t + (size_t)bh * kD)[c];
  } else if (tid < kD + 16) {
    const int c = tid - kD - 8;
    reinterpret_cast<uint4 *>(p.v_cache + (row0 + t) * kD)[c] =
        reinterpret_cast<const uint4 *>(p.v_t + (size_t)bh * kD)[c];
  }
  // theta_i / pi as a 13-bit head and a tail (products with |o| < 2^11 exact)
  if (tid < kD / 2) {
    const double x = pow(p.rope_base, -2.0 * tid / kD) / 3.14159265358979323846;
    const float hi = __uint_as_float(__float_as_uint((float)x) & 0xfffff800u);
    s_th_hi[tid] = hi;
    s_th_lo[tid] = (float)(x - (double)hi);
  }
  // ---- 2. the pool of block t / Bq
  const int beta = t / kBq, A = beta * (kBq / kS);
  int32_t *gpool = p.pool + (size_t)bh * cap;
  const float *am = p.amax + (size_t)bh * C;
  const bool advance = t > 0 && t % kBq == 0;
  const int cnt_prev = p.pool_count[bh];
  for (int i = tid; i < cap; i += kThreads) s_pool[i] = gpool[i];
  if (tid == 0) s_count = cnt_prev;
  if (advance) {
    // candidates: the previous ranked older cells, then the cells [Lp, L)
    // leaving the recency window; each one's rank among all of them is the
    // number that rank before it, so the kept P land in order in one pass
    const int Ap = A - kBq / kS;
    const int nrec_p = min(p.W, Ap), Lp = Ap - nrec_p;
    const int nrec = min(p.W, A), L = A - nrec;
    const int keep_p = cnt_prev - nrec_p;
    const int ncand = keep_p + (L - Lp);
    const int keep = min(p.P, L);
    __syncthreads();  // s_pool holds the previous pool
    if (tid < ncand) {
      s_cand_c[tid] = tid < keep_p ? s_pool[nrec_p + tid] : Lp + (tid - keep_p);
      s_cand_a[tid] = am[s_cand_c[tid]];
    }
    __syncthreads();
    int rank = 0, my_c = -1;
    if (tid < ncand) {
      my_c = s_cand_c[tid];
      const float my_a = s_cand_a[tid];
      for (int j = 0; j < ncand; ++j) rank += ranks_before(s_cand_a[j], s_cand_c[j], my_a, my_c);
    }
    __syncthreads();  // every candidate has been read before s_pool is rewritten
    for (int i = tid; i < cap; i += kThreads) s_pool[i] = i < nrec ? L + i : -1;
    __syncthreads();
    if (tid < ncand && rank < keep) s_pool[nrec + rank] = my_c;
    if (tid == 0) s_count = nrec + min(keep, ncand);
    __syncthreads();
    for (int i = tid; i < cap; i += kThreads) gpool[i] = s_pool[i];
    if (tid == 0) p.pool_count[bh] = s_count;
  }
  __syncthreads();
  // angle tables: rows r*theta (r < 64) and 64a*theta (a < 16), sign of o applied later
  for (int i = tid; i < (64 + kMaxWin / 64) * (kD / 2); i += kThreads) {
    const int row = i / (kD / 2), k = i % (kD / 2);
    const int o = row < 64 ? row : 64 * (row - 64);
    const float head = fmodf((float)o * s_th_hi[k], 2.f);  // exact: o < 2^11, head has 13 bits
    float sn, cs;
    sincospif(head + (float)o * s_th_lo[k], &sn, &cs);
    if (row < 64)
      s_tr[row][k] = make_float2(cs, sn);
    else
      s_ta[row - 64][k] = make_float2(cs, sn);
  }

  // ---- 3a. score the pool (a3): u = q . kbar_c + lambda * a_c * erf(sigma (t - p_c) / s)
  const int nc = s_count;
  const float lam = p.lambda[h], sig = p.sigma[h];
  for (int i = warp; i < nc; i += kThreads / 32) {
    const int c = s_pool[i];
    const float2 kb = reinterpret_cast<const float2 *>(p.kbar + ((size_t)bh * C + c) * kD)[lane];
    const float dot = warp_sum(fmaf(s_q[2 * lane], kb.x, s_q[2 * lane + 1] * kb.y));
    if (lane == 0) {
      const float pc = (float)(c * kS) + 0.5f * kS;
      s_u[i] = dot + lam * p.amax[(size_t)bh * C + c] * erff(sig * ((float)t - pc) / kS);
    }
  }
  __syncthreads();
  // top K by (u desc, c asc): rank of each candidate by counting
  if (tid < kMaxK) s_sel[tid] = -1;
  __syncthreads();
  if (tid < nc) {
    const float u = s_u[tid];
    const int c = s_pool[tid];
    int rank = 0;
    for (int j = 0; j < nc; ++j) rank += ranks_before(s_u[j], s_pool[j], u, c);
    if (rank < p.K) s_sel[rank] = c;
  }
  __syncthreads();
  if (p.sel_out && tid < p.K) p.sel_out[(size_t)bh * p.K + tid] = s_sel[tid];

  // ---- 3b. NoPE readout over the selected cells' tokens (a4), then RMSNorm
  int nsel = 0;
  for (int k = 0; k < p.K; ++k) nsel += s_sel[k] >= 0;
  const int ntok = nsel * kS;  // selected ids are packed first, -1 after
  float lg = -INFINITY;
  if (tid < ntok) {
    const int tok = s_sel[tid / kS] * kS + tid % kS;
    const uint4 *kr = reinterpret_cast<const uint4 *>(p.k_cache + (row0 + tok) * kD);
    float dot = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 x = kr[c];
      const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        dot = fmaf(s_q[8 * c + 2 * j], bf16_lo(wv[j]), dot);
        dot = fmaf(s_q[8 * c + 2 * j + 1], bf16_hi(wv[j]), dot);
      }
    }
    lg = dot * 0.125f;
  }
  const float mlong = block_max(lg, s_red);
  const float pl = tid < ntok ? __expf(lg - mlong) : 0.f;
  if (tid < kMaxTok) s_lg[tid] = pl;
  const float llong = block_sum(pl, s_red);  // also orders the s_lg writes
  weighted_rows(p.v_cache + row0 * kD, s_lg, ntok,
                [&](int i) { return (long long)(s_sel[i / kS] * kS + i % kS); }, s_v, s_part);
  __syncthreads();
  if (tid < kD) {
    float o = 0.f;
#pragma unroll
    for (int w8 = 0; w8 < kThreads / 32; ++w8) {
      const float2 pp = s_part[w8][tid >> 1];
      o += (tid & 1) ? pp.y : pp.x;
    }
    s_olong[tid] = ntok > 0 ? o / llong : 0.f;
  }
  __syncthreads();
  float ss = tid < kD ? s_olong[tid] * s_olong[tid] : 0.f;
  ss = block_sum(ss, s_red);
  const float rms_scale = ntok > 0 ? rsqrtf(ss / kD + p.rms_eps) : 0.f;

  // ---- 3c. RoPE window over rows [t - w + 1, t] (a5)
  const int j0 = max(0, t - p.w + 1), nwin = t - j0 + 1;
  float mloc = -INFINITY;
  for (int i = tid; i < nwin; i += kThreads) {
    const int j = j0 + i, o = t - j;  // R(j - t) = R(-o)
    const uint4 *kr = reinterpret_cast<const uint4 *>(p.k_cache + (row0 + j) * kD);
    float kx[kD];
    if (j == t) {
#pragma unroll
      for (int c = 0; c < kD; ++c) kx[c] = s_k[c];
    } else {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 x = kr[c];
        const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          kx[8 * c + 2 * jj] = bf16_lo(wv[jj]);
          kx[8 * c + 2 * jj + 1] = bf16_hi(wv[jj]);
        }
      }
    }
    const float2 *tr = s_tr[o & 63], *ta = s_ta[o >> 6];
    float dot = 0.f;
#pragma unroll
    for (int k = 0; k < kD / 2; ++k) {
      // cos / sin of o*theta by the angle sum, then of -o*theta
      const float2 a = tr[k], b = ta[k];
      const float c = fmaf(a.x, b.x, -a.y * b.y), s = -fmaf(a.y, b.x, a.x * b.y);
      const float y0 = fmaf(kx[k], c, -kx[k + kD / 2] * s);
      const float y1 = fmaf(kx[k], s, kx[k + kD / 2] * c);
      dot = fmaf(s_q[k], y0, fmaf(s_q[k + kD / 2], y1, dot));
    }
    s_lg[i] = dot * 0.125f;
    mloc = fmaxf(mloc, dot * 0.125f);
  }
  const float mwin = block_max(mloc, s_red);  // its barriers also order the s_lg writes
  float lsum = 0.f;
  for (int i = tid; i < nwin; i += kThreads) {
    const float e = __expf(s_lg[i] - mwin);
    s_lg[i] = e;
    lsum += e;
  }
  const float lwin = block_sum(lsum, s_red);
  weighted_rows(p.v_cache + row0 * kD, s_lg, nwin,
                [&](int i) { return j0 + i == t ? -1ll : (long long)(j0 + i); }, s_v, s_part);
  __syncthreads();
  if (tid < kD) {
    float owin = 0.f;
#pragma unroll
    for (int w8 = 0; w8 < kThreads / 32; ++w8) {
      const float2 pp = s_part[w8][tid >> 1];
      owin += (tid & 1) ? pp.y : pp.x;
    }
    owin /= lwin;
    p.out[(size_t)bh * kD + tid] = owin + p.mix[h] * s_olong[tid] * rms_scale;
  }

  // ---- 4. row t closes cell t / s: its summary, as the prefill computes it
  if ((t + 1) % kS == 0 && warp == 0) {
    const int c = t / kS;
    float x[8][8];
    load_cell_bf16<false>(reinterpret_cast<const uint4 *>(p.k_cache + (row0 + (size_t)c * kS) * kD),
                          lane, x);
    cell_summary_warp(x, lane, p.kbar + ((size_t)bh * C + c) * kD, p.amax + (size_t)bh * C + c);
  }
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t st) {
  DecodeParams p;
  p.q_t = static_cast<const uint16_t *>(a.q_t);
  p.k_t = static_cast<const uint16_t *>(a.k_t);
  p.v_t = static_cast<const uint16_t *>(a.v_t);
  p.k_cache = static_cast<uint16_t *>(a.k_cache);
  p.v_cache = static_cast<uint16_t *>(a.v_cache);
  p.kbar = a.kbar;
  p.amax = a.amax;
  p.pool = a.pool;
  p.pool_count = a.pool_count;
  p.lambda = a.lambda;
  p.sigma = a.sigma;
  p.mix = a.mix;
  p.H = a.H;
  p.t = a.t;
  p.n_cap = a.n_cap;
  p.P = a.P;
  p.W = a.W;
  p.K = a.K;
  p.w = a.w;
  p.rope_base = a.rope_base;
  p.rms_eps = a.rms_eps;
  p.out = a.out;
  p.sel_out = a.sel_out;
  k6_decode_kernel<<<a.batch * a.H, kThreads, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace fs
