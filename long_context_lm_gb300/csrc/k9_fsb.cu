// k9_fsb.cu -- FS-B cell selection: beam search over two causal forests per
// head, then a token-level rerank.
//
// FreeSolo (ai.info summary, "Methodology in Plain English", FS-B: two
// balanced trees per head, over the full prefix and over the cells whose
// largest key norm exceeds a threshold tau; every node stores a mean key, a
// radius bounding its children, the largest cell norm and the earliest
// position; a beam of 16 nodes per level descends each tree by a provable
// upper bound on the cell scores beneath a node; the union of both beams is
// reranked by token-level log-sum-exp and the top K cells are read;
// paper.rainbus.top summary, 方法步骤详情 ⑤, 技术新颖性).
//
// Forest: the leaves are the forest's cells in position order (all cells, or
// the cells with a_c > tau); level j node i covers leaves [i 2^j, (i+1) 2^j)
// and stores the mean of their mean keys, a radius r (max over children of
// |mean_child - mean| + r_child), the largest a_c and its first cell.  A
// query of block beta searches the maximal aligned runs tiling the forest's
// leaves below A = beta Bq / s (the binary decomposition of their count), so
// no node it visits holds an unavailable cell.  Node bound for query n:
//   q . mean + |q| r + lambda a_max erf(sigma (n - p_first) / s),
// p_first = first * s + s / 2, above the score u_c of every cell beneath.
//
//   k9_build_kernel   one CTA per (batch, head, forest): the leaf list (a
//                     block scan over the cells for the tau forest, with a
//                     prefix count for the queries), then the levels
//   k9_search_kernel  one warp per query: the beam descent of both forests
//                     (a lane per candidate node), then the rerank (a lane per
//                     token) and the top K by (LSE desc, c asc)
#include "fs_common.cuh"
#include "fs_internal.h"

namespace fs {

FsbLayout fsb_layout(int C) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  FsbLayout L;
  L.C = C;
  L.levels = 1;
  size_t nodes = 0;
  for (int m = C;; m = (m + 1) / 2, ++L.levels) {
    L.level_off[L.levels - 1] = (int)nodes;
    nodes += (size_t)m;
    if (m <= 1) break;
  }
  L.nodes = (int)nodes;
  // per (batch, head): leaf lists (two), the tau forest's prefix count, then
  // per forest the node means and (radius, amax, first)
  L.list = 0;
  L.hcount = up(2 * (size_t)C * 4);
  L.mean = L.hcount + up(((size_t)C + 1) * 4);
  L.meta = L.mean + up(2 * nodes * kD * 4);
  L.head_bytes = L.meta + up(2 * nodes * 16);
  return L;
}

namespace {

constexpr int kBuildThreads = 256;

__global__ void __launch_bounds__(kBuildThreads) k9_build_kernel(const float *__restrict__ kbar,
                                                                 const float *__restrict__ amax,
                                                                 float tau, FsbLayout L,
                                                                 unsigned char *ws) {
  __shared__ int s_scan[kBuildThreads];
  const int bh = blockIdx.x >> 1, f = blockIdx.x & 1;  // forest 0: all cells, 1: a_c > tau
  const int tid = threadIdx.x, C = L.C;
  unsigned char *hs = ws + (size_t)bh * L.head_bytes;
  int *list = reinterpret_cast<int *>(hs + L.list) + (size_t)f * C;
  int *hcount = reinterpret_cast<int *>(hs + L.hcount);
  float *mean = reinterpret_cast<float *>(hs + L.mean) + (size_t)f * L.nodes * kD;
  float4 *meta = reinterpret_cast<float4 *>(hs + L.meta) + (size_t)f * L.nodes;
  const float *kb = kbar + (size_t)bh * C * kD;
  const float *am = amax + (size_t)bh * C;
  // leaf list in position order (tau forest: a block scan of the keep flags)
  int M = C;
  if (f == 0) {
    for (int c = tid; c < C; c += kBuildThreads) list[c] = c;
  } else {
    int base = 0;
    for (int c0 = 0; c0 < C; c0 += kBuildThreads) {
      const int c = c0 + tid;
      const int keep = c < C && am[c] > tau;
      s_scan[tid] = keep;
      __syncthreads();
      for (int o = 1; o < kBuildThreads; o <<= 1) {  // inclusive scan
        const int x = tid >= o ? s_scan[tid - o] : 0;
        __syncthreads();
        s_scan[tid] += x;
        __syncthreads();
      }
      const int excl = base + s_scan[tid] - keep;
      if (c < C) hcount[c] = excl;  // leaves of the tau forest below cell c
      if (keep) list[excl] = c;
      base += s_scan[kBuildThreads - 1];
      __syncthreads();
    }
    if (tid == 0) hcount[C] = base;
    M = base;
  }
  __syncthreads();
  // level 0: one leaf per cell of the list
  for (int e = tid; e < M * kD; e += kBuildThreads) {
    const int i = e / kD, dd = e % kD;
    mean[(size_t)i * kD + dd] = kb[(size_t)list[i] * kD + dd];
  }
  for (int i = tid; i < M; i += kBuildThreads)
    meta[i] = make_float4(0.f, am[list[i]], __int_as_float(list[i]), 0.f);
  __syncthreads();
  // levels 1.. from their children, one warp per node
  const int warp = tid >> 5, lane = tid & 31;
  int m = M;
  for (int j = 1; j < L.levels && m > 1; ++j) {
    const int mc = m;
    m = (m + 1) / 2;
    const float *cmean = mean + (size_t)L.level_off[j - 1] * kD;
    const float4 *cmeta = meta + L.level_off[j - 1];
    float *pmean = mean + (size_t)L.level_off[j] * kD;
    float4 *pmeta = meta + L.level_off[j];
    const int half = 1 << (j - 1);  // leaves under a full child
    for (int i = warp; i < m; i += kBuildThreads / 32) {
      const int c0 = 2 * i, c1 = 2 * i + 1;
      const bool two = c1 < mc;
      const float w0 = (float)min(half, M - c0 * half);
      const float w1 = two ? (float)min(half, M - c1 * half) : 0.f;
      const float inv = 1.f / (w0 + w1);
      float mu[2], a0[2], a1[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int dd = 2 * lane + e;
        a0[e] = cmean[(size_t)c0 * kD + dd];
        a1[e] = two ? cmean[(size_t)c1 * kD + dd] : 0.f;
        mu[e] = (w0 * a0[e] + w1 * a1[e]) * inv;
        pmean[(size_t)i * kD + dd] = mu[e];
      }
      float d0 = (a0[0] - mu[0]) * (a0[0] - mu[0]) + (a0[1] - mu[1]) * (a0[1] - mu[1]);
      float d1 = (a1[0] - mu[0]) * (a1[0] - mu[0]) + (a1[1] - mu[1]) * (a1[1] - mu[1]);
      d0 = warp_sum(d0);
      d1 = warp_sum(d1);
      if (lane == 0) {
        const float4 m0 = cmeta[c0];
        float r = sqrtf(d0) + m0.x, a = m0.y;
        if (two) {
          const float4 m1 = cmeta[c1];
          r = fmaxf(r, sqrtf(d1) + m1.x);
          a = fmaxf(a, m1.y);
        }
        // the bound needs r to cover every leaf: round up by a relative ulp
        pmeta[i] = make_float4(r * (1.f + 4e-7f), a, m0.z, 0.f);
      }
    }
    __syncthreads();
  }
}

struct SearchParams {
  const uint16_t *q, *k;           // [BH, N, 64] bf16
  const unsigned char *ws;
  FsbLayout L;
  const float *lambda, *sigma;
  int H, N, K, beam;
  long long nq;                    // BH * N
  int32_t *sel;                    // [BH, N, K]
};

__device__ __forceinline__ float bfv(uint16_t x) { return __uint_as_float((uint32_t)x << 16); }


// Sort key of a candidate node: higher bound first, then the lower first
// leaf, then the level; an empty position sorts last.  The bound's bits are mapped so that unsigned order is float order,
// then inverted for "higher first".
__device__ __forceinline__ unsigned long long node_key(float u, int first, int j) {
  const uint32_t b = __float_as_uint(u);
  const uint32_t ord = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return ((unsigned long long)(~ord) << 32) | ((unsigned long long)(uint32_t)first << 5) |
         (unsigned long long)(uint32_t)j;
}
__device__ __forceinline__ unsigned long long shfl_xor_u64(unsigned long long x, int m) {
  const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)x, m);
  const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(x >> 32), m);
  return ((unsigned long long)hi << 32) | lo;
}
// Ascending bitonic sort of the warp's NS * 32 keys, key p in lane p % 32,
// slot p / 32 (NS = 1 or 2).
template <int NS>
__device__ __forceinline__ void warp_sort(unsigned long long (&key)[2], int lane) {
#pragma unroll
  for (int k = 2; k <= 32 * NS; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j == 32) {  // partner in the other slot of the lane (k = 64: ascending)
        const unsigned long long a = key[0], b = key[1];
        key[0] = a < b ? a : b;
        key[1] = a < b ? b : a;
        continue;
      }
#pragma unroll
      for (int e = 0; e < NS; ++e) {
        const int pos = 32 * e + lane;
        const unsigned long long other = shfl_xor_u64(key[e], j);
        const bool up = (pos & k) == 0, lower = (pos & j) == 0;
        const unsigned long long mn = key[e] < other ? key[e] : other;
        const unsigned long long mx = key[e] < other ? other : key[e];
        key[e] = (lower == up) ? mn : mx;
      }
    }
  }
}

__global__ void __launch_bounds__(256) k9_search_kernel(const SearchParams p) {
  __shared__ float s_q[8][kD];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long gq = (long long)blockIdx.x * 8 + warp;  // query (bh, n)
  if (gq >= p.nq) return;  // the whole warp
  const int bh = (int)(gq / p.N), n = (int)(gq % p.N);
  const int h = bh % p.H;
  const FsbLayout &L = p.L;
  const int C = L.C;
  const size_t row = (size_t)bh * p.N + n;
  for (int dd = lane; dd < kD; dd += 32) s_q[warp][dd] = bfv(p.q[row * kD + dd]);
  __syncwarp();
  float qn2 = s_q[warp][lane] * s_q[warp][lane] + s_q[warp][lane + 32] * s_q[warp][lane + 32];
  const float qnorm = sqrtf(warp_sum(qn2));
  const float lam = p.lambda[h], sig = p.sigma[h];
  const int A = (n / kBq) * (kBq / kS);
  const unsigned char *hs = p.ws + (size_t)bh * L.head_bytes;
  const int *hcount = reinterpret_cast<const int *>(hs + L.hcount);
  // candidates of the union, one per lane (-1: none)
  int cand = -1, ncand = 0;
  for (int f = 0; f < 2; ++f) {
    const int m = f == 0 ? A : (A > 0 ? hcount[A] : 0);
    if (m == 0) continue;
    const int *list = reinterpret_cast<const int *>(hs + L.list) + (size_t)f * C;
    const float *mean = reinterpret_cast<const float *>(hs + L.mean) + (size_t)f * L.nodes * kD;
    const float4 *meta = reinterpret_cast<const float4 *>(hs + L.meta) + (size_t)f * L.nodes;
    // the beam: at most 32 (level, index) nodes, node b in lane b (the roots
    // number at most 24, the kept beams at most `beam` <= 16)
    int bj = -1, bi = 0;
    int nb = 0;
    {
      int start = 0;
      for (int j = 31 - __clz(m); j >= 0; --j)
        if (m & (1 << j)) {
          if (nb == lane) {
            bj = j;
            bi = start >> j;
          }
          ++nb;
          start += 1 << j;
        }
    }
    while (__any_sync(0xffffffffu, bj > 0)) {  // an inner node is left
      // candidates at fixed indices: beam node b gives index 2b (its first
      // child, or itself for a leaf) and 2b + 1 (its second child).  Eight
      // candidates per pass, four lanes each (16 contiguous dimensions of the
      // node mean); candidate (pass, g) keeps its key in lane 4g + pass % 4,
      // slot pass / 4 (the sort reorders all positions anyway).
      unsigned long long key[2] = {~0ull, ~0ull};
      const int npass = (2 * nb + 7) >> 3;
      const int g = lane >> 2, sub = lane & 3;
#pragma unroll
      for (int pass = 0; pass < 6; ++pass) {
        if (pass >= npass) break;  // the same for the whole warp
        const int c = pass * 8 + g, b = c >> 1, child = c & 1;
        const int pj = __shfl_sync(0xffffffffu, bj, b & 31);
        const int pi = __shfl_sync(0xffffffffu, bi, b & 31);
        const bool valid = b < nb && pj >= 0 && (pj > 0 || child == 0);
        const int cj = pj <= 0 ? 0 : pj - 1, ci = pj <= 0 ? pi : 2 * pi + child;
        const int node = L.level_off[cj] + ci;
        float dot = 0.f;
        if (valid) {
          const float4 *mu = reinterpret_cast<const float4 *>(mean + (size_t)node * kD) + 4 * sub;
          const float *qq = s_q[warp] + 16 * sub;
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const float4 x = __ldg(mu + v);
            dot = fmaf(qq[4 * v], x.x, fmaf(qq[4 * v + 1], x.y,
                  fmaf(qq[4 * v + 2], x.z, fmaf(qq[4 * v + 3], x.w, dot))));
          }
        }
        dot += __shfl_xor_sync(0xffffffffu, dot, 1);
        dot += __shfl_xor_sync(0xffffffffu, dot, 2);
        if (valid && sub == (pass & 3)) {
          // the bound: the dot, then the radius, norm and erf terms
          const float4 mt = __ldg(meta + node);
          const int first = __float_as_int(mt.z);
          const float pf = (float)(first * kS) + 0.5f * kS;
          // erf(x) rounds to 1 in fp32 once x >= 4 (erfc(4) = 1.5e-8): only
          // nodes that reach the newest cells need the special function
          const float x = sig * ((float)n - pf) / kS;
          const float u = dot + qnorm * mt.x + lam * mt.y * (x < 4.0f ? erff(x) : 1.0f);
          key[pass >> 2] = node_key(u, ci << cj, cj);
        }
      }
      // an inner node gives two candidates, a leaf one
      const int nvalid = __popc(__ballot_sync(0xffffffffu, lane < nb)) +
                         __popc(__ballot_sync(0xffffffffu, lane < nb && bj > 0));
      // rank order by one sort; the best `beam` form the next beam
      if (npass > 4)
        warp_sort<2>(key, lane);
      else
        warp_sort<1>(key, lane);
      nb = min(nvalid, p.beam);
      bj = lane < nb ? (int)(key[0] & 31u) : -1;
      bi = lane < nb ? (int)((uint32_t)(key[0] >> 5) & 0xffffffu) >> bj : 0;
    }
    // the beam's leaves join the union (cells, deduplicated; two beams of at
    // most 16 fit a lane each)
    for (int b = 0; b < nb; ++b) {
      const int i = __shfl_sync(0xffffffffu, bi, b);
      const int c = list[i];
      const bool dup = __any_sync(0xffffffffu, lane < ncand && cand == c);
      if (!dup) {
        if (lane == ncand) cand = c;
        ++ncand;
      }
    }
  }
  // rerank: LSE of the 32 token logits of each union cell.  Eight lanes per
  // token row (one 16-byte chunk each), four rows per load: lane l takes
  // chunk l % 8 of rows 4v + l / 8, v < 8, then the eight lanes of a row add
  // up its partial dots.
  float lse_mine = -INFINITY;
  const int tg = lane >> 3, chk = lane & 7;
  float qv[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) qv[e] = s_q[warp][8 * chk + e];
  for (int u = 0; u < ncand; ++u) {
    const int c = __shfl_sync(0xffffffffu, cand, u);
    const uint4 *kr = reinterpret_cast<const uint4 *>(p.k + ((size_t)bh * p.N + (size_t)c * kS) * kD);
    float part[8];
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      const uint4 x = __ldg(kr + (4 * v + tg) * (kD / 8) + chk);
      const uint32_t w[4] = {x.x, x.y, x.z, x.w};
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        dot = fmaf(qv[2 * e], bf16_lo(w[e]), dot);
        dot = fmaf(qv[2 * e + 1], bf16_hi(w[e]), dot);
      }
      part[v] = dot;
    }
#pragma unroll
    for (int o = 1; o < 8; o <<= 1)
#pragma unroll
      for (int v = 0; v < 8; ++v) part[v] += __shfl_xor_sync(0xffffffffu, part[v], o);
    // the lanes of row group tg now hold the logits of rows 4v + tg
    float mx = -INFINITY;
#pragma unroll
    for (int v = 0; v < 8; ++v) mx = fmaxf(mx, part[v] * 0.125f);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    float sum = 0.f;
#pragma unroll
    for (int v = 0; v < 8; ++v) sum += __expf(part[v] * 0.125f - mx);
    sum += __shfl_xor_sync(0xffffffffu, sum, 8);
    sum += __shfl_xor_sync(0xffffffffu, sum, 16);
    if (lane == u) lse_mine = mx + __logf(sum);
  }
  // top K by (LSE desc, c asc)
  int rank = 0;
  for (int u = 0; u < ncand; ++u) {
    const float x = __shfl_sync(0xffffffffu, lse_mine, u);
    const int c = __shfl_sync(0xffffffffu, cand, u);
    rank += lane < ncand && (x > lse_mine || (x == lse_mine && c < cand));
  }
  int32_t *dst = p.sel + row * p.K;
  if (lane < p.K) dst[lane] = -1;
  __syncwarp();
  if (lane < ncand && rank < p.K) dst[rank] = cand;
}

}  // namespace

cudaError_t launch_fsb(const void *q, const void *k, const float *kbar, const float *amax,
                       const float *lambda, const float *sigma, const Shape &sh, int K, int beam,
                       float tau, void *ws, int32_t *sel, cudaStream_t st) {
  const FsbLayout L = fsb_layout(sh.C());
  unsigned char *w = static_cast<unsigned char *>(ws);
  k9_build_kernel<<<sh.BH() * 2, kBuildThreads, 0, st>>>(kbar, amax, tau, L, w);
  SearchParams p;
  p.q = static_cast<const uint16_t *>(q);
  p.k = static_cast<const uint16_t *>(k);
  p.ws = w;
  p.L = L;
  p.lambda = lambda;
  p.sigma = sigma;
  p.H = sh.H;
  p.N = sh.N;
  p.K = K;
  p.beam = beam;
  p.sel = sel;
  const long long nq = (long long)sh.BH() * sh.N;
  p.nq = nq;
  k9_search_kernel<<<(unsigned)((nq + 7) / 8), 256, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace fs
