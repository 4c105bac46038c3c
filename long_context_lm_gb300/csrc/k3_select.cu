// k3_select.cu -- per-query cell scores and top-K selection on the tensor
// cores (tcgen05 + TMEM).
//
// FreeSolo (paper.rainbus.top summary, 核心方法 and 方法步骤详情 ⑤; 局限与改进
// for the erf factor g_h >= erf(2); ai.info summary, "Methodology in Plain
// English"): a candidate cell c of query n scores
//     u = q_n . kbar_c + lambda_h * a_c * erf(sigma_h * (n - p_c) / s),
// p_c = c*s + s/2, with the unrotated query, and the K best cells are read.
// Candidates are the block's FS-L pool (<= P+W cells) or, in FS mode, every
// cell that ends at or before the block start (processed in chunks of 128).
//
// One CTA per (head, 128-query block).  The content term of all 128 queries
// against all candidates is one tcgen05 product D[128 x Nc] in TMEM: q is
// exactly bf16, and every fp32 mean key is split into three bf16 terms
// (hi + mid + lo, 24 significant bits), so three MMA chains accumulating in
// fp32 give fp32-grade dot products -- the scores decide indices, so they
// must not carry bf16 rounding.  Each scoring thread owns one query row
// (= TMEM lane): it adds the erf bias and keeps a register top-K ranked by
// (u desc, c asc).  erf(x) is exactly 1 in fp32 once x >= 4 (erfc(4) = 1.5e-8
// is below half an ulp of 1), which holds for every cell but the newest few,
// so the special function is evaluated only below that point.
#include "fs_common.cuh"
#include "fs_internal.h"
#include "tc05.cuh"

namespace fs {
namespace {

constexpr int kChunk = 128;       // candidates per MMA (N <= 128)
constexpr int kThreads = 192;     // warps 0-3 score, warp 4 MMA, all stage operands
constexpr int kGather = 4;        // 16-byte key chunks a thread gathers per pass
constexpr int kInvalid = 0x7fffffff;          // candidate slot holding no cell
constexpr int kNeedsErf = int(0x80000000u);   // flag bit on a candidate's cell id
constexpr uint32_t kOffQ = 0, kOffK = 16384;  // then 3 split tiles of `rows` x 128 B

// candidate rows a chunk holds: the pool capacity (FS-L) or a full chunk (FS)
__host__ __device__ constexpr int chunk_rows(int fs_mode, int cap) {
  return fs_mode ? kChunk : ((cap < kChunk ? cap : kChunk) + 15) / 16 * 16;
}

__device__ __forceinline__ bool ranks_before(float u, int c, float u2, int c2) {
  return u > u2 || (u == u2 && c < c2);
}

// erf of the bias argument; only the newest few cells need it (x < 4), so it
// is kept out of line to keep the unrolled scoring loop small
__device__ __noinline__ float erf_bias(float x) { return erff(x); }

template <int K>
__global__ void __launch_bounds__(kThreads, K <= 5 ? 4 : 3) k3_select_tc_kernel(
    const __nv_bfloat16 *__restrict__ q, const float *__restrict__ kbar,
    const float *__restrict__ amax, const int32_t *__restrict__ pool,
    const int32_t *__restrict__ pool_count, const float *__restrict__ lambda,
    const float *__restrict__ sigma, int H, int N, int cap, int W, int fs_mode,
    int32_t *__restrict__ sel, float *__restrict__ sel_score, int *err) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // per candidate, what every row shares: (cell id, lambda_h * a_c).  The id
  // is kInvalid for an empty or skipped slot (lambda * a then -inf, so it never
  // ranks), and carries kNeedsErf when the bias factor can fall below 1 for
  // some row of the block.
  __shared__ int2 s_ca[kChunk];
  __shared__ uint32_t s_gerf;  // bit g: a candidate of group g (16) needs the erf
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t s_tmem;

  const int tid = threadIdx.x, warp = tid >> 5;
  const int beta = blockIdx.x, bh = blockIdx.y, h = bh % H;
  const int C = N / kS, nblk = N / kBq;
  const int b0 = beta * kBq;
  const size_t head = (size_t)bh * N;
  const int A = beta * (kBq / kS);
  const int count = fs_mode ? A : min(max(pool_count[(size_t)bh * nblk + beta], 0), min(cap, kChunk));
  const int32_t *pl = fs_mode ? nullptr : pool + ((size_t)bh * nblk + beta) * cap;

  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_fence_init();
  }
  if (warp == 4) {
    tc::tmem_alloc(&s_tmem, 128);
    tc::tmem_relinquish();
  }
  // query tile -> shared (K-major SW128) by asynchronous copies, so that it
  // lands while the candidate gathers below are in flight
  for (int p = tid; p < kBq * 8; p += kThreads) {
    const int r = p >> 3, ch = p & 7;
    cp_async16(smem + kOffQ + swz128(r, ch), q + (head + b0 + r) * kD + ch * 8);
  }
  cp_async_commit();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s_tmem;
  const uint32_t sbase = smem_u32(smem);

  const int r = tid;  // query row of a scoring thread
  const int n = b0 + r;
  const float lam = lambda[h], sig_s = sigma[h] * (1.0f / kS);
  // ranked top-K (u desc, c asc) in registers; wu mirrors the K-th score,
  // so that a group of candidates that no row can take costs one comparison each
  float bu[K];
  int bc[K];
#pragma unroll
  for (int i = 0; i < K; ++i) {
    bu[i] = -INFINITY;
    bc[i] = kInvalid;
  }
  float wu = -INFINITY;
  bool ok = true;

  for (int base = 0, chunk = 0; base < count; base += kChunk, ++chunk) {
    if (tid == 0) s_gerf = 0u;
    __syncthreads();
    const int nc = min(kChunk, count - base);
    const int np = (nc + 15) / 16 * 16;
    // candidate ids, norms and mean keys in one pass: eight threads share a
    // candidate (one 16-byte output chunk each), and the id is the only load
    // ahead of the gathers.  Rows beyond nc or skipped cells stay zero.
    const uint32_t tile = (uint32_t)chunk_rows(fs_mode, cap) * 128;
    for (int p0 = 0; p0 < np * 8; p0 += kGather * kThreads) {
      int cj[kGather];
#pragma unroll
      for (int it = 0; it < kGather; ++it) {
        const int j = (p0 + tid + it * kThreads) >> 3;
        int c = -1;
        if (j < nc) {
          // FS-L: the ranked older cells (a_c desc) first, the W recent
          // ones last: the rows' K-th scores rise sooner, so the warp vote
          // turns more groups of candidates away (the result does not depend
          // on the order)
          const int nrec = min(min(W, A), count), jj = j < count - nrec ? nrec + j : j - (count - nrec);
          c = fs_mode ? base + j : __ldg(pl + jj);
          if (c < 0 || c >= A) c = -1;  // not a cell this block may read: skipped
        }
        cj[it] = c;
      }
      float x[kGather][8];
#pragma unroll
      for (int it = 0; it < kGather; ++it) {
        const int p = p0 + tid + it * kThreads, j = p >> 3, ch = p & 7;
        const int c = cj[it];
        if (c >= 0) {
          const float4 *src = reinterpret_cast<const float4 *>(kbar + ((size_t)bh * C + c) * kD) + 2 * ch;
          const float4 u0 = __ldg(src), u1 = __ldg(src + 1);
          x[it][0] = u0.x; x[it][1] = u0.y; x[it][2] = u0.z; x[it][3] = u0.w;
          x[it][4] = u1.x; x[it][5] = u1.y; x[it][6] = u1.z; x[it][7] = u1.w;
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) x[it][e] = 0.f;
        }
        if (ch == 0 && j < np) {
          int cf = kInvalid;
          float la = -INFINITY;
          if (c >= 0) {
            la = lam * __ldg(amax + (size_t)bh * C + c);
            // x grows with n, so the block's first row has the smallest one
            const float x0 = sig_s * ((float)(b0 - c * kS) - 0.5f * kS);
            cf = x0 < 4.0f ? (c | kNeedsErf) : c;
          }
          s_ca[j] = make_int2(cf, __float_as_int(la));
          if (cf < 0) atomicOr(&s_gerf, 1u << (j >> 4));
        }
      }
#pragma unroll
      for (int it = 0; it < kGather; ++it) {
        const int p = p0 + tid + it * kThreads, j = p >> 3, ch = p & 7;
        if (j >= np) break;
        uint32_t hw[4], mw[4], lw[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          hw[e] = pack_bf16(x[it][2 * e], x[it][2 * e + 1]);
          const float r0 = x[it][2 * e] - bf16_lo(hw[e]), r1 = x[it][2 * e + 1] - bf16_hi(hw[e]);
          mw[e] = pack_bf16(r0, r1);
          lw[e] = pack_bf16(r0 - bf16_lo(mw[e]), r1 - bf16_hi(mw[e]));
        }
        const uint32_t off = swz128(j, ch);
        *reinterpret_cast<uint4 *>(smem + kOffK + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        *reinterpret_cast<uint4 *>(smem + kOffK + tile + off) = make_uint4(mw[0], mw[1], mw[2], mw[3]);
        *reinterpret_cast<uint4 *>(smem + kOffK + 2 * tile + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
      }
    }
    cp_async_wait<0>();  // the query tile (first chunk; a no-op afterwards)
    tc::fence_async_smem();
    __syncthreads();
    if (tid == 128) {  // warp 4, one thread: D = Q.(hi + mid + lo)^T
      tc::fence_after_sync();
      const uint32_t id = tc::idesc_bf16(128, np, 0);
      const uint32_t sq = sbase + kOffQ;
#pragma unroll
      for (int part = 0; part < 3; ++part) {
        const uint32_t sk = sbase + kOffK + part * tile;
#pragma unroll
        for (int k = 0; k < kD / 16; ++k)
          tc::mma_ss(tmem, tc::desc_sw128(sq + 32 * k), tc::desc_sw128(sk + 32 * k), id,
                     (part > 0 || k > 0) ? 1u : 0u);
      }
      tc::mma_commit(&bar);
    }
    if (warp < 4) {
      ok = tc::mbar_wait(&bar, chunk & 1, err) && ok;
      tc::fence_after_sync();
      const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
      for (int j0 = 0; j0 < np; j0 += 32) {
        uint32_t d[32];
        tc::tmem_ld32(taddr + j0, d);  // columns past np are read, never used
        tc::tmem_wait_ld();
        // sixteen candidates at a time: their scores, then one warp vote on
        // whether any lane's row may take one of them (score >= its K-th)
#pragma unroll
        for (int j16 = 0; j16 < 32; j16 += 16) {
          if (j16 == 16 && j0 + 16 >= np) break;  // np is a multiple of 16
          float u16[16];
          int c16[16];
          bool any16 = false;
          if ((s_gerf >> ((j0 + j16) >> 4)) & 1u) {  // some candidate of the group needs the erf
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int2 ca = s_ca[j0 + j16 + e];
              const float la = __int_as_float(ca.y);
              int c = ca.x;
              float u;
              if (c < 0) {  // kNeedsErf (the same for every lane of the warp)
                c &= ~kNeedsErf;
                const float x = sig_s * ((float)(n - c * kS) - 0.5f * kS);
                const float g = x < 4.0f ? erf_bias(x) : 1.0f;
                u = __uint_as_float(d[j16 + e]) + la * g;
              } else {
                u = __uint_as_float(d[j16 + e]) + la;  // g = 1 exactly
              }
              u16[e] = u;
              c16[e] = c;
              any16 |= u >= wu;  // a superset of the candidates that rank before the K-th
            }
          } else {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int2 ca = s_ca[j0 + j16 + e];
              const float u = __uint_as_float(d[j16 + e]) + __int_as_float(ca.y);
              u16[e] = u;
              c16[e] = ca.x;
              any16 |= u >= wu;
            }
          }
          if (!__any_sync(0xffffffffu, any16)) continue;
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            // where the candidate goes: its rank against each kept entry, all
            // tests independent (the list is sorted, so they are monotone in
            // k); then every entry moves in one step.  A lane whose row does
            // not take it fails every test and keeps its list.
            const float u = u16[e];
            const int cu = c16[e];
            bool s[K];
#pragma unroll
            for (int k = 0; k < K; ++k) s[k] = ranks_before(u, cu, bu[k], bc[k]);
#pragma unroll
            for (int k = K - 1; k > 0; --k) {
              bu[k] = s[k] ? (s[k - 1] ? bu[k - 1] : u) : bu[k];
              bc[k] = s[k] ? (s[k - 1] ? bc[k - 1] : cu) : bc[k];
            }
            bu[0] = s[0] ? u : bu[0];
            bc[0] = s[0] ? cu : bc[0];
            wu = bu[K - 1];
          }
        }
      }
    }
    tc::fence_before_sync();
    __syncthreads();  // shared tiles and TMEM are reused by the next chunk
  }
  cp_async_wait<0>();  // a block with no candidates never waited above
  if (warp < 4 && ok) {
#pragma unroll
    for (int i = 0; i < K; ++i) {
      const bool valid = bc[i] != kInvalid;  // fewer than K readable cells
      sel[(head + n) * K + i] = valid ? bc[i] : -1;
      if (sel_score) sel_score[(head + n) * K + i] = valid ? bu[i] : 0.f;
    }
  }
  if (warp == 4) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 128);
  }
}

}  // namespace

cudaError_t launch_select(const void *q, const float *kbar, const float *amax,
                          const int32_t *pool, const int32_t *pool_count, const float *lambda,
                          const float *sigma, const Shape &sh, int K, int cap, int W,
                          bool fs_mode, int32_t *sel, float *sel_score, int *err,
                          cudaStream_t st) {
  const int smem = 16384 + 3 * chunk_rows(fs_mode ? 1 : 0, cap) * 128 + 1024;
  dim3 grid(sh.nblk(), sh.BH());
  const __nv_bfloat16 *qb = static_cast<const __nv_bfloat16 *>(q);
  const int fsm = fs_mode ? 1 : 0;
  auto go = [&](auto kern) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kThreads, smem, st>>>(qb, kbar, amax, pool, pool_count, lambda, sigma, sh.H,
                                       sh.N, cap, W, fsm, sel, sel_score, err);
    return cudaSuccess;
  };
  cudaError_t e;
  switch (K) {
    case 1: e = go(k3_select_tc_kernel<1>); break;
    case 2: e = go(k3_select_tc_kernel<2>); break;
    case 3: e = go(k3_select_tc_kernel<3>); break;
    case 4: e = go(k3_select_tc_kernel<4>); break;
    case 5: e = go(k3_select_tc_kernel<5>); break;
    case 6: e = go(k3_select_tc_kernel<6>); break;
    case 7: e = go(k3_select_tc_kernel<7>); break;
    default: e = go(k3_select_tc_kernel<8>); break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace fs
