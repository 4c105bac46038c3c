// k6_decode.cu -- FS-L decoding from a bounded per-head state.
//
// FreeSolo (ai.info summary, "Methodology in Plain English": the FS-L pool
// holds at most 72 cells -- the 8 most recent plus the 64 with the largest key
// norm -- and changes only at query-block boundaries, so the streaming cache
// stays small; "Why This Matters": a bounded state; paper.rainbus.top summary,
// 核心方法: linear prefill and a decode state of constant size, 实验结果: the
// attention buffer stays constant from 4k to 256k, 局限与改进: repeated buffer
// copies are the weakness of the reference streaming cache).
//
// State of one (batch, head), fixed in size whatever the position t:
//   window ring    the last w keys and values (raw bf16), row j at j mod w;
//   cell slots     P + W + Bq/s + 1 slots of one cell each: raw keys and
//                  values (s rows), mean key kbar_c (fp32), largest key norm
//                  a_c and the cell id;
//   lists          the W recent available cells, the running top-P older
//                  cells in rank order (a_c desc, c asc), the closed cells
//                  not yet available (at most Bq/s), the open cell, and the
//                  free slots.
// A cell lives in one slot from its first token until it leaves the pool:
// nothing is ever moved between slots.  One step for token t:
//   1. at a block start (t % Bq == 0, t > 0) the pending cells become
//      recent; the cells leaving the W-cell recency window join the ranked
//      older list, which keeps its best P (a dropped cell frees its slot:
//      the top-P threshold only rises, so it is never needed again);
//   2. writes k_t, v_t into the ring and the open cell's slot (opening one
//      from the free list when t starts a cell);
//   3. scores the pool with q_t (a3), reads the K best cells' raw rows out
//      with RMSNorm (a4), attends over the ring with RoPE and mixes (a5);
//   4. when row t closes its cell ((t+1) % s == 0), writes the cell's kbar
//      and a_c, bit-identical to the prefill's cell summaries, and queues it.
// A step runs on a cluster of 8 CTAs of 256 threads per (batch, head), so
// that a head's window and cells are read through 8 SMs: each CTA stages the
// pool's summaries (a bulk asynchronous copy) and takes the same list, score
// and top-K decisions; CTA c reads the window's keys 64c .. 64c + 63 and the
// c-th selected cell, and the partial softmax results meet in CTA 0's shared
// memory, which writes the output and the state.
//
// Angles: RoPE enters the window as q_t . R(j - t) k_j.  cos / sin of o*theta_i
// for o = 64a + r (r < 64, a < 16) are two tables built once with the state
// (fp64 reduction, fp32 sincospi) and joined by the angle-sum identity.
#include "cell_summary.cuh"
#include "fs_common.cuh"
#include "fs_internal.h"
#include "tc05.cuh"

#include <cooperative_groups.h>

namespace cg = cooperative_groups;

namespace fs {

DecodeLayout decode_layout(int w, int P, int W, int K) {
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  DecodeLayout L;
  L.w = w;
  L.P = P;
  L.W = W;
  L.K = K;
  L.pend = kBq / kS;
  L.nslots = P + W + L.pend + 1;
  size_t off = 0;
  L.hdr = off;
  off = up(off + kDecodeHeaderInts * 4);
  L.slot_cell = off;
  off = up(off + (size_t)(L.nslots + 3) / 4 * 16);
  L.slot_amax = off;
  off = up(off + (size_t)(L.nslots + 3) / 4 * 16);
  L.slot_kbar = off;
  off = up(off + (size_t)L.nslots * kD * 4);
  L.slot_k = off;
  off = up(off + (size_t)L.nslots * kS * kD * 2);
  L.slot_v = off;
  off = up(off + (size_t)L.nslots * kS * kD * 2);
  L.ring_k = off;  // rotated by absolute position, fp32
  off = up(off + (size_t)w * kD * 4);
  L.ring_v = off;
  off = up(off + (size_t)w * kD * 2);
  L.head_bytes = off;
  L.tab = 256;  // after the error word's 256-byte header: theta_i / pi (fp64)
  L.global_bytes = up(L.tab + (size_t)(kD / 2) * 8);
  return L;
}

namespace {

constexpr int kThreads = 256;
constexpr int kCluster = 8;                    // CTAs per (batch, head)
constexpr int kWinPerCta = 512 / kCluster;     // window keys per CTA (w <= 512): 8 per warp
static_assert(kWinPerCta == 8 * (kThreads / 32), "eight window keys per warp");
static_assert(kS * kD * 2 == 16 * kThreads, "one 16-byte piece of a cell per thread");
static_assert(kMaxK <= kCluster, "one selected cell per CTA");
constexpr int kMaxSlots = kMaxP + 8 + kBq / kS + 1;
// header ints of one head: counts, then the lists
enum { kHT = 0, kHRecent = 1, kHTop = 2, kHPend = 3, kHOpen = 4, kHFree = 5 };
// the recent list briefly holds W + Bq/s cells at a block start, before the
// leavers move on
constexpr int kLRecent = 8, kLTop = kLRecent + 8 + kBq / kS, kLPend = kLTop + kMaxP,
              kLFree = kLPend + kBq / kS;
static_assert(kLFree + kMaxSlots <= kDecodeHeaderInts, "decode header too small");

struct StepParams {
  const uint16_t *q_t, *k_t, *v_t;  // [BH, d] bf16
  unsigned char *state;             // global part, then one head after another
  const float *lambda, *sigma, *mix;
  DecodeLayout L;
  int H, t;
  float rms_eps;
  float *out;                       // [BH, d] f32
  int32_t *sel_out;                 // [BH, K] (nullable)
};

__device__ __forceinline__ float bf16f(uint16_t x) { return __uint_as_float((uint32_t)x << 16); }

// (cos, sin) of pos * theta_i, th_pi = theta_i / pi: the product and its
// reduction modulo 2 in fp64 (exact to about 2^-29 at pos < 2^24), then the
// fp32 sine and cosine of pi times the reduced value
__device__ __forceinline__ float2 angle_cs(double th_pi, int pos) {
  const double x = (double)pos * th_pi;
  const double red = x - 2.0 * floor(0.5 * x);
  float sn, cs;
  sincospif((float)red, &sn, &cs);
  return make_float2(cs, sn);
}

// R(angles) on the pairs (i, i + d/2) of x, i < d/2: (x cos - y sin, x sin + y cos)
__device__ __forceinline__ void rotate_pair(float x0, float x1, float2 cs, float &y0, float &y1) {
  y0 = fmaf(x0, cs.x, -x1 * cs.y);
  y1 = fmaf(x0, cs.y, x1 * cs.x);
}

__device__ __forceinline__ bool ranks_before(float a, int c, float a2, int c2) {
  return a > a2 || (a == a2 && c < c2);
}

// sum_i wgt[i] * v(row_of(i)) for i < n, rows in shared memory (64 bf16 each):
// warp w takes i = w, w+8, ...; lane l owns dims 2l, 2l+1; the eight warp
// partials go to part[w] for the caller to add up.
template <typename RowOf>
__device__ __forceinline__ void weighted_rows(const float *wgt, int n, RowOf row_of,
                                              float2 (*part)[kD / 2]) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float ax = 0.f, ay = 0.f;
#pragma unroll 4
  for (int i = warp; i < n; i += kThreads / 32) {
    const uint32_t x = reinterpret_cast<const uint32_t *>(row_of(i))[lane];
    const float wv = wgt[i];
    ax = fmaf(wv, bf16_lo(x), ax);
    ay = fmaf(wv, bf16_hi(x), ay);
  }
  part[warp][lane] = make_float2(ax, ay);
}

__device__ __forceinline__ float sum_parts(const float2 (*part)[kD / 2], int dim) {
  float o = 0.f;
#pragma unroll
  for (int w8 = 0; w8 < kThreads / 32; ++w8) {
    const float2 pp = part[w8][dim >> 1];
    o += (dim & 1) ? pp.y : pp.x;
  }
  return o;
}

// One step, run by a cluster of kCluster CTAs per (batch, head).  Every CTA
// takes the same decisions from the same state (the lists at a block start,
// the pool's scores and the top K), so they need not talk until the end;
// CTA c then attends over its 64 of the window's keys and over the c-th
// selected cell, and hands its partial softmax (maximum, sum, weighted
// values) of each branch to CTA 0, which adds them up, writes the output and
// alone writes the state.
__global__ void __launch_bounds__(kThreads) k6_decode_kernel(const StepParams p) {
  extern __shared__ __align__(1024) unsigned char dsm[];
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  const DecodeLayout &L = p.L;
  // dynamic shared memory: slot summaries, then this CTA's cell rows
  float *s_kbar = reinterpret_cast<float *>(dsm);
  float *s_amax = s_kbar + (size_t)L.nslots * kD;
  int *s_cell = reinterpret_cast<int *>(s_amax + (L.nslots + 3) / 4 * 4);
  unsigned char *s_ck = reinterpret_cast<unsigned char *>(s_cell + (L.nslots + 3) / 4 * 4);
  unsigned char *s_cv = s_ck + (size_t)kS * kD * 2;

  __shared__ __align__(8) uint64_t barA;
  __shared__ int s_hdr[kDecodeHeaderInts];
  __shared__ float s_q[kD], s_k[kD];
  // R(t) q_t, R(t) k_t (the new key is read as float4: 16-byte aligned)
  __shared__ __align__(16) float s_qr[kD], s_kr[kD];
  __shared__ int s_pool[kMaxP + 8];
  __shared__ float s_u[kMaxP + 8];
  __shared__ int s_rank[3][kMaxP + 8];
  __shared__ int s_pc[kMaxP + 8];
  __shared__ int s_sel[kMaxK];
  __shared__ float s_w[kWinPerCta];
  __shared__ float2 s_part[kThreads / 32][kD / 2];
  __shared__ float s_wm[kThreads / 32], s_wl[kThreads / 32];  // per warp: window max, sum
  __shared__ int s_ok;
  // CTA 0 only: every CTA's partials, written there by the CTA itself
  __shared__ float s_cm[2][kCluster], s_cl[2][kCluster];  // [branch][CTA]: max, sum
  __shared__ float s_co[2][kCluster][kD];                  // weighted values
  __shared__ int s_cok[kCluster];

  const int bh = blockIdx.x / kCluster, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = bh % p.H;
  int *err = reinterpret_cast<int *>(p.state);
  const double *th_pi = reinterpret_cast<const double *>(p.state + L.tab);
  unsigned char *hs = p.state + L.global_bytes + (size_t)bh * L.head_bytes;
  int *g_hdr = reinterpret_cast<int *>(hs + L.hdr);
  int *g_cell = reinterpret_cast<int *>(hs + L.slot_cell);
  float *g_amax = reinterpret_cast<float *>(hs + L.slot_amax);
  float *g_kbar = reinterpret_cast<float *>(hs + L.slot_kbar);
  uint16_t *g_sk = reinterpret_cast<uint16_t *>(hs + L.slot_k);
  uint16_t *g_sv = reinterpret_cast<uint16_t *>(hs + L.slot_v);
  float *g_rk = reinterpret_cast<float *>(hs + L.ring_k);
  uint16_t *g_rv = reinterpret_cast<uint16_t *>(hs + L.ring_v);

  // ---- the window's ring rows for this warp (they do not depend on the
  // selection): loads issued now, used after the pool is scored.  Keys i in
  // [kWinPerCta * rank + 8 * warp, + 8), four lanes per key (a contiguous
  // 64-byte slice of R(j) k_j, fp32), and lane l's two dimensions of each
  // key's value.  The newest key and value (j = t) come from the step's
  // inputs: CTA 0 writes them into the ring only at the end.
  const int t = p.t;
  const int j0 = max(0, t - L.w + 1), nwin_all = t - j0 + 1;
  const int r0 = j0 % L.w;  // ring row of key i: r0 + i, less w past the end
  const auto ring_row = [&](int i) { const int rr = r0 + i; return rr >= L.w ? rr - L.w : rr; };
  const int ibase = kWinPerCta * (int)rank + 8 * warp;  // the warp's first key
  float4 xs[4];
  uint32_t xv[8];
  {
    const int i = ibase + (lane >> 2);
    if (i < nwin_all - 1) {
      const float4 *kr =
          reinterpret_cast<const float4 *>(g_rk + (size_t)ring_row(i) * kD + 16 * (lane & 3));
#pragma unroll
      for (int c = 0; c < 4; ++c) xs[c] = kr[c];
    }
#pragma unroll
    for (int k8 = 0; k8 < 8; ++k8) {
      const int ik = ibase + k8;
      xv[k8] = ik < nwin_all - 1
          ? reinterpret_cast<const uint32_t *>(g_rv + (size_t)ring_row(ik) * kD)[lane]
          : ik == nwin_all - 1 ? reinterpret_cast<const uint32_t *>(p.v_t + (size_t)bh * kD)[lane]
                               : 0u;
    }
  }

  // ---- stage the slot summaries: one bulk copy
  if (tid == 0) {
    tc::mbar_init(&barA, 1);
    tc::mbar_fence_init();
    const uint32_t sums = (uint32_t)L.nslots * kD * 4;
    const uint32_t small = (uint32_t)(L.nslots + 3) / 4 * 16;
    tc::mbar_arrive_expect_tx(&barA, sums + 2 * small);
    tc::bulk_load(s_kbar, g_kbar, sums, &barA);
    tc::bulk_load(s_amax, g_amax, small, &barA);
    tc::bulk_load(s_cell, g_cell, small, &barA);
  }
  for (int i = tid; i < kDecodeHeaderInts; i += kThreads) s_hdr[i] = g_hdr[i];
  if (tid < kD) {
    s_q[tid] = bf16f(p.q_t[(size_t)bh * kD + tid]);
    s_k[tid] = bf16f(p.k_t[(size_t)bh * kD + tid]);
  }
  __syncthreads();
  // the query and the new key rotated by the absolute position t: the window
  // score R(t) q . R(j) k equals q . R(j - t) k
  if (tid < kD / 2) {
    const float2 cs = angle_cs(th_pi[tid], t);
    rotate_pair(s_q[tid], s_q[tid + kD / 2], cs, s_qr[tid], s_qr[tid + kD / 2]);
    rotate_pair(s_k[tid], s_k[tid + kD / 2], cs, s_kr[tid], s_kr[tid + kD / 2]);
  }
  // the state must be at position t: the same answer in every CTA, so they
  // all leave here together (the copy is awaited first)
  const bool in_step = s_hdr[kHT] == t;
  const bool staged = tc::mbar_wait(&barA, 0, err);
  if (!in_step) {
    if (tid == 0 && rank == 0) tc::report_error(err, FS_ERR_STATE);
    if (!staged) tc::mbar_wait(&barA, 0, nullptr);  // no copy in flight at exit
    return;
  }
  // every CTA of the cluster has started once all have arrived here: awaited
  // before the first write into CTA 0's shared memory
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  // a copy that did not land is this CTA's alone: it goes on to the meeting
  // with the others and flags its partials as missing
  if (tid == 0) s_ok = staged;
  __syncthreads();
  const bool ok = s_ok;

  // ---- 1. block start: pending cells become recent, leavers join the top list
  if (tid == 0 && ok) {
    int *recent = s_hdr + kLRecent, *top = s_hdr + kLTop, *pend = s_hdr + kLPend;
    int *freel = s_hdr + kLFree;
    if (t > 0 && t % kBq == 0) {
      for (int k = 0; k < s_hdr[kHPend]; ++k) recent[s_hdr[kHRecent]++] = pend[k];
      s_hdr[kHPend] = 0;
      while (s_hdr[kHRecent] > L.W) {
        const int slot = recent[0];
        for (int k = 1; k < s_hdr[kHRecent]; ++k) recent[k - 1] = recent[k];
        --s_hdr[kHRecent];
        // insert by (a desc, c asc) into the ranked older list of at most P
        const float a = s_amax[slot];
        const int c = s_cell[slot];
        int n = s_hdr[kHTop], pos = n;
        while (pos > 0 && ranks_before(a, c, s_amax[top[pos - 1]], s_cell[top[pos - 1]])) --pos;
        if (pos >= L.P) {
          freel[s_hdr[kHFree]++] = slot;  // ranks past the top P: dropped
        } else {
          int dropped = -1;
          if (n == L.P) dropped = top[--n];  // the list was full: its last cell leaves
          for (int q = n; q > pos; --q) top[q] = top[q - 1];
          top[pos] = slot;
          s_hdr[kHTop] = n + 1;
          if (dropped >= 0) freel[s_hdr[kHFree]++] = dropped;
        }
      }
    }
    // 2. a new cell opens (a slot is always free: at most W + P + Bq/s cells
    // are held when one opens, of P + W + Bq/s + 1 slots)
    if (t % kS == 0) {
      if (s_hdr[kHFree] > 0) {
        s_hdr[kHOpen] = freel[--s_hdr[kHFree]];
      } else {
        s_hdr[kHOpen] = -1;
        if (rank == 0) tc::report_error(err, FS_ERR_STATE);
      }
    }
    s_ok = s_hdr[kHOpen] >= 0;
  }
  __syncthreads();
  // a state that lost track of its slots is left as it was (the same answer
  // in every CTA whose copy landed)
  const bool go = ok && s_ok;
  const int open = s_hdr[kHOpen];

  // ---- 3a. score the pool: u = q . kbar_c + lambda * a_c * erf(sigma (t - p_c) / s)
  const int nrec = go ? s_hdr[kHRecent] : 0, nc = go ? nrec + s_hdr[kHTop] : 0;
  if (tid < nc) {
    s_pool[tid] = tid < nrec ? s_hdr[kLRecent + tid] : s_hdr[kLTop + tid - nrec];
    s_pc[tid] = s_cell[s_pool[tid]];  // the candidate's cell id
  }
  __syncthreads();
  const float lam = p.lambda[h], sig = p.sigma[h];
  // four lanes per candidate (16 dimensions each), eight candidates per warp
  for (int i0 = warp * 8; i0 < nc; i0 += kThreads / 4) {
    const int i = i0 + (lane >> 2), sub = lane & 3;
    float dot = 0.f;
    int slot = 0;
    if (i < nc) {
      slot = s_pool[i];
      const float4 *kb = reinterpret_cast<const float4 *>(s_kbar + (size_t)slot * kD + 16 * sub);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float4 x = kb[c];
        const float *qq = s_q + 16 * sub + 4 * c;
        dot = fmaf(qq[0], x.x, fmaf(qq[1], x.y, fmaf(qq[2], x.z, fmaf(qq[3], x.w, dot))));
      }
    }
    dot += __shfl_xor_sync(0xffffffffu, dot, 1);
    dot += __shfl_xor_sync(0xffffffffu, dot, 2);
    if (i < nc && sub == 0) {
      const float pc = (float)(s_cell[slot] * kS) + 0.5f * kS;
      s_u[i] = dot + lam * s_amax[slot] * erff(sig * ((float)t - pc) / kS);
    }
  }
  if (tid < kMaxK) s_sel[tid] = -1;
  __syncthreads();
  // top K by (u desc, c asc): rank of each candidate by counting, the
  // comparisons split in three ranges of j
  const int third = (nc + 2) / 3;
  if (tid < 3 * nc) {
    const int i = tid % nc, part = tid / nc;
    const float u = s_u[i];
    const int c = s_pc[i];
    int rank_i = 0;
    for (int j = part * third; j < min(nc, (part + 1) * third); ++j)
      rank_i += ranks_before(s_u[j], s_pc[j], u, c);
    s_rank[part][i] = rank_i;
  }
  __syncthreads();
  if (tid < nc) {
    const int rank_i = s_rank[0][tid] + s_rank[1][tid] + s_rank[2][tid];
    if (rank_i < L.K) s_sel[rank_i] = s_pool[tid];
  }
  __syncthreads();
  int nsel = 0;
  for (int k = 0; k < L.K; ++k) nsel += s_sel[k] >= 0;
  if (rank == 0 && go && tid < L.K && p.sel_out)
    p.sel_out[(size_t)bh * L.K + tid] = s_sel[tid] >= 0 ? s_cell[s_sel[tid]] : -1;
  // this CTA's selected cell (the rank-th of the K best, if any): its rows,
  // loaded now and stored after the window branch
  const int my_slot = (int)rank < nsel ? s_sel[rank] : -1;
  uint4 ck_row = make_uint4(0, 0, 0, 0), cv_row = ck_row;
  if (my_slot >= 0) {
    ck_row = reinterpret_cast<const uint4 *>(g_sk + (size_t)my_slot * kS * kD)[tid];
    cv_row = reinterpret_cast<const uint4 *>(g_sv + (size_t)my_slot * kS * kD)[tid];
  }

  // ---- 3c. RoPE window over rows [t - w + 1, t] (a5): the warp's eight keys
  // (loaded at the start) against R(t) q_t
  const int nwin = go ? nwin_all : 0;
  float dot = -INFINITY;
  {
    const int i = ibase + (lane >> 2);
    if (i < nwin) {
      if (i == nwin - 1) {
#pragma unroll
        for (int c = 0; c < 4; ++c) xs[c] = reinterpret_cast<const float4 *>(s_kr + 16 * (lane & 3))[c];
      }
      const float *qq = s_qr + 16 * (lane & 3);
      float d = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c)
        d = fmaf(qq[4 * c], xs[c].x, fmaf(qq[4 * c + 1], xs[c].y,
            fmaf(qq[4 * c + 2], xs[c].z, fmaf(qq[4 * c + 3], xs[c].w, d))));
      dot = d;
    }
    dot += __shfl_xor_sync(0xffffffffu, dot, 1);
    dot += __shfl_xor_sync(0xffffffffu, dot, 2);
    dot = i < nwin ? dot * 0.125f : -INFINITY;
  }
  // the warp's maximum and sum (the four lanes of a key hold the same value:
  // reduce over the keys only)
  float mw = dot;
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, o));
  const float wgt = mw == -INFINITY ? 0.f : __expf(dot - mw);
  float lw = (lane & 3) == 0 ? wgt : 0.f;
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
  // P.V over the warp's eight keys (key k8's weight sits in lane 4 * k8):
  // lane l owns dimensions 2l, 2l + 1
  float ax = 0.f, ay = 0.f;
#pragma unroll
  for (int k8 = 0; k8 < 8; ++k8) {
    const float wv = __shfl_sync(0xffffffffu, wgt, 4 * k8);
    if (ibase + k8 < nwin) {
      ax = fmaf(wv, bf16_lo(xv[k8]), ax);
      ay = fmaf(wv, bf16_hi(xv[k8]), ay);
    }
  }
  s_part[warp][lane] = make_float2(ax, ay);
  if (lane == 0) {
    s_wm[warp] = mw;
    s_wl[warp] = lw;
  }
  // this CTA's cell rows into shared memory
  if (my_slot >= 0) {
    reinterpret_cast<uint4 *>(s_ck)[tid] = ck_row;
    reinterpret_cast<uint4 *>(s_cv)[tid] = cv_row;
  }
  __syncthreads();
  // the CTA's window partial: maximum, sum and weighted values over its keys
  float cm_w = s_wm[0];
#pragma unroll
  for (int w8 = 1; w8 < kThreads / 32; ++w8) cm_w = fmaxf(cm_w, s_wm[w8]);
  float cl_w = 0.f, co_w = 0.f;
  if (tid < kD) {
#pragma unroll
    for (int w8 = 0; w8 < kThreads / 32; ++w8) {
      const float sc = s_wm[w8] == -INFINITY ? 0.f : __expf(s_wm[w8] - cm_w);
      const float2 pp = s_part[w8][tid >> 1];
      cl_w = fmaf(s_wl[w8], sc, cl_w);
      co_w = fmaf((tid & 1) ? pp.y : pp.x, sc, co_w);
    }
  }
  __syncthreads();  // s_part is reused below

  // ---- 3b. NoPE readout over this CTA's cell (a4): warp 0, one lane per
  // token, takes the logits, their maximum and sum; every warp then adds up
  // weighted value rows
  float cm_l = -INFINITY, cl_l = 0.f;
  if (warp == 0) {
    float lg = -INFINITY;
    if (my_slot >= 0) {
      const uint4 *kr = reinterpret_cast<const uint4 *>(s_ck + (size_t)lane * kD * 2);
      float d = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 x = kr[c];
        const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          d = fmaf(s_q[8 * c + 2 * j], bf16_lo(wv[j]), d);
          d = fmaf(s_q[8 * c + 2 * j + 1], bf16_hi(wv[j]), d);
        }
      }
      lg = d * 0.125f;
    }
    cm_l = lg;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cm_l = fmaxf(cm_l, __shfl_xor_sync(0xffffffffu, cm_l, o));
    const float pl = my_slot >= 0 ? __expf(lg - cm_l) : 0.f;
    s_w[lane] = pl;
    cl_l = warp_sum(pl);
  }
  __syncthreads();
  weighted_rows(s_w, my_slot >= 0 ? kS : 0, [&](int i) { return s_cv + (size_t)i * kD * 2; }, s_part);
  __syncthreads();
  const float co_l = tid < kD ? sum_parts(s_part, tid) : 0.f;

  // ---- partials to CTA 0, one meeting of the cluster
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  {
    float(*r_cm)[kCluster] = cluster.map_shared_rank(s_cm, 0);
    float(*r_cl)[kCluster] = cluster.map_shared_rank(s_cl, 0);
    float(*r_co)[kCluster][kD] = cluster.map_shared_rank(s_co, 0);
    int *r_cok = cluster.map_shared_rank(s_cok, 0);
    if (tid == 0) {
      r_cm[0][rank] = cm_w;
      r_cl[0][rank] = cl_w;
      r_cm[1][rank] = my_slot >= 0 ? cm_l : -INFINITY;
      r_cl[1][rank] = my_slot >= 0 ? cl_l : 0.f;
      r_cok[rank] = go ? 1 : (ok ? 2 : 0);  // 2: a state that lost its slots
    }
    if (tid < kD) {
      r_co[0][rank][tid] = co_w;
      r_co[1][rank][tid] = my_slot >= 0 ? co_l : 0.f;
    }
  }
  cluster.sync();
  if (!ok) tc::mbar_wait(&barA, 0, nullptr);  // no copy in flight at exit
  if (rank != 0) return;

  // ---- CTA 0: the totals, the output, then the state (only if every CTA
  // worked from a staged state; otherwise the state is left as it was)
  bool all_go = true;
#pragma unroll
  for (int c = 0; c < kCluster; ++c) all_go = all_go && s_cok[c] == 1;
  if (!all_go) return;
  // warp 0: lane l takes dimensions 2l, 2l + 1 of both branches; the CTAs'
  // partials are added in CTA order
  if (warp == 0) {
    // each CTA's scale exp(m_c - M) per branch, once; then the sums
    float sc[2][kCluster], lt[2];
#pragma unroll
    for (int br = 0; br < 2; ++br) {
      float m = s_cm[br][0];
#pragma unroll
      for (int c = 1; c < kCluster; ++c) m = fmaxf(m, s_cm[br][c]);
      float l = 0.f;
#pragma unroll
      for (int c = 0; c < kCluster; ++c) {
        sc[br][c] = s_cm[br][c] == -INFINITY ? 0.f : __expf(s_cm[br][c] - m);
        l = fmaf(s_cl[br][c], sc[br][c], l);
      }
      lt[br] = l;
    }
    float owin[2], olong[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int dim = 2 * lane + e;
      float ow = 0.f, ol = 0.f;
#pragma unroll
      for (int c = 0; c < kCluster; ++c) {
        ow = fmaf(s_co[0][c][dim], sc[0][c], ow);
        ol = fmaf(s_co[1][c][dim], sc[1][c], ol);
      }
      owin[e] = ow / lt[0];
      olong[e] = nsel > 0 ? ol / lt[1] : 0.f;
    }
    const float ss = warp_sum(olong[0] * olong[0] + olong[1] * olong[1]);
    const float rms_scale = nsel > 0 ? rsqrtf(ss / kD + p.rms_eps) : 0.f;
    const float mh = p.mix[h];
    *reinterpret_cast<float2 *>(p.out + (size_t)bh * kD + 2 * lane) =
        make_float2(owin[0] + mh * olong[0] * rms_scale, owin[1] + mh * olong[1] * rms_scale);
  }

  // ---- 2. the new token: ring row t mod w (the rotated key, fp32, and the
  // value) and the open slot's row t mod s
  if (tid < 8) {
    const uint4 kv = reinterpret_cast<const uint4 *>(p.k_t + (size_t)bh * kD)[tid];
    reinterpret_cast<uint4 *>(g_sk + (size_t)open * kS * kD + (size_t)(t % kS) * kD)[tid] = kv;
  } else if (tid < 16) {
    const int c = tid - 8;
    const uint4 vv = reinterpret_cast<const uint4 *>(p.v_t + (size_t)bh * kD)[c];
    reinterpret_cast<uint4 *>(g_rv + (size_t)(t % L.w) * kD)[c] = vv;
    reinterpret_cast<uint4 *>(g_sv + (size_t)open * kS * kD + (size_t)(t % kS) * kD)[c] = vv;
  } else if (tid >= 32 && tid < 48) {
    const int c = tid - 32;
    reinterpret_cast<float4 *>(g_rk + (size_t)(t % L.w) * kD)[c] =
        make_float4(s_kr[4 * c], s_kr[4 * c + 1], s_kr[4 * c + 2], s_kr[4 * c + 3]);
  }
  __syncthreads();  // the open slot's new row is read back below

  // ---- 4. row t closes its cell: summary, as the prefill computes it; the
  // cell waits in the pending list for the next block start
  if ((t + 1) % kS == 0 && warp == 0) {
    float x[8][8];
    load_cell_bf16<false>(reinterpret_cast<const uint4 *>(g_sk + (size_t)open * kS * kD), lane, x);
    cell_summary_warp(x, lane, g_kbar + (size_t)open * kD, g_amax + open);
    if (lane == 0) g_cell[open] = t / kS;
  }
  if (tid == 0) {
    if ((t + 1) % kS == 0) {
      s_hdr[kLPend + s_hdr[kHPend]++] = open;
      s_hdr[kHOpen] = -1;
    }
    s_hdr[kHT] = t + 1;
  }
  __syncthreads();
  for (int i = tid; i < kDecodeHeaderInts; i += kThreads) g_hdr[i] = s_hdr[i];
}

// Build the state after the first N0 tokens from the prefix's keys, values,
// cell summaries and the pool of block (N0-1)/Bq: recent then ranked older
// cells in slots 0.., the pending cells after them, the open cell's rows, the
// ring, the free list.  CTA 0 also writes the angle tables.
__global__ void __launch_bounds__(kThreads) k6_init_kernel(
    const uint16_t *__restrict__ k, const uint16_t *__restrict__ v, const float *__restrict__ kbar,
    const float *__restrict__ amax, const int32_t *__restrict__ pool,
    const int32_t *__restrict__ pool_count, int N, int N0, double rope_base, DecodeLayout L,
    unsigned char *state) {
  __shared__ int s_hdr[kDecodeHeaderInts];
  __shared__ int s_slot_cell[kMaxSlots];
  const int bh = blockIdx.x, tid = threadIdx.x;
  const int C = N / kS, nblk = N / kBq, cap = L.P + L.W;
  unsigned char *hs = state + L.global_bytes + (size_t)bh * L.head_bytes;
  if (bh == 0) {
    // theta_i / pi, fp64, for the steps' rotations
    if (tid == 0) *reinterpret_cast<int *>(state) = 0;
    double *th = reinterpret_cast<double *>(state + L.tab);
    if (tid < kD / 2) th[tid] = pow(rope_base, -2.0 * tid / kD) / 3.14159265358979323846;
  }
  if (tid == 0) {
    for (int i = 0; i < kDecodeHeaderInts; ++i) s_hdr[i] = 0;
    for (int i = 0; i < kMaxSlots; ++i) s_slot_cell[i] = -1;
    int nslot = 0;
    s_hdr[kHT] = N0;
    s_hdr[kHOpen] = -1;
    if (N0 > 0) {
      const int beta = (N0 - 1) / kBq, A = beta * (kBq / kS);
      const int cnt = min(max(pool_count[(size_t)bh * nblk + beta], 0), cap);
      const int nrec = min(L.W, A);
      const int32_t *row = pool + ((size_t)bh * nblk + beta) * cap;
      for (int i = 0; i < cnt; ++i) {
        s_slot_cell[nslot] = row[i];
        if (i < nrec)
          s_hdr[kLRecent + s_hdr[kHRecent]++] = nslot;
        else
          s_hdr[kLTop + s_hdr[kHTop]++] = nslot;
        ++nslot;
      }
      for (int c = beta * (kBq / kS); c < N0 / kS; ++c) {  // closed, not yet available
        s_slot_cell[nslot] = c;
        s_hdr[kLPend + s_hdr[kHPend]++] = nslot++;
      }
      if (N0 % kS) {  // the open cell
        s_slot_cell[nslot] = N0 / kS;
        s_hdr[kHOpen] = nslot++;
      }
    }
    // free slots, handed out from the end of the list
    for (int i = L.nslots - 1; i >= nslot; --i) s_hdr[kLFree + s_hdr[kHFree]++] = i;
  }
  __syncthreads();
  int *g_hdr = reinterpret_cast<int *>(hs + L.hdr);
  int *g_cell = reinterpret_cast<int *>(hs + L.slot_cell);
  float *g_amax = reinterpret_cast<float *>(hs + L.slot_amax);
  float *g_kbar = reinterpret_cast<float *>(hs + L.slot_kbar);
  uint4 *g_sk = reinterpret_cast<uint4 *>(hs + L.slot_k);
  uint4 *g_sv = reinterpret_cast<uint4 *>(hs + L.slot_v);
  for (int i = tid; i < kDecodeHeaderInts; i += kThreads) g_hdr[i] = s_hdr[i];
  const size_t head = (size_t)bh * N;
  const int full_cells = N0 / kS;
  for (int sl = 0; sl < L.nslots; ++sl) {
    const int c = s_slot_cell[sl];
    if (tid == 0) {
      const bool closed = c >= 0 && c < full_cells;
      g_cell[sl] = closed ? c : -1;
      g_amax[sl] = closed ? amax[(size_t)bh * C + c] : 0.f;
    }
    if (c < 0) continue;
    const bool closed = c < full_cells;
    if (closed && tid < kD) g_kbar[(size_t)sl * kD + tid] = kbar[((size_t)bh * C + c) * kD + tid];
    // the cell's rows below N0 (all of them for a closed cell)
    const int rows = min(kS, N0 - c * kS);
    for (int e = tid; e < rows * 8; e += kThreads) {
      const size_t src = (head + (size_t)c * kS) * 8 + e;
      g_sk[(size_t)sl * kS * 8 + e] = reinterpret_cast<const uint4 *>(k)[src];
      g_sv[(size_t)sl * kS * 8 + e] = reinterpret_cast<const uint4 *>(v)[src];
    }
  }
  // the ring: rows [max(0, N0 - w), N0) at j mod w
  float *g_rk = reinterpret_cast<float *>(hs + L.ring_k);
  uint4 *g_rv = reinterpret_cast<uint4 *>(hs + L.ring_v);
  const int r0 = max(0, N0 - L.w);
  for (int e = tid; e < (N0 - r0) * 8; e += kThreads) {
    const int j = r0 + e / 8;
    g_rv[(size_t)(j % L.w) * 8 + e % 8] = reinterpret_cast<const uint4 *>(v)[(head + j) * 8 + e % 8];
  }
  // keys rotated by their absolute position, fp32
  for (int e = tid; e < (N0 - r0) * (kD / 2); e += kThreads) {
    const int j = r0 + e / (kD / 2), i = e % (kD / 2);
    const double thp = pow(rope_base, -2.0 * i / kD) / 3.14159265358979323846;
    const double x = (double)j * thp;
    const double red = x - 2.0 * floor(0.5 * x);
    float sn, cs;
    sincospif((float)red, &sn, &cs);
    const float x0 = __uint_as_float((uint32_t)k[(head + j) * kD + i] << 16);
    const float x1 = __uint_as_float((uint32_t)k[(head + j) * kD + i + kD / 2] << 16);
    float *dst = g_rk + (size_t)(j % L.w) * kD;
    dst[i] = fmaf(x0, cs, -x1 * sn);
    dst[i + kD / 2] = fmaf(x0, sn, x1 * cs);
  }
}

}  // namespace

size_t decode_smem_bytes(const DecodeLayout &L) {
  return (size_t)L.nslots * kD * 4 + 2 * (size_t)(L.nslots + 3) / 4 * 16 + 2 * (size_t)kS * kD * 2;
}

cudaError_t launch_decode_init(const void *k, const void *v, const float *kbar, const float *amax,
                               const int32_t *pool, const int32_t *pool_count, int BH, int N,
                               int N0, float rope_base, const DecodeLayout &L, void *state,
                               cudaStream_t st) {
  k6_init_kernel<<<BH, kThreads, 0, st>>>(
      static_cast<const uint16_t *>(k), static_cast<const uint16_t *>(v), kbar, amax, pool,
      pool_count, N, N0, (double)rope_base, L, static_cast<unsigned char *>(state));
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t st) {
  StepParams p;
  p.q_t = static_cast<const uint16_t *>(a.q_t);
  p.k_t = static_cast<const uint16_t *>(a.k_t);
  p.v_t = static_cast<const uint16_t *>(a.v_t);
  p.state = static_cast<unsigned char *>(a.state);
  p.lambda = a.lambda;
  p.sigma = a.sigma;
  p.mix = a.mix;
  p.L = a.L;
  p.H = a.H;
  p.t = a.t;
  p.rms_eps = a.rms_eps;
  p.out = a.out;
  p.sel_out = a.sel_out;
  const size_t smem = decode_smem_bytes(a.L);
  cudaError_t e =
      cudaFuncSetAttribute(k6_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(a.batch * a.H * kCluster));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k6_decode_kernel, p);
}

}  // namespace fs
