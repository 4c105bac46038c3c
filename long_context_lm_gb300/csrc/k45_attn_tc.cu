// k45_attn_tc.cu -- both attention branches of FS-L on the 5th-generation
// tensor cores (tcgen05 + TMEM), with the branch mix in the epilogue.
//
// FreeSolo (paper.rainbus.top summary, 方法步骤详情 ② window branch, ⑥ "选中
// token 上做 NoPE softmax 再 RMSNorm，与局部分支相加", 前置知识 RoPE / NoPE;
// ai.info summary, "Methodology in Plain English"):
//     o_win[n]  = softmax_j((R(n) q_n . R(j) k_j) / sqrt(d)) v_j,  j in [n-w+1, n]
//     o_long[n] = RMSNorm(softmax_t(q_n . k_t / sqrt(d)) v_t),     t in the K
//                 selected cells of n (no rotation), 0 if none
//     out[n]    = o_win[n] + mix_h * o_long[n].
//
// Persistent kernel: one CTA per SM walks 128-query tiles (q-tiles).  Each
// q-tile is a list of 128-key tiles: first the window tiles covering
// [b - w + 1, b + 127], then the "long" tiles, each gathering four of the
// cells that any query of the tile selected (their union, built per q-tile).
// Sixteen warps with fixed roles and mbarrier hand-offs; every counter runs
// across q-tiles, so producers start the next q-tile while the softmax
// finishes the current one:
//   warps 0-7   softmax: warp w owns TMEM lanes / query rows 32*(w%4).. and
//               key columns 64*(w/4).. of each key tile; the two warps of a
//               row block exchange row maxima through shared memory (one
//               bounded mbarrier phase per tile)
//   warp  8     TMEM allocation; lane 0 issues the S = Q.K^T MMAs
//   warp  9     lane 0 issues the P.V MMAs (one issuing thread sustains about
//               one tcgen05.mma per ~100 cycles, hence two issuers)
//   warp  10    lane 0: TMA producer (contiguous window tiles; gathered cells)
//   warp  11    builds the union of the q-tile's selected cells
//   warps 12-15 stage the query tile: raw (long branch) and rotated (window);
//               then the epilogue of the previous q-tile (one thread per row)
// Window key tiles arrive already rotated (absolute positions, bf16 hi | lo)
// with fp16 values, from the preparation pass; the query tile is rotated
// here by the same absolute angles, so q_n . k_j carries R(n - j).
// TMEM: two 128-column score buffers S; the softmax overwrites each with
// its tile's probabilities (fp16 pairs, or bf16 hi / lo pairs for the long
// branch alone; the A operand of P.V) in place, so P is double-buffered with
// S.  Two accumulator sets (O_win, O_long; 64 columns each) alternate between
// q-tiles, so the epilogue of a q-tile has the whole next q-tile to run in,
// off the softmax and MMA paths.
//
// Precision.  Window: the rotated q and k (fp32, absolute angles from the
// angle table) are split into bf16 hi + lo halves and S takes three MMA
// chains (hi.hi + hi.lo + lo.hi): a single bf16 rounding of the rotated
// vectors exceeds the output tolerance on lognormal keys.  The window P.V
// product runs in fp16 (P below 2^14, V re-encoded exactly from bf16): with a
// lagging maximum the dominant probability is not exactly 1, and bf16's
// 8-bit significand on it alone reaches the tolerance on peaked rows.  Long
// branch: q and k are exact bf16, so S is one chain.  RMSNorm rescales the
// branch output, which amplifies the rounding of P: a plain bf16 P reaches
// about 5e-3 after the norm, fp16 P about 6e-4.  So next to the window
// branch (whose fp16 values exist) the long P is fp16 with one P.V chain;
// the long branch alone splits P into bf16 hi + lo (two chains) against the
// raw bf16 values.
#include <cuda.h>
#include <string.h>

#include "fs_common.cuh"
#include "fs_internal.h"
#include "tc05.cuh"

namespace fs {
namespace {

constexpr int kKT = 128;          // keys per tile
constexpr int kRing = 3;          // key / value ring depth
constexpr int kThreads = 512;
constexpr int kRotBase = 384;     // first query-staging thread (warps 12-15)
constexpr int kRotThreads = 128;  // one 64-element row each
constexpr int kT64Stride = 272;   // bytes per row of the r*theta table (padded: no bank conflicts)
constexpr int kMaxSel = kBq * kMaxK;

// shared-memory layout, offsets from a 1024-byte aligned base
constexpr uint32_t kOffQ = 0;                          // rotated query [hi 16 KB, lo 16 KB]
constexpr uint32_t kOffQR = 32768;                     // raw query 16 KB
constexpr uint32_t kOffK = 49152;                      // kRing x [hi 16 KB, lo 16 KB]
constexpr uint32_t kOffV = kOffK + kRing * 32768;      // kRing x 16 KB
constexpr uint32_t kOffT64 = kOffV + kRing * 16384;    // 64 rows x 272 B
constexpr uint32_t kOffUL = kOffT64 + 64 * kT64Stride; // union list: kMaxSel int32
constexpr uint32_t kOffRS = kOffUL + kMaxSel * 4;      // per row / pick: union slot, uint16
constexpr int kBW = 256;                               // union bitmap words (8192 cells per pass)
constexpr uint32_t kOffBM = kOffRS + kMaxSel * 2;      // union bitmap: kBW uint32
constexpr uint32_t kOffPW = kOffBM + kBW * 4;          // cells before each bitmap word: kBW uint16
constexpr uint32_t kSmemBytes = kOffPW + kBW * 2 + 1024;  // + alignment slack

// TMEM columns: S / P buffers at 0 and 128; accumulator sets at 256 and 384
// (O_win at +0, O_long at +64).  Inside a score buffer, key chunk c (32 keys)
// keeps its P in columns 32c..32c+15 (and, for a bf16 hi + lo long tile, P_lo
// in 32c+16..32c+31), so each softmax warp writes only the columns it has
// already read.
constexpr uint32_t kColS = 0, kColO = 256;
constexpr uint32_t kTmemCols = 512;
// The running maximum is raised only when a tile's maximum exceeds it by more
// than 2^kLazy (log2 units); below that, probabilities are taken against the
// old maximum and the accumulator is left alone (a raise rescales it, which
// waits for the previous P.V).  The bound is what the formats hold: fp16 P
// (values up to 2^14 < 65504); bf16 hi + lo long-branch P with fp32 sums and
// accumulators (2^30 leaves room for 128 keys times |v|).
constexpr float kLazyWin = 14.f, kLazyLong = 30.f;

__device__ __forceinline__ uint32_t p_col(int k) {  // P of key group k (16 keys)
  return 32 * (k >> 1) + 8 * (k & 1);
}

struct Barriers {
  uint64_t q_full, q_empty;
  uint64_t raw_full[kRing];  // TMA: key and value tile landed
  uint64_t k_empty[kRing];   // S MMAs of the tile done
  uint64_t v_empty[kRing];   // P.V MMAs of the tile done
  uint64_t s_full[2], s_free[2];  // s_free: the tile's P.V (last reader of S / P) done
  uint64_t p_full[2], pv_done;     // p_full per score buffer: the softmax may run a
                                  // tile ahead of the P.V issuer
  uint64_t o_done[2], o_free[2];  // per accumulator set
  uint64_t stats_full[2], stat_free[2];  // per q-tile parity: row sums published / read
  uint64_t pair[4];               // the two softmax warps of a row block meet here
  uint64_t u_full, u_free;   // union of the q-tile's cells built / consumed
  uint64_t g_full[4];        // the CTA's q-tile sequence: item i published in slot i % 4
  int g_ring[4];
  uint64_t fin[2];
  uint32_t tmem;
  int nu;                    // cells in the current union
  float2 stat[2][2][128];    // [q-tile parity][warp half][row]: (l_win, l_long) partial sums
  int item_nl[2];            // [q-tile parity]: long tiles of that q-tile
  float2 xch[2][2][128];     // row values the two softmax warps of a row block
                             // exchange: [exchange parity][warp half][row]
};

struct Params {
  const __nv_bfloat16 *q;
  const int32_t *sel;      // [BH, N, K] selected cells (long branch)
  const float *o_long_in;  // window-only mode: branch to mix in (nullable)
  const float *mix;
  const float2 *tab;       // (cos, sin) of r*theta_i (rows r < 64), 64*u*theta_i (row 64 + u)
  int H, N, w, K, nblk, nitems;
  int *sched;              // nullable: [0] next item ticket, [1] CTAs finished (zero at launch)
  long long *timeline;     // nullable: per CTA, global-timer ns at its start and at its end
  float rms_eps;
  size_t nrows;            // BH * N (first out-of-range key row: zero fill)
  float *out;
  int *err;
};

__device__ __forceinline__ bool wait_nth(uint64_t *bar, uint32_t k, int *err) {
  return tc::mbar_wait(bar, k & 1, err);
}

// The kernel is compiled once per configuration, so that each carries only
// the code of its own branches:
//   kLongOnly  the long branch alone, written as RMSNorm(o_long) (bf16 hi + lo
//              P against the raw bf16 values)
//   kWindow    the window branch, plus mix_h times a long-branch output read
//              from memory if one is given
//   kFused     both branches; the long-branch P in fp16 against the fp16
//              values the window branch uses
enum Mode { kLongOnly = 0, kWindow = 1, kFused = 2 };
template <int M>
struct Flags {
  static constexpr bool window = M != kLongOnly;
  static constexpr bool lng = M != kWindow;
  static constexpr bool long16 = M == kFused;
  static constexpr bool write_long = M == kLongOnly;
};

struct Item {
  int bh, b0, kt0, nw;  // nw: window tiles
};
template <int M>
__device__ __forceinline__ Item item_of(const Params &p, int g) {
  Item it;
  it.bh = g / p.nblk;
  it.b0 = (g % p.nblk) * kBq;
  it.kt0 = max(0, it.b0 - p.w + 1) / kKT * kKT;
  it.nw = Flags<M>::window ? (it.b0 + kBq - it.kt0) / kKT : 0;
  return it;
}

// The CTA's i-th q-tile.  Without a scheduler word the CTAs take q-tiles
// round-robin; with one, each CTA starts with q-tile blockIdx.x and then
// takes the next unclaimed one (one atomic ticket per q-tile, drawn by the
// union warp one q-tile ahead and published to the CTA's roles in a ring of
// four), so CTAs that drew cheap q-tiles take more of them and all finish
// together.  A value >= nitems ends the sequence; -1 is a failed wait.
__device__ __forceinline__ int next_item(const Params &p, Barriers &bar, uint32_t i) {
  if (!p.sched) return blockIdx.x + (int)i * gridDim.x;
  if (!wait_nth(&bar.g_full[i & 3], i >> 2, p.err)) return -1;
  return *reinterpret_cast<volatile int *>(&bar.g_ring[i & 3]);
}
__device__ __forceinline__ void publish_item(Barriers &bar, uint32_t i, int g) {
  bar.g_ring[i & 3] = g;
  tc::mbar_arrive(&bar.g_full[i & 3]);  // release: the roles read the slot after their wait
}
template <int M>
__device__ __forceinline__ int long_tiles(const Barriers &bar) {
  return Flags<M>::lng ? (bar.nu + 3) / 4 : 0;
}

// --------------------------------------------------------------------------
// RoPE rotation (window tiles)
// --------------------------------------------------------------------------
// Rotate half of one 64-element row in place: pairs i in [16*half, 16*half+16)
// (dims 16*half.. and 32+16*half..), angles composed from rows t64r (position
// mod 64, shared memory) and tur (64*u, global) by the angle-sum identity.  The raw row is read from
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
      const float4 bb = __ldg(reinterpret_cast<const float4 *>(tur + i0));
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

// Rotate row r (64 elements, in place) by the absolute position n.
__device__ __forceinline__ void rotate_row(unsigned char *hi, unsigned char *lo, int r, int n,
                                           const unsigned char *smem, const float2 *tab) {
  const float2 *t64r = reinterpret_cast<const float2 *>(smem + kOffT64 + (n & 63) * kT64Stride);
  const float2 *tur = tab + (size_t)(64 + (n >> 6)) * (kD / 2);
  // one copy of the half-row code: the staging warps also run the epilogue,
  // and straight-line code here competes with the softmax loop for the
  // instruction cache
#pragma unroll 1
  for (int half = 0; half < 2; ++half) rotate_half_row(hi, lo, r, half, t64r, tur);
}

// --------------------------------------------------------------------------
// roles
// --------------------------------------------------------------------------

template <int M>
__device__ void role_qk(const Params &p, Barriers &bar, uint32_t tmem, uint32_t base) {
  const uint32_t id_qk = tc::idesc_bf16(128, kKT, 0);
  const uint64_t dqh = tc::desc_sw128(base + kOffQ), dql = tc::desc_sw128(base + kOffQ + 16384);
  const uint64_t dqr = tc::desc_sw128(base + kOffQR);
  uint32_t T = 0, i = 0;
  for (;; ++i) {
    const int g = next_item(p, bar, i);
    if (g < 0) return;
    if (g >= p.nitems) break;
    const Item it = item_of<M>(p, g);
    if (!wait_nth(&bar.q_full, i, p.err)) return;
    int nl = 0;
    for (int t = 0;; ++t, ++T) {
      if (t == it.nw) {  // the window tiles do not wait for the union
        if (!wait_nth(&bar.u_full, i, p.err)) return;
        nl = long_tiles<M>(bar);
        tc::mbar_arrive(&bar.u_free);
      }
      if (t >= it.nw + nl) break;
      const int slot = T % kRing, b = T & 1;
      if (!wait_nth(&bar.raw_full[slot], T / kRing, p.err)) return;
      if (T >= 2 && !wait_nth(&bar.s_free[b], T / 2 - 1, p.err)) return;
      tc::fence_after_sync();
      const uint32_t kh = base + kOffK + slot * 32768;
      const uint64_t dkh = tc::desc_sw128(kh), dkl = tc::desc_sw128(kh + 16384);
      const uint32_t s_col = tmem + kColS + 128 * b;
      if (t < it.nw) {  // window: three split-precision chains
#pragma unroll
        for (int part = 0; part < 3; ++part) {
          const uint64_t a = part == 2 ? dql : dqh, bd = part == 1 ? dkl : dkh;
#pragma unroll
          for (int k = 0; k < kD / 16; ++k)
            tc::mma_ss(s_col, a + (uint64_t)(2 * k), bd + (uint64_t)(2 * k), id_qk,
                       (part > 0 || k > 0) ? 1u : 0u);
        }
      } else {  // long: unrotated query against the gathered cells
#pragma unroll
        for (int k = 0; k < kD / 16; ++k)
          tc::mma_ss(s_col, dqr + (uint64_t)(2 * k), dkh + (uint64_t)(2 * k), id_qk,
                     k > 0 ? 1u : 0u);
      }
      tc::mma_commit(&bar.s_full[b]);
      tc::mma_commit(&bar.k_empty[slot]);
    }
    tc::mma_commit(&bar.q_empty);
  }
}

// The P.V MMA loops stay rolled: the issuing thread waits on the tensor pipe
// either way, and the smaller loop body leaves more of the instruction cache
// to the softmax warps that share its SMSP (measured: 5% faster attention).
template <int M>
__device__ void role_pv(const Params &p, Barriers &bar, uint32_t tmem, uint32_t base) {
  const uint32_t id_pv = tc::idesc_bf16(128, kD, 1);  // long: bf16 P hi / lo, bf16 V
  const uint32_t id_pv_h = tc::idesc_f16(128, kD, 1);  // window (and long16): fp16 P, V
  uint32_t T = 0, i = 0;
  for (;; ++i) {
    const int g = next_item(p, bar, i);
    if (g < 0) return;
    if (g >= p.nitems) break;
    const Item it = item_of<M>(p, g);
    const uint32_t ob = tmem + kColO + 128 * (i & 1);
    // an accumulator set is reused once the epilogue two q-tiles back has read it
    if (i >= 2 && !wait_nth(&bar.o_free[i & 1], (i - 2) >> 1, p.err)) return;
    int nl = 0;
    for (int t = 0;; ++t, ++T) {
      if (t == it.nw) {
        if (!wait_nth(&bar.u_full, i, p.err)) return;
        nl = long_tiles<M>(bar);
        tc::mbar_arrive(&bar.u_free);
      }
      if (t >= it.nw + nl) break;
      const int slot = T % kRing, b = T & 1;
      if (!wait_nth(&bar.p_full[b], T / 2, p.err)) return;
      // the value tile is read by this thread's MMAs: observe its arrival here too
      if (!wait_nth(&bar.raw_full[slot], T / kRing, p.err)) return;
      tc::fence_after_sync();
      const uint64_t dv = tc::desc_sw128(base + kOffV + slot * 16384);
      const uint32_t sp = tmem + kColS + 128 * b;
      if (t < it.nw) {
#pragma unroll 1
        for (int k = 0; k < kKT / 16; ++k)
          tc::mma_ts(ob, sp + p_col(k), dv + (uint64_t)(k * 128), id_pv_h,
                     (t > 0 || k > 0) ? 1u : 0u);
      } else if (Flags<M>::long16) {
        const bool first = t == it.nw;
#pragma unroll 1
        for (int k = 0; k < kKT / 16; ++k)
          tc::mma_ts(ob + 64, sp + p_col(k), dv + (uint64_t)(k * 128), id_pv_h,
                     (!first || k > 0) ? 1u : 0u);
      } else {
        const bool first = t == it.nw;
#pragma unroll 1
        for (int part = 0; part < 2; ++part)
#pragma unroll 1
          for (int k = 0; k < kKT / 16; ++k)
            tc::mma_ts(ob + 64, sp + p_col(k) + 16 * part, dv + (uint64_t)(k * 128), id_pv,
                       (!first || part > 0 || k > 0) ? 1u : 0u);
      }
      tc::mma_commit(&bar.pv_done);
      tc::mma_commit(&bar.v_empty[slot]);
      tc::mma_commit(&bar.s_free[b]);
    }
    tc::mma_commit(&bar.o_done[i & 1]);
  }
}

// Before the CTA exits, every tile load this thread issued has landed (the
// normal path consumed them all; after a wait gave up, this bounds the
// wait for the ones still in flight by time only).
__device__ void drain_tma(Barriers &bar, uint32_t issued) {
  for (uint32_t T = issued > kRing ? issued - kRing : 0; T < issued; ++T)
    tc::mbar_wait(&bar.raw_full[T % kRing], T / kRing, nullptr);
}

template <int M>
__device__ void role_tma(const Params &p, Barriers &bar, unsigned char *smem,
                         const CUtensorMap *tkt, const CUtensorMap *tv16, const CUtensorMap *ck,
                         const CUtensorMap *cv) {
  uint32_t T = 0, i = 0;
  const int *ul = reinterpret_cast<const int *>(smem + kOffUL);
  for (;; ++i) {
    const int g = next_item(p, bar, i);
    if (g < 0) return drain_tma(bar, T);
    if (g >= p.nitems) break;
    const Item it = item_of<M>(p, g);
    const int row0 = it.bh * p.N;
    int nl = 0;
    for (int t = 0;; ++t, ++T) {
      if (t == it.nw) {
        if (!wait_nth(&bar.u_full, i, p.err)) return drain_tma(bar, T);
        nl = long_tiles<M>(bar);
      }
      if (t >= it.nw + nl) break;
      const int slot = T % kRing;
      if (T >= kRing) {
        if (!wait_nth(&bar.k_empty[slot], T / kRing - 1, p.err)) return drain_tma(bar, T);
        if (!wait_nth(&bar.v_empty[slot], T / kRing - 1, p.err)) return drain_tma(bar, T);
      }
      unsigned char *kd = smem + kOffK + slot * 32768, *vd = smem + kOffV + slot * 16384;
      if (t < it.nw) {  // rotated keys (hi, lo) and fp16 values: 48 KB
        const int y = row0 + it.kt0 + t * kKT;
        tc::mbar_arrive_expect_tx(&bar.raw_full[slot], 3 * kKT * kD * 2);
        tc::tma_load_2d(kd, tkt, &bar.raw_full[slot], 0, y);
        tc::tma_load_2d(kd + 16384, tkt, &bar.raw_full[slot], kD, y);
        tc::tma_load_2d(vd, tv16, &bar.raw_full[slot], 0, y);
      } else {  // raw keys and values (fp16 copy under long16) of four cells: 32 KB
        tc::mbar_arrive_expect_tx(&bar.raw_full[slot], 2 * kKT * kD * 2);
        // four cells of the union; a missing cell reads zeros from past the
        // last row, so stale data never meets a zero probability
        const int lt = t - it.nw;
#pragma unroll
        for (int cs = 0; cs < 4; ++cs) {
          const int u = 4 * lt + cs;
          const int y = u < bar.nu ? row0 + ul[u] * kS : (int)p.nrows;
          tc::tma_load_2d(kd + cs * 4096, ck, &bar.raw_full[slot], 0, y);
          tc::tma_load_2d(vd + cs * 4096, cv, &bar.raw_full[slot], 0, y);
        }
      }
    }
    tc::mbar_arrive(&bar.u_free);  // the union list is no longer read
  }
  drain_tma(bar, T);
}

// Union of the q-tile's selected cells, sorted ascending, and each
// selection's slot in it (for the softmax masks).  The warp marks the
// selections in a shared bitmap over a window of 32 * kBW cell ids, then one
// prefix sum of the words' bit counts gives every cell its rank: the union
// is the set bits in order (ul), and a selection's slot is its word's prefix
// plus the set bits below it.
//
// Ranking the words of one window, from word 0: the set bits in order go to
// ul[nu...], each word's first rank to pw.  Returns the new union size.
__device__ __forceinline__ int union_scan(const uint32_t *bm, uint16_t *pw, int *ul, int nwd,
                                          int base, int nu, int lane) {
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
    int k = nu + incl - cnt;
    if (w < nwd) pw[w] = (uint16_t)k;
    while (bits) {
      ul[k++] = base + 32 * w + (__ffs(bits) - 1);
      bits &= bits - 1;
    }
    nu += __shfl_sync(0xffffffffu, incl, 31);
  }
  return nu;
}

// Cells are placed window by window (32 * kBW ids each, from the smallest
// cell not yet placed; one window while N / s <= 8192): mark, rank, then
// look up each selection's slot, reading the selections again for each step.
// They are brought into L1 before the wait for the previous union's readers
// (one line per lane: 128 K int32, 4 KB at most).  The fused kernel has
// time to spare for this (the union is needed only after the window tiles)
// and gains from the small code.  Alone, the long branch waits for each
// union, so its kernel takes a register path when K <= 4 and every cell id is
// below 8192: the selections (16 per lane at most) are loaded before the
// wait, marked from the registers, and their slot lookups go out together.
constexpr int kFastSel = 16;
template <int M>
__device__ void role_union(const Params &p, Barriers &bar, unsigned char *smem) {
  const int lane = threadIdx.x & 31;
  int *ul = reinterpret_cast<int *>(smem + kOffUL);
  uint16_t *rs = reinterpret_cast<uint16_t *>(smem + kOffRS);
  uint32_t *bm = reinterpret_cast<uint32_t *>(smem + kOffBM);
  uint16_t *pw = reinterpret_cast<uint16_t *>(smem + kOffPW);
  const int ne = p.K * (kBq / 32);  // selections per lane (a multiple of 4)
  uint32_t i = 0;
  // the scheduler (see next_item): the CTA's first q-tile is its own index,
  // each later one a ticket drawn one q-tile ahead
  if (p.sched && lane == 0) publish_item(bar, 0, blockIdx.x < p.nitems ? blockIdx.x : p.nitems);
  for (int g = blockIdx.x, g_next = 0; g < p.nitems; g = g_next, ++i) {
    g_next = g + gridDim.x;
    if (p.sched) {
      int tk = 0;
      if (lane == 0) {
        tk = gridDim.x + atomicAdd(p.sched, 1);
        publish_item(bar, i + 1, tk < p.nitems ? tk : p.nitems);
      }
      g_next = __shfl_sync(0xffffffffu, tk, 0);
    }
    const Item it = item_of<M>(p, g);
    const int A = it.b0 / kS;  // cells ending at or before the block start
    const int32_t *blk = p.sel + ((size_t)it.bh * p.N + it.b0) * p.K;
    const int32_t *src = blk + lane;
    const bool fast = M == kLongOnly && ne <= kFastSel && A <= 32 * kBW;
    int c[kFastSel];
    if (fast) {
#pragma unroll
      for (int e = 0; e < kFastSel; ++e) c[e] = e < ne ? __ldg(src + 32 * e) : -1;
    } else if (Flags<M>::lng && 128 * lane < 4 * kBq * p.K + 127) {
      asm volatile("prefetch.global.L1 [%0];" ::"l"(reinterpret_cast<const char *>(blk) + 128 * lane));
    }
    if (i > 0 && !wait_nth(&bar.u_free, i - 1, p.err)) return;
    int nu = 0;
    if (fast) {
      for (int w = lane; w < (A + 31) >> 5; w += 32) bm[w] = 0u;
      __syncwarp();
      int hi = -1;
#pragma unroll
      for (int e = 0; e < kFastSel; ++e) {
        if (c[e] >= A) c[e] = -1;  // not yet complete
        hi = max(hi, c[e]);
        if (c[e] >= 0) atomicOr(&bm[c[e] >> 5], 1u << (c[e] & 31));
        else if (e < ne) rs[32 * e + lane] = 0xffff;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
      __syncwarp();
      nu = union_scan(bm, pw, ul, (hi >> 5) + 1, 0, 0, lane);
      __syncwarp();
#pragma unroll
      for (int e = 0; e < kFastSel; ++e)
        if (c[e] >= 0)
          rs[32 * e + lane] =
              (uint16_t)(pw[c[e] >> 5] + __popc(bm[c[e] >> 5] & ((1u << (c[e] & 31)) - 1u)));
    } else if (Flags<M>::lng) {
      // a selection's cell, or -1 for none / not yet complete
      auto cell_of = [&](int e) {
        const int v = __ldg(src + 32 * e);
        return (v >= 0 && v < A) ? v : -1;
      };
      int lo = 0x7fffffff, hi = -1;
#pragma unroll 4
      for (int e = 0; e < ne; ++e) {
        const int v = cell_of(e);
        if (v < 0) rs[32 * e + lane] = 0xffff;
        else lo = min(lo, v);
        hi = max(hi, v);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
      }
      while (lo <= hi) {  // one pass per window of cells (warp-uniform)
        const int base = lo & ~31, end = base + 32 * kBW;
        const int nwd = min(kBW, ((hi - base) >> 5) + 1);
        for (int w = lane; w < nwd; w += 32) bm[w] = 0u;
        __syncwarp();
#pragma unroll 4
        for (int e = 0; e < ne; ++e) {
          const int v = cell_of(e);
          if (v >= base && v < end) atomicOr(&bm[(v - base) >> 5], 1u << (v & 31));
        }
        __syncwarp();
        nu = union_scan(bm, pw, ul, nwd, base, nu, lane);
        __syncwarp();
        int next = 0x7fffffff;
#pragma unroll 4
        for (int e = 0; e < ne; ++e) {
          const int v = cell_of(e);
          if (v >= base && v < end) {
            const int w = (v - base) >> 5;
            rs[32 * e + lane] = (uint16_t)(pw[w] + __popc(bm[w] & ((1u << (v & 31)) - 1u)));
          } else if (v >= end) {
            next = min(next, v);
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) next = min(next, __shfl_xor_sync(0xffffffffu, next, o));
        lo = next;
        __syncwarp();  // the bitmap is read before the next pass clears it
      }
    }
    if (lane == 0) bar.nu = nu;
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&bar.u_full);
  }
}

template <int M>
__device__ bool epilogue_rows(const Params &p, Barriers &bar, uint32_t tmem, int g, uint32_t i,
                              int r);

// Query staging and epilogue: row r of each q-tile, raw (NoPE long branch)
// and, for the window, rotated by its absolute position and split into bf16
// hi / lo; after staging q-tile i, the epilogue of q-tile i-1.  One pass
// past the last q-tile runs the last epilogue.
template <int M>
__device__ void role_qprep(const Params &p, Barriers &bar, unsigned char *smem, uint32_t tmem,
                           int r) {
  uint32_t i = 0;
  int g_prev = -1;
  for (;; ++i) {
    const int g = next_item(p, bar, i);
    if (g < 0) return;
    const bool real = g < p.nitems;
    if (real) {
      const Item it = item_of<M>(p, g);
      // fetch the row first, then wait until the previous q-tile's S MMAs no
      // longer read the query tiles
      const uint4 *src =
          reinterpret_cast<const uint4 *>(p.q + ((size_t)it.bh * p.N + it.b0 + r) * kD);
      uint4 raw[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) raw[c] = __ldg(src + c);
      if (i > 0 && !wait_nth(&bar.q_empty, i - 1, p.err)) return;
      unsigned char *qh = smem + kOffQ, *qr = smem + kOffQR;
#pragma unroll
      for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(qr + swz128(r, c)) = raw[c];
      if (Flags<M>::window) {
#pragma unroll
        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4 *>(qh + swz128(r, c)) = raw[c];
        rotate_row(qh, qh + 16384, r, it.b0 + r, smem, p.tab);
      }
      tc::fence_async_smem();
      tc::mbar_arrive(&bar.q_full);
    }
    if (g_prev >= 0 && !epilogue_rows<M>(p, bar, tmem, g_prev, i - 1, r)) return;
    if (!real) break;
    g_prev = g;
  }
}

// A warp's 64 score columns of a row are held in registers as two 32-column
// chunks: loaded once, masked, reduced to the row maximum, then turned into
// probabilities in place of the scores.
constexpr uint32_t kNegInf = 0xff800000u;

// window: columns outside [lo, hi] (tile columns) become -inf; the test is
// uniform across the warp except in a chunk a triangular edge crosses.
// Returns whether any row of the warp reads a column of the chunk.
__device__ __forceinline__ bool mask_window(uint32_t (&x)[32], int lo, int hi, int c0) {
  const bool full = lo <= c0 && hi >= c0 + 31;
  const bool empty = hi < c0 || lo > c0 + 31;
  if (__all_sync(0xffffffffu, full)) return true;
  if (__all_sync(0xffffffffu, empty)) {
#pragma unroll
    for (int c = 0; c < 32; ++c) x[c] = kNegInf;
    return false;
  }
  // bit c set iff column c0 + c lies in [lo, hi]; then one select per element
  // (no per-element branches)
  const int a = min(max(lo - c0, 0), 32), b = min(max(hi - c0 + 1, 0), 32);
  const uint32_t below_b = b >= 32 ? 0xffffffffu : (1u << b) - 1u;
  const uint32_t below_a = a >= 32 ? 0xffffffffu : (1u << a) - 1u;
  const uint32_t valid = below_b & ~below_a;
#pragma unroll
  for (int c = 0; c < 32; ++c) x[c] = (valid & (1u << c)) ? x[c] : kNegInf;
  return true;
}

__device__ __forceinline__ float max_chunk(const uint32_t (&x)[32]) {
  // four running maxima, two new elements per three-input max
  float mx[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) mx[j] = __uint_as_float(x[j]);
#pragma unroll
  for (int c = 4; c < 32; c += 2)
    mx[(c >> 1) & 3] = max3f(mx[(c >> 1) & 3], __uint_as_float(x[c]), __uint_as_float(x[c + 1]));
  return max3f(mx[0], mx[1], fmaxf(mx[2], mx[3]));
}

// 2^(s*sl2 - m) for one chunk, written as pairs into 16 P columns: fp16 for a
// window tile; bf16 for a long tile, with the bf16 rounding remainders in 16
// P_lo columns (kSplit).  Returns the sum of the unrounded values.
template <bool kSplit>
__device__ __forceinline__ float exp_chunk(const uint32_t (&x)[32], uint32_t p_addr,
                                           uint32_t pl_addr, float sl2, float m) {
  // two pairs of partial sums (packed adds), arguments by packed FMA
  float part[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int h16 = 0; h16 < 2; ++h16) {
    uint32_t pk[8], pl[8];
#pragma unroll
    for (int c = 0; c < 16; c += 2) {
      float a0, a1;
      fma2(a0, a1, __uint_as_float(x[16 * h16 + c]), __uint_as_float(x[16 * h16 + c + 1]), sl2, -m);
      const float e0 = tc::ex2(a0);
      const float e1 = tc::ex2(a1);
      const int q = (c >> 1) & 1;
      add2(part[2 * q], part[2 * q + 1], e0, e1);
      if (kSplit) {  // long tile: bf16 hi + lo (remainders by one packed subtract)
        pk[c / 2] = pack_bf16(e0, e1);
        const unsigned long long hi2 =
            (unsigned long long)(pk[c / 2] << 16) | ((unsigned long long)(pk[c / 2] & 0xffff0000u) << 32);
        const unsigned long long rem = sub2_bits(f2_bits(e0, e1), hi2);
        pl[c / 2] = pack_bf16(__uint_as_float((uint32_t)rem), __uint_as_float((uint32_t)(rem >> 32)));
      } else {  // window tile: fp16
        pk[c / 2] = pack_f16(e0, e1);
      }
    }
    tc::tmem_st8(p_addr + 8 * h16, pk);
    if (kSplit) tc::tmem_st8(pl_addr + 8 * h16, pl);
  }
  return (part[0] + part[1]) + (part[2] + part[3]);
}

// The two softmax warps that share a row block swap one float2 per row:
// publish, meet on an mbarrier (one phase per swap; bounded wait, so a failed
// partner cannot hang the CTA), read the partner's.  Slots alternate by swap
// parity: a slot is rewritten two swaps later, after the partner has met us
// once more and so has read it.
struct Pair {
  uint64_t *bar;
  float2 (*slot)[2][128];
  uint32_t phase;
  __device__ __forceinline__ bool swap(float2 mine, float2 &theirs, int half, int r, int lane,
                                       int *err) {
    const uint32_t par = phase & 1;
    slot[par][half][r] = mine;
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(bar);
    const bool ok = tc::mbar_wait(bar, par, err);
    theirs = slot[par][half ^ 1][r];
    ++phase;
    return ok;
  }
};

__device__ __forceinline__ void rescale(uint32_t addr, float alpha) {
  uint32_t o[32];
  tc::tmem_ld32(addr, o);
  tc::tmem_wait_ld();
#pragma unroll
  for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
  tc::tmem_st32(addr, o);
}

// Epilogue of one q-tile, run by the query-staging warpgroup (warp 12 + q
// reads TMEM lanes 32q..32q+31), one thread per query row and all 64 output
// columns: O_long / l_long and its RMSNorm, O_win / l_win, the mix, the
// store.  The softmax warps have moved on to the next q-tile; the P.V
// issuer reuses this accumulator set only for the q-tile after that.
template <int M>
__device__ bool epilogue_rows(const Params &p, Barriers &bar, uint32_t tmem, int g, uint32_t i,
                              int r) {
  const Item it = item_of<M>(p, g);
  const int lane = r & 31, par = i & 1;
  const uint32_t lane_base = (uint32_t)(r & ~31) << 16;
  if (!wait_nth(&bar.o_done[par], i >> 1, p.err)) return false;
  if (!wait_nth(&bar.stats_full[par], i >> 1, p.err)) return false;
  tc::fence_after_sync();
  const float2 s0 = bar.stat[par][0][r], s1 = bar.stat[par][1][r];
  const int nl = bar.item_nl[par];
  const float lw = s0.x + s1.x, ll = s0.y + s1.y;
  const uint32_t ow = tmem + kColO + 128 * par + lane_base, ol = ow + 64;
  const bool load_long = Flags<M>::lng && nl > 0;      // the whole warp (same q-tile)
  const bool use_win = !Flags<M>::write_long && it.nw > 0;  // the whole warp
  const float invl = ll > 0.f ? 1.f / ll : 0.f;
  float lo_scale = 0.f;
  if (load_long) {
    float sq[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int c32 = 0; c32 < 2; ++c32) {
      uint32_t o[32];
      tc::tmem_ld32(ol + 32 * c32, o);
      tc::tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const float y = __uint_as_float(o[c]) * invl;
        sq[c & 3] = fmaf(y, y, sq[c & 3]);
      }
    }
    const float ss = (sq[0] + sq[1]) + (sq[2] + sq[3]);
    lo_scale = ll > 0.f ? invl * rsqrtf(ss / kD + p.rms_eps) : 0.f;
  }
  const float wscale = it.nw > 0 ? 1.f / lw : 0.f;
  const size_t row = (size_t)it.bh * p.N + it.b0 + r;
  float4 *dst = reinterpret_cast<float4 *>(p.out + row * kD);
  const float mh = p.mix ? p.mix[it.bh % p.H] : 0.f;
  const bool use_long = lo_scale != 0.f;  // this row
  const float4 *oin = (!Flags<M>::write_long && !use_long && p.o_long_in)
      ? reinterpret_cast<const float4 *>(p.o_long_in + row * kD) : nullptr;
  const float ls = Flags<M>::write_long ? lo_scale : mh * lo_scale;
#pragma unroll 1
  for (int c16 = 0; c16 < kD / 16; ++c16) {
    uint32_t w[16], l16[16];
    if (use_win) tc::tmem_ld16(ow + 16 * c16, w);
    if (load_long) tc::tmem_ld16(ol + 16 * c16, l16);
    tc::tmem_wait_ld();
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = 4 * c4 + e;
        float y = use_win ? __uint_as_float(w[c]) * wscale : 0.f;
        if (load_long) y = fmaf(ls, __uint_as_float(l16[c]), y);
        v[e] = y;
      }
      float4 o4 = make_float4(v[0], v[1], v[2], v[3]);
      if (oin) {
        const float4 u4 = __ldg(oin + 4 * c16 + c4);
        o4.x = fmaf(mh, u4.x, o4.x);
        o4.y = fmaf(mh, u4.y, o4.y);
        o4.z = fmaf(mh, u4.z, o4.z);
        o4.w = fmaf(mh, u4.w, o4.w);
      }
      dst[4 * c16 + c4] = o4;
    }
  }
  // accumulator set and row-sum slot may be reused
  tc::fence_before_sync();
  __syncwarp();
  if (lane == 0) {
    tc::mbar_arrive(&bar.o_free[par]);
    tc::mbar_arrive(&bar.stat_free[par]);
  }
  return true;
}

// Which of the warp's 64 columns of key tile t its rows read: the window
// bounds [lo, hi] of the row, or which of the long tile's two cells the row
// picked.  Returns whether any lane of the warp reads a column.
__device__ __forceinline__ bool tile_cols(const Params &p, const Item &it, int t, int n, int half,
                                          const uint32_t (&pick)[kMaxK / 2], int &lo, int &hi,
                                          bool (&cell)[2]) {
  cell[0] = cell[1] = false;
  lo = 0;
  hi = -1;
  if (t < it.nw) {
    const int kt = it.kt0 + t * kKT;
    lo = max(0, n - p.w + 1 - kt);
    hi = min(kKT - 1, n - kt);
    return __any_sync(0xffffffffu, lo <= hi && hi >= 64 * half && lo <= 64 * half + 63);
  }
  const uint32_t u0 = 4 * (t - it.nw) + 2 * half;
#pragma unroll
  for (int k = 0; k < kMaxK / 2; ++k) {
    const uint32_t a = pick[k] & 0xffffu, bb = pick[k] >> 16;
    cell[0] |= (a == u0) || (bb == u0);
    cell[1] |= (a == u0 + 1) || (bb == u0 + 1);
  }
  return __any_sync(0xffffffffu, cell[0] || cell[1]);
}

template <int M>
__device__ void role_softmax(const Params &p, Barriers &bar, uint32_t tmem, unsigned char *smem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3, half = warp >> 2;
  const int r = quarter * 32 + lane;  // query row of this thread
  const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
  const uint16_t *rs = reinterpret_cast<const uint16_t *>(smem + kOffRS);
  const float sl2 = 1.4426950408889634f * 0.125f;  // log2(e) / sqrt(64)
  uint32_t T = 0, i = 0;
  Pair pr{&bar.pair[quarter], bar.xch, 0u};
  for (;; ++i) {
    const int g = next_item(p, bar, i);
    if (g < 0) return;
    if (g >= p.nitems) break;
    const Item it = item_of<M>(p, g);
    const int n = it.b0 + r;
    const uint32_t ow_addr = tmem + kColO + 128 * (i & 1) + 32 * half + lane_base;
    float mw = -INFINITY, lw = 0.f, ml = -INFINITY, ll = 0.f;
    int nl = 0;
    uint32_t pick[kMaxK / 2];  // this row's union slots, two 16-bit slots per word
    for (int t = 0;; ++t, ++T) {
      if (t == it.nw) {
        if (!wait_nth(&bar.u_full, i, p.err)) return;
        nl = long_tiles<M>(bar);
#pragma unroll
        for (int k = 0; k < kMaxK / 2; ++k) {
          const uint32_t a = (2 * k < p.K) ? rs[r * p.K + 2 * k] : 0xffffu;
          const uint32_t b = (2 * k + 1 < p.K) ? rs[r * p.K + 2 * k + 1] : 0xffffu;
          pick[k] = a | (b << 16);
        }
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bar.u_free);  // union data read
      }
      const bool done = t >= it.nw + nl;
      if (!done) {
        const bool is_long = t >= it.nw;
        const bool split = is_long && !Flags<M>::long16;  // bf16 hi + lo P
        const int b = T & 1;
        const uint32_t s_addr = tmem + kColS + 128 * b + 64 * half + lane_base;
        if (!wait_nth(&bar.s_full[b], T / 2, p.err)) return;
        tc::fence_after_sync();
        bool cell[2];
        int lo, hi;
        const bool any = tile_cols(p, it, t, n, half, pick, lo, hi, cell);
        // the warp's 64 score columns in one TMEM round trip
        uint32_t xa[32], xb[32];
        float mx = -INFINITY;
        // per 32-key chunk: does any row of the warp read it (else its
        // probabilities are zeros, written without exponentials)
        bool live0 = false, live1 = false;
        if (any) {
          tc::tmem_ld32(s_addr, xa);
          tc::tmem_ld32(s_addr + 32, xb);
          tc::tmem_wait_ld();
          if (!is_long) {
            live0 = mask_window(xa, lo, hi, 64 * half);
            live1 = mask_window(xb, lo, hi, 64 * half + 32);
            mx = fmaxf(max_chunk(xa), max_chunk(xb));
          } else {
            live0 = __any_sync(0xffffffffu, cell[0]);
            live1 = __any_sync(0xffffffffu, cell[1]);
            // a long tile's chunk is one cell, picked by the row or not: its
            // scores are left as they are and the pick enters the maximum
            // here and the probabilities below (through their reference)
            const float ma = max_chunk(xa), mb = max_chunk(xb);
            mx = fmaxf(cell[0] ? ma : -INFINITY, cell[1] ? mb : -INFINITY);
          }
        }
        float2 o;
        if (!pr.swap(make_float2(mx, 0.f), o, half, r, lane, p.err)) return;
        mx = fmaxf(mx, o.x);
        const float m = is_long ? ml : mw;
        float l = is_long ? ll : lw;
        const float mt = mx * sl2;
        const float mnew = mt > m + (split ? kLazyLong : kLazyWin) ? mt : m;
        const bool first = is_long ? t == it.nw : t == 0;
        // the accumulator holds exact zeros while m is -inf: nothing to rescale
        const bool resc = !first && m != -INFINITY && mnew != m;
        const float alpha = resc ? tc::ex2(m - mnew) : 1.f;
        const float muse = mnew == -INFINITY ? 0.f : mnew;
        // rounded products and sums, never contracted into an FMA: every
        // instantiation of this kernel gives the window branch the same bits
        l = __fmul_rn(l, alpha);
        if (any) {
          // chunk 0 from xa, then chunk 1 moved into xa (one copy of the code)
#pragma unroll 1
          for (int ch = 0; ch < 2; ++ch) {
            const uint32_t pa = s_addr + 32 * ch;
            if (ch ? live1 : live0) {
              // an unpicked cell gets reference +inf: 2^(x - inf) = 0 exactly
              const float mref = (is_long && !(ch ? cell[1] : cell[0])) ? INFINITY : muse;
              l = __fadd_rn(l, split ? exp_chunk<true>(xa, pa, pa + 16, sl2, mref)
                                     : exp_chunk<false>(xa, pa, pa + 16, sl2, mref));
            } else {
              uint32_t z[16];
#pragma unroll
              for (int c = 0; c < 16; ++c) z[c] = 0u;
              tc::tmem_st16(pa, z);
              if (split) tc::tmem_st16(pa + 16, z);
            }
            if (ch == 0) {
#pragma unroll
              for (int c = 0; c < 32; ++c) xa[c] = xb[c];
            }
          }
        } else {
          uint32_t z[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) z[c] = 0u;
          tc::tmem_st16(s_addr, z);
          tc::tmem_st16(s_addr + 32, z);
          if (split) {
            tc::tmem_st16(s_addr + 16, z);
            tc::tmem_st16(s_addr + 48, z);
          }
        }
        if (is_long) {
          ml = mnew;
          ll = l;
        } else {
          mw = mnew;
          lw = l;
        }
        if (__any_sync(0xffffffffu, resc)) {
          // the previous P.V accumulates into the same set: let it finish
          if (!wait_nth(&bar.pv_done, T - 1, p.err)) return;
          tc::fence_after_sync();
          rescale(ow_addr + (is_long ? 64 : 0), alpha);
        }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&bar.p_full[b]);
      }
      if (done) break;
    }
    // hand this half-row's sums to the epilogue warpgroup (slot of the
    // q-tile's parity; it was read two q-tiles ago)
    const int par = i & 1;
    if (i >= 2 && !wait_nth(&bar.stat_free[par], (i >> 1) - 1, p.err)) return;
    bar.stat[par][half][r] = make_float2(lw, ll);
    if (warp == 0 && lane == 0) bar.item_nl[par] = nl;
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&bar.stats_full[par]);
  }
}

template <int M>
__global__ void __launch_bounds__(kThreads, 1) fs_attn_tc_kernel(
    const __grid_constant__ CUtensorMap tmap_kt, const __grid_constant__ CUtensorMap tmap_v16,
    const __grid_constant__ CUtensorMap cmap_k, const __grid_constant__ CUtensorMap cmap_v,
    const Params p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ Barriers bar;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0 && p.timeline) p.timeline[2 * blockIdx.x] = tc::global_ns();

  if (threadIdx.x == 0) {
    tc::mbar_init(&bar.q_full, kRotThreads);
    tc::mbar_init(&bar.q_empty, 1);
    for (int i = 0; i < kRing; ++i) {
      tc::mbar_init(&bar.raw_full[i], 1);
      tc::mbar_init(&bar.k_empty[i], 1);
      tc::mbar_init(&bar.v_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bar.s_full[b], 1);
      tc::mbar_init(&bar.s_free[b], 1);
      tc::mbar_init(&bar.fin[b], 1);
      tc::mbar_init(&bar.o_done[b], 1);
      tc::mbar_init(&bar.o_free[b], 4);      // the epilogue (query-staging) warps
      tc::mbar_init(&bar.stats_full[b], 8);  // the softmax warps
      tc::mbar_init(&bar.stat_free[b], 4);
    }
    for (int b = 0; b < 2; ++b) tc::mbar_init(&bar.p_full[b], 8);
    for (int q4 = 0; q4 < 4; ++q4) tc::mbar_init(&bar.pair[q4], 2);
    tc::mbar_init(&bar.pv_done, 1);
    tc::mbar_init(&bar.u_full, 1);
    for (int j = 0; j < 4; ++j) tc::mbar_init(&bar.g_full[j], 1);
    // the union may be rebuilt once every role has read it: 8 softmax warps,
    // the two issuers and the TMA thread
    tc::mbar_init(&bar.u_free, 11);
    tc::mbar_fence_init();
  }
  if (warp == 8) {
    tc::tmem_alloc(&bar.tmem, kTmemCols);
    tc::tmem_relinquish();
  }
  // rows r*theta (r < 64) of the angle table, staged once per CTA (window only)
  if (threadIdx.x >= kRotBase && Flags<M>::window) {
    const float4 *tab = reinterpret_cast<const float4 *>(p.tab);
    for (int i = threadIdx.x - kRotBase; i < 64 * 16; i += kRotThreads) {
      const int row = i >> 4, part = i & 15;
      *reinterpret_cast<float4 *>(smem + kOffT64 + row * kT64Stride + part * 16) =
          __ldg(tab + (size_t)row * 16 + part);
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bar.tmem;
  const uint32_t sbase = smem_u32(smem);

  // Registers: the issuer / TMA / union warpgroup (warps 8-11) gives up 56
  // per thread, the query-staging / epilogue warpgroup (12-15) 24, the two
  // softmax warpgroups (0-7) take 40 more: 8*32*168 + 4*32*72 + 4*32*104 =
  // 65536, the block's launch allotment of 512 x 128.  Each change sits
  // inside its role's branch, so that the compiler sizes every role's code by
  // its own count.
  if (warp < 8) {
    tc::regs_inc<168>();
    role_softmax<M>(p, bar, tmem, smem);
  } else if (warp < 12) {
    tc::regs_dec<72>();
    if (warp == 8 || warp == 9) {
      if (lane == 0) {
        if (warp == 8)
          role_qk<M>(p, bar, tmem, sbase);
        else
          role_pv<M>(p, bar, tmem, sbase);
        // every MMA this thread issued has completed before TMEM is released
        // (bounded by time only, even after an error was recorded)
        tc::mma_commit(&bar.fin[warp - 8]);
        tc::mbar_wait(&bar.fin[warp - 8], 0, nullptr);
      }
    } else if (warp == 10) {
      if (lane == 0) role_tma<M>(p, bar, smem, &tmap_kt, &tmap_v16, &cmap_k, &cmap_v);
    } else {
      role_union<M>(p, bar, smem);
    }
  } else {
    tc::regs_dec<104>();
    role_qprep<M>(p, bar, smem, tmem, threadIdx.x - kRotBase);
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 8) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && p.timeline) p.timeline[2 * blockIdx.x + 1] = tc::global_ns();
  // the last CTA to finish clears the scheduler words for the next launch
  if (threadIdx.x == 0 && p.sched && atomicAdd(p.sched + 1, 1) == (int)gridDim.x - 1) {
    atomicExch(p.sched, 0);
    atomicExch(p.sched + 1, 0);
  }
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

// [rows, cols] 16-bit row-major (bf16 or fp16), boxes of box_rows x 64 with
// the 128-byte swizzle; rows past the end read as zeros.
bool make_rows_map(CUtensorMap *map, const void *ptr, size_t rows, int cols, int box_rows,
                   bool f16) {
  EncodeTiled fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kD, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

}  // namespace

namespace {
thread_local long long *g_timeline = nullptr;
thread_local int g_timeline_entries = 0;
}  // namespace

void set_attention_timeline(long long *timeline, int entries) {
  g_timeline = timeline;
  g_timeline_entries = entries;
}

cudaError_t launch_attn_tc(const AttnArgs &a, cudaStream_t st) {
  const Shape &sh = a.sh;
  if (!a.window && !a.sel) return cudaErrorInvalidValue;
  // the window branch reads the prepared operands and the angle table
  if (a.window && (!a.kt || !a.v16 || !a.tab)) return cudaErrorInvalidValue;
  CUtensorMap mkt, mv16, ck, cv;
  const size_t nrows = (size_t)sh.BH() * sh.N;
  memset(&mkt, 0, sizeof(mkt));
  memset(&mv16, 0, sizeof(mv16));
  if (a.window && (!make_rows_map(&mkt, a.kt, nrows, 2 * kD, kKT, false) ||
                   !make_rows_map(&mv16, a.v16, nrows, kD, kKT, true)))
    return cudaErrorInvalidValue;
  // with the window branch the fp16 values exist, and the long branch reads
  // its cells from them too
  const bool long16 = a.window && a.sel != nullptr;
  if (!make_rows_map(&ck, a.k, nrows, kD, kS, false) ||
      !make_rows_map(&cv, long16 ? a.v16 : a.v, nrows, kD, kS, long16))
    return cudaErrorInvalidValue;
  Params p{};
  p.q = static_cast<const __nv_bfloat16 *>(a.q);
  p.sel = a.sel;
  p.o_long_in = a.o_long_in;
  p.mix = a.mix;
  p.tab = static_cast<const float2 *>(a.tab);
  p.H = sh.H;
  p.N = sh.N;
  p.w = a.w;
  p.K = a.K;
  p.nblk = sh.nblk();
  p.nitems = sh.BH() * sh.nblk();
  p.sched = a.sched;
  p.timeline = a.timeline;
  p.rms_eps = a.rms_eps;
  p.nrows = nrows;
  p.out = a.out;
  p.err = a.err;
  // the three configurations the entry points use
  void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, Params);
  if (a.window && a.sel && !a.write_long)
    kern = fs_attn_tc_kernel<kFused>;
  else if (a.window && !a.sel && !a.write_long)
    kern = fs_attn_tc_kernel<kWindow>;
  else if (!a.window && a.sel && a.write_long)
    kern = fs_attn_tc_kernel<kLongOnly>;
  else
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = p.nitems < sm_count() ? p.nitems : sm_count();
  if (!p.timeline && g_timeline && g_timeline_entries >= 2 * grid) p.timeline = g_timeline;
  kern<<<grid, kThreads, kSmemBytes, st>>>(mkt, mv16, ck, cv, p);
  return cudaGetLastError();
}

}  // namespace fs
