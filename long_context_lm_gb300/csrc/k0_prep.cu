// k0_prep.cu -- window-branch operands, prepared once per call.
//
// FreeSolo (paper.rainbus.top summary, 方法步骤详情 ② window branch, 前置知识
// RoPE; ai.info summary, "Methodology in Plain English"): the sliding-window
// branch scores q_n . k_j after rotating both by their own positions (RoPE,
// half-split pairs (i, i + d/2) at angles p * theta_i, theta_i =
// base^(-2i/d)).  A key enters the windows of about (w + Bq) / Bq query
// tiles, so it is rotated here once, at its absolute position, instead of
// once per query tile inside the attention kernel:
//   kt[row] = [bf16 hi (64) | bf16 lo (64)] of R(n) k_n (fp32), 256 B per row
//   v16[row] = fp16(v_n) (exact from bf16 inside the fp16 range), 128 B per row
// Streaming, HBM-bound: per token-head it reads 256 B and writes 384 B.  The
// whole forward runs k0_prep_summary_kernel instead, which also writes the
// cell summaries of the keys it reads (8.1 B more per token-head), so that
// the keys are read once per call.
//
// Angles: row r < 64 of the table holds (cos, sin)(r theta_i); row 64 + u
// holds (cos, sin)(64 u theta_i), each from the angle reduced modulo 2 pi in
// fp64 and an fp32 sincospi; an absolute angle is composed from its two rows
// by the angle-sum identity in fp32 (error of a few fp32 ulps, independent of
// the position).
#include <cmath>

#include "cell_summary.cuh"
#include "fs_common.cuh"
#include "fs_internal.h"
#include "tc05.cuh"

namespace fs {
namespace {

// theta_i / pi in fp64, formed once on the host
struct Theta {
  double over_pi[kD / 2];
};

// Per entry one fp64 product reduced modulo 2 exactly and an fp32 sincospi of
// the remainder: the fp64 work is a multiply and a floor, not a trigonometric
// evaluation (fp64 throughput is small on this chip).  Entry error: the fp32
// rounding of the reduced angle (<= 2^-24 * pi rad) plus sincospif's ulp,
// against the fp64 reference values.
// `clear` (nullable): four status ints the caller's first kernel zeroes in
// place of a memset (the kernels that use them run after this one).
__global__ void __launch_bounds__(256) rope_table_kernel(float2 *__restrict__ tab, int rows,
                                                         const Theta th, int *clear) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (clear && idx < 4) clear[idx] = 0;
  if (idx >= rows * (kD / 2)) return;
  const int row = idx / (kD / 2), i = idx % (kD / 2);
  const double pos = row < 64 ? (double)row : 64.0 * (double)(row - 64);
  const double x = pos * th.over_pi[i];          // angle / pi
  const double r = x - 2.0 * floor(0.5 * x);     // in [0, 2), exact
  float sn, cs;
  sincospif((float)r, &sn, &cs);
  tab[idx] = make_float2(cs, sn);
}

// Four threads per token row; thread part p rotates pairs 8p .. 8p+7 (dims
// 8p.. and 32+8p..) and re-encodes value dims 16p .. 16p+15.  Eight rows per
// warp: every load and store instruction of a warp covers contiguous bytes.
__global__ void __launch_bounds__(256) k0_prep_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, const float4 *__restrict__ tab,
    int N, long long rows, uint4 *__restrict__ kt, uint4 *__restrict__ v16, int *err) {
  const long long nthreads = rows * 4;
  bool range_ok = true;
  for (long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x; t < nthreads;
       t += (long long)gridDim.x * blockDim.x) {
    const long long row = t >> 2;
    const int part = (int)(t & 3);
    const int n = (int)(row % N);
    const uint4 xa = __ldg(k + row * 8 + part), xb = __ldg(k + row * 8 + 4 + part);
    const uint4 va = __ldg(v + row * 8 + 2 * part), vb = __ldg(v + row * 8 + 2 * part + 1);
    // (cos, sin) pairs 8p..8p+7 of rows n mod 64 and 64 + n / 64: four float4 each
    const float4 *tr = tab + (size_t)(n & 63) * 16 + 4 * part;
    const float4 *tu = tab + (size_t)(64 + (n >> 6)) * 16 + 4 * part;
    const uint32_t wa[4] = {xa.x, xa.y, xa.z, xa.w}, wb[4] = {xb.x, xb.y, xb.z, xb.w};
    uint32_t ah[4], al[4], bh[4], bl[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // pairs 8p + 2j, 8p + 2j + 1
      const float4 rr = __ldg(tr + j), uu = __ldg(tu + j);
      float y0[2], y1[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float cr = e ? rr.z : rr.x, sr = e ? rr.w : rr.y;
        const float cu = e ? uu.z : uu.x, su = e ? uu.w : uu.y;
        const float c = fmaf(cu, cr, -su * sr), sn = fmaf(su, cr, cu * sr);
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
    uint4 *dst = kt + row * 16;
    dst[part] = make_uint4(ah[0], ah[1], ah[2], ah[3]);
    dst[4 + part] = make_uint4(bh[0], bh[1], bh[2], bh[3]);
    dst[8 + part] = make_uint4(al[0], al[1], al[2], al[3]);
    dst[12 + part] = make_uint4(bl[0], bl[1], bl[2], bl[3]);
    // values: bf16 -> fp16; a finite |v| >= 65520 would round to infinity
    const uint32_t vw[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
    uint32_t h[8];
    float big = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float lo = bf16_lo(vw[j]), hi = bf16_hi(vw[j]);
      big = fmaxf(big, fmaxf(fabsf(lo), fabsf(hi)));
      h[j] = pack_f16(lo, hi);
    }
    range_ok &= !(big >= 65520.f && big != INFINITY);
    uint4 *vd = v16 + row * 8 + 2 * part;
    vd[0] = make_uint4(h[0], h[1], h[2], h[3]);
    vd[1] = make_uint4(h[4], h[5], h[6], h[7]);
  }
  if (!range_ok) tc::report_error(err, FS_ERR_RANGE);
}

// The same pass with the cell summaries of the keys it reads (one read of
// the keys instead of two): one warp per 32-token cell, in the lane layout of
// cell_summary_warp (lane = 8 * t0 + g holds 16-byte chunk g of tokens
// t0 + 4i), so kbar and a_c are bit-identical to the summary kernel's.  A
// lane rotates the pairs of its chunk with the other half of each pair from
// lane ^ 4 (chunk g ^ 4 of the same tokens), by the arithmetic of
// k0_prep_kernel, so the rotated keys are bit-identical too; values are
// re-encoded chunk by chunk.
// Three blocks per SM (registers capped at 85, a few spilled), with the value
// loads issued after the summary: measured 132 us at 64k against 139 us for
// two blocks per SM with every load up front.
__global__ void __launch_bounds__(256, 3) k0_prep_summary_kernel(
    const uint4 *__restrict__ k, const uint4 *__restrict__ v, const float4 *__restrict__ tab,
    int N, long long ncells, uint4 *__restrict__ kt, uint4 *__restrict__ v16,
    float *__restrict__ kbar, float *__restrict__ amax, int *err) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long cell = (long long)blockIdx.x * 8 + warp;
  if (cell >= ncells) return;
  const int g = lane & 7, t0 = lane >> 3;
  const long long row0 = cell * kS;  // first token row of the cell (rows of all heads)
  uint4 kr[8], vr[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) kr[i] = __ldg(k + (row0 + t0 + 4 * i) * 8 + g);
  {
    float x[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t w[4] = {kr[i].x, kr[i].y, kr[i].z, kr[i].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[i][2 * j] = bf16_lo(w[j]);
        x[i][2 * j + 1] = bf16_hi(w[j]);
      }
    }
    cell_summary_warp(x, lane, kbar + cell * kD, amax + cell);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) vr[i] = __ldg(v + (row0 + t0 + 4 * i) * 8 + g);
  const bool first = g < 4;  // dims 8g.. are the first halves of their pairs
  const int pq = g & 3;      // pairs 8pq .. 8pq+7
  bool range_ok = true;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const long long row = row0 + t0 + 4 * i;
    const int n = (int)(row % N);
    const uint32_t mine[4] = {kr[i].x, kr[i].y, kr[i].z, kr[i].w};
    uint32_t other[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) other[j] = __shfl_xor_sync(0xffffffffu, mine[j], 4);
    const float4 *tr = tab + (size_t)(n & 63) * 16 + 4 * pq;
    const float4 *tu = tab + (size_t)(64 + (n >> 6)) * 16 + 4 * pq;
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // pairs 8pq + 2j, 8pq + 2j + 1
      const float4 rr = __ldg(tr + j), uu = __ldg(tu + j);
      const uint32_t wa = first ? mine[j] : other[j], wb = first ? other[j] : mine[j];
      float y[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float cr = e ? rr.z : rr.x, sr = e ? rr.w : rr.y;
        const float cu = e ? uu.z : uu.x, su = e ? uu.w : uu.y;
        const float c = fmaf(cu, cr, -su * sr), sn = fmaf(su, cr, cu * sr);
        const float x0 = e ? bf16_hi(wa) : bf16_lo(wa);
        const float x1 = e ? bf16_hi(wb) : bf16_lo(wb);
        y[e] = first ? fmaf(x0, c, -x1 * sn) : fmaf(x0, sn, x1 * c);
      }
      hw[j] = pack_bf16(y[0], y[1]);
      lw[j] = pack_bf16(y[0] - bf16_lo(hw[j]), y[1] - bf16_hi(hw[j]));
    }
    uint4 *dst = kt + row * 16;
    dst[g] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    dst[8 + g] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    // values: bf16 -> fp16; a finite |v| >= 65520 would round to infinity
    const uint32_t vw[4] = {vr[i].x, vr[i].y, vr[i].z, vr[i].w};
    uint32_t h[4];
    float big = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float lo = bf16_lo(vw[j]), hi = bf16_hi(vw[j]);
      big = fmaxf(big, fmaxf(fabsf(lo), fabsf(hi)));
      h[j] = pack_f16(lo, hi);
    }
    range_ok &= !(big >= 65520.f && big != INFINITY);
    v16[row * 8 + g] = make_uint4(h[0], h[1], h[2], h[3]);
  }
  if (!range_ok) tc::report_error(err, FS_ERR_RANGE);
}

}  // namespace

size_t rope_table_bytes(int N) { return (size_t)(64 + (N + 63) / 64) * (kD / 2) * sizeof(float2); }

cudaError_t launch_rope_table(void *tab, int N, float rope_base, cudaStream_t st, int *clear) {
  const int rows = 64 + (N + 63) / 64;
  Theta th;
  for (int i = 0; i < kD / 2; ++i)
    th.over_pi[i] = std::pow((double)rope_base, -2.0 * i / (double)kD) / 3.14159265358979323846;
  rope_table_kernel<<<(rows * (kD / 2) + 255) / 256, 256, 0, st>>>(static_cast<float2 *>(tab),
                                                                  rows, th, clear);
  return cudaGetLastError();
}

cudaError_t launch_prep_summary(const void *k, const void *v, const void *tab, const Shape &sh,
                                void *kt, void *v16, float *kbar, float *amax, int *err,
                                cudaStream_t st) {
  const long long ncells = (long long)sh.BH() * sh.C();
  k0_prep_summary_kernel<<<(unsigned)((ncells + 7) / 8), 256, 0, st>>>(
      static_cast<const uint4 *>(k), static_cast<const uint4 *>(v),
      static_cast<const float4 *>(tab), sh.N, ncells, static_cast<uint4 *>(kt),
      static_cast<uint4 *>(v16), kbar, amax, err);
  return cudaGetLastError();
}

cudaError_t launch_prep(const void *k, const void *v, const void *tab, const Shape &sh, void *kt,
                        void *v16, int *err, cudaStream_t st) {
  const long long rows = (long long)sh.BH() * sh.N;
  const long long blocks = (rows * 4 + 255) / 256;
  const int grid = (int)(blocks < 152 * 8 ? blocks : 152 * 8);
  k0_prep_kernel<<<grid, 256, 0, st>>>(static_cast<const uint4 *>(k),
                                       static_cast<const uint4 *>(v),
                                       static_cast<const float4 *>(tab), sh.N, rows,
                                       static_cast<uint4 *>(kt), static_cast<uint4 *>(v16), err);
  return cudaGetLastError();
}

}  // namespace fs
