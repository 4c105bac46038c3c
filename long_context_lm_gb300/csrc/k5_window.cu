// k5_window.cu -- sliding-window RoPE branch with the branch mix fused into
// the epilogue (legacy warp-MMA version).
//
// FreeSolo (paper.rainbus.top summary, 方法步骤详情 ② "在 w=512 窗口内做
// RoPE 注意力" and ⑥ "与局部分支相加"; 前置知识 RoPE; ai.info summary,
// "Methodology in Plain English": an ordinary 512-token sliding window with
// RoPE, whose output is added to the long branch with a per-head weight):
//     o_win[n] = softmax_j((R(n) q_n . R(j) k_j) / sqrt(d)) v_j,  j in [n-w+1, n]
//     out[n]   = o_win[n] + mix_h * o_long[n].
//
// One CTA per (head, 128-query tile); eight warps own 16 query rows each.
// Keys stream in 64-key tiles through a cp.async double buffer; each tile is
// rotated once in shared memory.  The rotated q and k are split into bf16
// hi + lo halves and the logits take three MMAs (hi.hi + hi.lo + lo.hi): a
// plain bf16 rounding of the rotated vectors alone exceeds the output
// tolerance on lognormal keys.  Probabilities enter P.V as bf16.
//
// RoPE angles: theta_i = base^(-2i/d); the angle n*theta_i is formed from two
// small fp32 tables computed in fp64 (n = 128*hi + lo, angle-sum identity),
// so positions up to 2^24 keep ~1e-7 accuracy without fp64 in the hot loop.
#include "fs_common.cuh"
#include "fs_internal.h"

namespace fs {

constexpr int kKT = 64;  // keys per tile

__global__ void rope_tables_kernel(float2 *__restrict__ t_hi, int n_hi, float2 *__restrict__ t_lo,
                                   double base) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  const int half = kD / 2;
  const int total = (n_hi + kBq) * half;
  if (idx >= total) return;
  const int row = idx / half, i = idx % half;
  const double theta = pow(base, -2.0 * (double)i / (double)kD);
  const bool hi = row < n_hi;
  const double pos = hi ? (double)row * kBq : (double)(row - n_hi);
  double s, c;
  sincos(pos * theta, &s, &c);
  (hi ? t_hi[row * half + i] : t_lo[(row - n_hi) * half + i]) = make_float2((float)c, (float)s);
}

// Rotate 8 pairs (dims 8*ig .. 8*ig+7 with their partners +32) of one row at
// position n and write bf16 hi / lo halves into two swizzled tiles.
__device__ __forceinline__ void rope_row_group(const uint4 xa, const uint4 xb, int n, int ig,
                                               const float2 *__restrict__ t_hi,
                                               const float2 *__restrict__ t_lo, char *dst_hi,
                                               char *dst_lo, int r) {
  const float4 *th = reinterpret_cast<const float4 *>(t_hi + (size_t)(n >> 7) * (kD / 2) + 8 * ig);
  const float4 *tl = reinterpret_cast<const float4 *>(t_lo + (size_t)(n & 127) * (kD / 2) + 8 * ig);
  const uint32_t wa[4] = {xa.x, xa.y, xa.z, xa.w}, wb[4] = {xb.x, xb.y, xb.z, xb.w};
  uint32_t ya_hi[4], ya_lo[4], yb_hi[4], yb_lo[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float4 h = __ldg(th + j), l = __ldg(tl + j);  // two (cos, sin) pairs each
    float y0[2], y1[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float ch = e ? h.z : h.x, sh = e ? h.w : h.y;
      const float cl = e ? l.z : l.x, sl = e ? l.w : l.y;
      const float c = ch * cl - sh * sl, s = sh * cl + ch * sl;
      const float x0 = e ? bf16_hi(wa[j]) : bf16_lo(wa[j]);
      const float x1 = e ? bf16_hi(wb[j]) : bf16_lo(wb[j]);
      y0[e] = x0 * c - x1 * s;
      y1[e] = x0 * s + x1 * c;
    }
    ya_hi[j] = pack_bf16(y0[0], y0[1]);
    ya_lo[j] = pack_bf16(y0[0] - bf16_lo(ya_hi[j]), y0[1] - bf16_hi(ya_hi[j]));
    yb_hi[j] = pack_bf16(y1[0], y1[1]);
    yb_lo[j] = pack_bf16(y1[0] - bf16_lo(yb_hi[j]), y1[1] - bf16_hi(yb_hi[j]));
  }
  *reinterpret_cast<uint4 *>(dst_hi + swz128(r, ig)) = make_uint4(ya_hi[0], ya_hi[1], ya_hi[2], ya_hi[3]);
  *reinterpret_cast<uint4 *>(dst_hi + swz128(r, ig + 4)) = make_uint4(yb_hi[0], yb_hi[1], yb_hi[2], yb_hi[3]);
  *reinterpret_cast<uint4 *>(dst_lo + swz128(r, ig)) = make_uint4(ya_lo[0], ya_lo[1], ya_lo[2], ya_lo[3]);
  *reinterpret_cast<uint4 *>(dst_lo + swz128(r, ig + 4)) = make_uint4(yb_lo[0], yb_lo[1], yb_lo[2], yb_lo[3]);
}

struct WindowSmem {
  __nv_bfloat16 qhi[kBq * kD], qlo[kBq * kD];  // 32 KB
  __nv_bfloat16 kraw[2][kKT * kD];              // 16 KB
  __nv_bfloat16 vraw[2][kKT * kD];              // 16 KB
  __nv_bfloat16 khi[kKT * kD], klo[kKT * kD];   // 16 KB
};

__global__ void __launch_bounds__(256) k5_window_kernel(
    const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
    const __nv_bfloat16 *__restrict__ v, const float *__restrict__ o_long,
    const float *__restrict__ mix, const float2 *__restrict__ t_hi,
    const float2 *__restrict__ t_lo, int H, int N, int w, float *__restrict__ out) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  WindowSmem &sm = *reinterpret_cast<WindowSmem *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int beta = blockIdx.x, bh = blockIdx.y, h = bh % H;
  const size_t head = (size_t)bh * N;
  const int b0 = beta * kBq;

  // key tiles covering [max(0, b0-w+1), b0+127]
  const int kt_first = max(0, b0 - w + 1) / kKT * kKT;
  const int ntiles = (b0 + kBq - kt_first) / kKT;

  auto load_tile = [&](int it) {
    const int kt = kt_first + it * kKT;
    const int stg = it & 1;
#pragma unroll
    for (int rep = 0; rep < 4; ++rep) {
      const int p = tid + rep * 256;  // 0..1023: 512 pieces of k, then 512 of v
      const int which = p >> 9, r = (p >> 3) & 63, ch = p & 7;
      const __nv_bfloat16 *src = (which ? v : k) + (head + kt + r) * kD + ch * 8;
      cp_async16(reinterpret_cast<char *>(which ? sm.vraw[stg] : sm.kraw[stg]) + swz128(r, ch), src);
    }
  };

  // raw Q into the hi tile, then rotate in place (each thread owns its pieces)
  for (int p = tid; p < kBq * 8; p += 256) {
    const int r = p >> 3, ch = p & 7;
    cp_async16(reinterpret_cast<char *>(sm.qhi) + swz128(r, ch), q + (head + b0 + r) * kD + ch * 8);
  }
  load_tile(0);
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  for (int p = tid; p < kBq * 4; p += 256) {
    const int r = p >> 2, ig = p & 3;
    const char *src = reinterpret_cast<const char *>(sm.qhi);
    const uint4 xa = *reinterpret_cast<const uint4 *>(src + swz128(r, ig));
    const uint4 xb = *reinterpret_cast<const uint4 *>(src + swz128(r, ig + 4));
    rope_row_group(xa, xb, b0 + r, ig, t_hi, t_lo, reinterpret_cast<char *>(sm.qhi),
                   reinterpret_cast<char *>(sm.qlo), r);
  }
  __syncthreads();
  uint32_t qh[4][4], ql[4][4];
  {
    const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int kc = 0; kc < 4; ++kc) {
      const int ch = 2 * kc + (lane >> 4);
      ldsm_x4(qh[kc][0], qh[kc][1], qh[kc][2], qh[kc][3], smem_u32(sm.qhi) + swz128(r, ch));
      ldsm_x4(ql[kc][0], ql[kc][1], ql[kc][2], ql[kc][3], smem_u32(sm.qlo) + swz128(r, ch));
    }
  }

  const int g = lane >> 2, t = lane & 3;
  const int n0 = b0 + warp * 16;
  const int nrow[2] = {n0 + g, n0 + g + 8};
  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const float sl2 = 1.4426950408889634f * rsqrtf((float)kD);

  for (int it = 0; it < ntiles; ++it) {
    const int kt = kt_first + it * kKT;
    if (it + 1 < ntiles) load_tile(it + 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    {  // rotate this tile's keys: 64 rows x 4 groups, one per thread
      const int r = tid >> 2, ig = tid & 3;
      const char *src = reinterpret_cast<const char *>(sm.kraw[it & 1]);
      const uint4 xa = *reinterpret_cast<const uint4 *>(src + swz128(r, ig));
      const uint4 xb = *reinterpret_cast<const uint4 *>(src + swz128(r, ig + 4));
      rope_row_group(xa, xb, kt + r, ig, t_hi, t_lo, reinterpret_cast<char *>(sm.khi),
                     reinterpret_cast<char *>(sm.klo), r);
    }
    __syncthreads();
    const bool skip = (kt > n0 + 15) || (kt + kKT - 1 < n0 - w + 1);
    if (!skip) {
      const bool need_mask = !((kt + kKT - 1 <= n0) && (kt > n0 + 15 - w));
      float s[8][4];
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
      const uint32_t khb = smem_u32(sm.khi), klb = smem_u32(sm.klo);
#pragma unroll
      for (int kc = 0; kc < 4; ++kc)
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          const int r = np * 16 + (lane & 7) + ((lane >> 4) << 3);
          const int ch = 2 * kc + ((lane >> 3) & 1);
          uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
          ldsm_x4(h0, h1, h2, h3, khb + swz128(r, ch));
          ldsm_x4(l0, l1, l2, l3, klb + swz128(r, ch));
          mma_bf16_16816(s[2 * np], qh[kc], h0, h1);
          mma_bf16_16816(s[2 * np + 1], qh[kc], h2, h3);
          mma_bf16_16816(s[2 * np], qh[kc], l0, l1);
          mma_bf16_16816(s[2 * np + 1], qh[kc], l2, l3);
          mma_bf16_16816(s[2 * np], ql[kc], h0, h1);
          mma_bf16_16816(s[2 * np + 1], ql[kc], h2, h3);
        }
      float alpha[2];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            float x = s[nt][2 * hr + e] * sl2;
            if (need_mask) {
              const int j = kt + nt * 8 + 2 * t + e;
              if (j > nrow[hr] || j <= nrow[hr] - w) x = -INFINITY;
            }
            s[nt][2 * hr + e] = x;
            mx = fmaxf(mx, x);
          }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mnew = fmaxf(mrow[hr], mx);
        const float muse = mnew == -INFINITY ? 0.f : mnew;
        alpha[hr] = exp2f(mrow[hr] - muse);
        mrow[hr] = mnew;
        float ls = 0.f;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float p = exp2f(s[nt][2 * hr + e] - muse);
            s[nt][2 * hr + e] = p;
            ls += p;
          }
        lrow[hr] = lrow[hr] * alpha[hr] + ls;
      }
#pragma unroll
      for (int dt = 0; dt < 8; ++dt) {
        o[dt][0] *= alpha[0];
        o[dt][1] *= alpha[0];
        o[dt][2] *= alpha[1];
        o[dt][3] *= alpha[1];
      }
      const uint32_t vb = smem_u32(sm.vraw[it & 1]);
#pragma unroll
      for (int kc = 0; kc < 4; ++kc) {
        uint32_t pa[4];
        pa[0] = pack_bf16(s[2 * kc][0], s[2 * kc][1]);
        pa[1] = pack_bf16(s[2 * kc][2], s[2 * kc][3]);
        pa[2] = pack_bf16(s[2 * kc + 1][0], s[2 * kc + 1][1]);
        pa[3] = pack_bf16(s[2 * kc + 1][2], s[2 * kc + 1][3]);
#pragma unroll
        for (int dp = 0; dp < 4; ++dp) {
          uint32_t b0, b1, b2, b3;
          const int r = kc * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
          const int ch = 2 * dp + (lane >> 4);
          ldsm_x4_t(b0, b1, b2, b3, vb + swz128(r, ch));
          mma_bf16_16816(o[2 * dp], pa, b0, b1);
          mma_bf16_16816(o[2 * dp + 1], pa, b2, b3);
        }
      }
    }
    __syncthreads();
  }

  const float mh = mix ? mix[h] : 0.f;
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    lrow[hr] += __shfl_xor_sync(0xffffffffu, lrow[hr], 1);
    lrow[hr] += __shfl_xor_sync(0xffffffffu, lrow[hr], 2);
    const float inv = 1.f / lrow[hr];
    const int n = nrow[hr];
    float *dst = out + (head + n) * kD;
    const float *ol = o_long ? o_long + (head + n) * kD : nullptr;
#pragma unroll
    for (int dt = 0; dt < 8; ++dt) {
      float2 r = make_float2(o[dt][2 * hr] * inv, o[dt][2 * hr + 1] * inv);
      if (ol) {
        const float2 x = *reinterpret_cast<const float2 *>(ol + dt * 8 + 2 * t);
        r.x = fmaf(mh, x.x, r.x);
        r.y = fmaf(mh, x.y, r.y);
      }
      *reinterpret_cast<float2 *>(dst + dt * 8 + 2 * t) = r;
    }
  }
}

size_t rope_table_bytes(const Shape &sh) {
  return ((size_t)(sh.N + kBq - 1) / kBq + kBq) * (kD / 2) * sizeof(float2);
}

cudaError_t launch_rope_tables(const Shape &sh, float base, float2 *tables, cudaStream_t st) {
  const int n_hi = (sh.N + kBq - 1) / kBq;
  const int total = (n_hi + kBq) * (kD / 2);
  rope_tables_kernel<<<(total + 255) / 256, 256, 0, st>>>(tables, n_hi,
                                                          tables + (size_t)n_hi * (kD / 2),
                                                          (double)base);
  return cudaGetLastError();
}

cudaError_t launch_window(const void *q, const void *k, const void *v, const float *o_long,
                          const float *mix, const float2 *tables, const Shape &sh, int w,
                          float *out, cudaStream_t st) {
  const size_t smem = sizeof(WindowSmem);
  cudaFuncSetAttribute(k5_window_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  const int n_hi = (sh.N + kBq - 1) / kBq;
  dim3 grid(sh.nblk(), sh.BH());
  k5_window_kernel<<<grid, 256, smem, st>>>(
      static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
      static_cast<const __nv_bfloat16 *>(v), o_long, mix, tables, tables + (size_t)n_hi * (kD / 2),
      sh.H, sh.N, w, out);
  return cudaGetLastError();
}

}  // namespace fs
