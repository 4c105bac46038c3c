// k4_readout.cu -- NoPE sparse readout over the selected cells + RMSNorm.
//
// FreeSolo (paper.rainbus.top summary, 方法步骤详情 ⑥ "NoPE softmax then
// RMSNorm", 前置知识 NoPE; ai.info summary, "Key Contributions" 1): every
// query attends, without any rotation, to the original keys and values of
// its K selected cells (at most K*s = 128 tokens), and the branch output is
// RMS-normalised (no gain here).
//
// Masked block x union tiling.  The queries of one 128-query block pick their
// cells from the same small pool, so the union of their selections is small
// (about 7-18 cells on the synthetic workloads).  One CTA owns a block: it
// sorts the block's 128*K selections into the union list, records for every
// union cell which of each warp's 16 queries chose it, then streams the
// union's key/value cells (4 KB each, contiguous) through a cp.async double
// buffer.  Each warp runs legacy m16n8k16 MMAs for the 16 x 32 score tile
// only when one of its queries chose the cell, masks the others, and keeps a
// flash-style online softmax.  The probabilities are split into bf16 hi + lo
// halves for the P.V product so the result stays within fp32-grade error.
#include "fs_common.cuh"
#include "fs_internal.h"

namespace fs {

constexpr int kMaxSel = kBq * kMaxK;  // 1024 selections per block at most

struct ReadoutSmem {
  __nv_bfloat16 q[kBq * kD];                // 16 KB, swizzled rows
  __nv_bfloat16 kv[2][2][kS * kD];          // [stage][k|v] 2 x 2 x 4 KB
  int ids[kMaxSel];                         // sorted selections / union
  uint32_t mask[kMaxSel][8];                // per union cell, per warp: 16-bit row mask
  int nu;
};

__device__ __forceinline__ void load_cell_async(__nv_bfloat16 *dst_k, __nv_bfloat16 *dst_v,
                                                const __nv_bfloat16 *k, const __nv_bfloat16 *v,
                                                size_t cell_base, int tid) {
  // 32 rows x 8 chunks for k and for v: 512 16-byte pieces, two per thread
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int p = tid + it * 256;
    const int which = p >> 8, r = (p >> 3) & 31, ch = p & 7;
    const __nv_bfloat16 *src = (which ? v : k) + cell_base + (size_t)r * kD + ch * 8;
    char *dst = reinterpret_cast<char *>(which ? dst_v : dst_k) + swz128(r, ch);
    cp_async16(dst, src);
  }
}

__global__ void __launch_bounds__(256) k4_readout_kernel(
    const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
    const __nv_bfloat16 *__restrict__ v, const int32_t *__restrict__ sel, int N, int K,
    float rms_eps, float *__restrict__ o_long) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  ReadoutSmem &sm = *reinterpret_cast<ReadoutSmem *>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int beta = blockIdx.x, bh = blockIdx.y;
  const size_t head = (size_t)bh * N;
  const int b0 = beta * kBq;

  // ---- Q tile (unrotated) -> shared, swizzled
  for (int p = tid; p < kBq * 8; p += 256) {
    const int r = p >> 3, ch = p & 7;
    cp_async16(reinterpret_cast<char *>(sm.q) + swz128(r, ch), q + (head + b0 + r) * kD + ch * 8);
  }
  cp_async_commit();

  // ---- union of the block's selections: bitonic sort, then unique
  const int nsel = kBq * K;
  int nsort = 1;
  while (nsort < nsel) nsort <<= 1;
  // a selection outside [0, A) (no cell, or a cell the block may not read)
  // is ignored; A = cells that end at or before the block start
  const int A = beta * (kBq / kS);
  for (int i = tid; i < nsort; i += 256) {
    int c = 0x7fffffff;
    if (i < nsel) {
      const int x = sel[(head + b0) * K + i];
      c = (x >= 0 && x < A) ? x : 0x7fffffff;
    }
    sm.ids[i] = c;
  }
  __syncthreads();
  for (int kk = 2; kk <= nsort; kk <<= 1)
    for (int j = kk >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < nsort; i += 256) {
        const int p = i ^ j;
        if (p > i) {
          const int a = sm.ids[i], b = sm.ids[p];
          const bool asc = (i & kk) == 0;
          if ((a > b) == asc) {
            sm.ids[i] = b;
            sm.ids[p] = a;
          }
        }
      }
      __syncthreads();
    }
  if (warp == 0) {  // compact unique valid ids in place (reads stay ahead of writes)
    int nu = 0;
    for (int base = 0; base < nsort; base += 32) {
      const int i = base + lane;
      const int x = sm.ids[i];
      const bool keep = x != 0x7fffffff && (i == 0 || sm.ids[i - 1] != x);
      const uint32_t bal = __ballot_sync(0xffffffffu, keep);
      __syncwarp();
      if (keep) sm.ids[nu + __popc(bal & ((1u << lane) - 1))] = x;
      nu += __popc(bal);
      __syncwarp();
    }
    if (lane == 0) sm.nu = nu;
  }
  __syncthreads();
  const int nu = sm.nu;
  for (int i = tid; i < nu * 8; i += 256) (&sm.mask[0][0])[i] = 0u;
  __syncthreads();
  for (int i = tid; i < nsel; i += 256) {
    const int c = sel[(head + b0) * K + i];
    if (c < 0 || c >= A) continue;
    int lo = 0, hi = nu - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (sm.ids[mid] < c) lo = mid + 1; else hi = mid;
    }
    const int qr = i / K;
    atomicOr(&sm.mask[lo][qr >> 4], 1u << (qr & 15));
  }

  // ---- Q fragments
  cp_async_wait<0>();
  __syncthreads();
  uint32_t qa[4][4];
  {
    const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
    for (int kc = 0; kc < 4; ++kc) {
      const int ch = 2 * kc + (lane >> 4);
      ldsm_x4(qa[kc][0], qa[kc][1], qa[kc][2], qa[kc][3], smem_u32(sm.q) + swz128(r, ch));
    }
  }

  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const float sl2 = 1.4426950408889634f * rsqrtf((float)kD);
  const int g = lane >> 2, t = lane & 3;

  if (nu > 0) load_cell_async(sm.kv[0][0], sm.kv[0][1], k, v, (head + (size_t)sm.ids[0] * kS) * kD, tid);
  cp_async_commit();
  for (int ui = 0; ui < nu; ++ui) {
    const int stg = ui & 1;
    if (ui + 1 < nu)
      load_cell_async(sm.kv[stg ^ 1][0], sm.kv[stg ^ 1][1], k, v,
                      (head + (size_t)sm.ids[ui + 1] * kS) * kD, tid);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint32_t m = sm.mask[ui][warp];
    if (m != 0u) {
      const uint32_t kb = smem_u32(sm.kv[stg][0]), vb = smem_u32(sm.kv[stg][1]);
      float s[4][4];
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int kc = 0; kc < 4; ++kc)
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          uint32_t b0, b1, b2, b3;
          const int r = np * 16 + (lane & 7) + ((lane >> 4) << 3);
          const int ch = 2 * kc + ((lane >> 3) & 1);
          ldsm_x4(b0, b1, b2, b3, kb + swz128(r, ch));
          mma_bf16_16816(s[2 * np], qa[kc], b0, b1);
          mma_bf16_16816(s[2 * np + 1], qa[kc], b2, b3);
        }
      const bool valid[2] = {((m >> g) & 1u) != 0u, ((m >> (g + 8)) & 1u) != 0u};
      float alpha[2];
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) mx = fmaxf(mx, fmaxf(s[nt][2 * hr], s[nt][2 * hr + 1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mnew = valid[hr] ? fmaxf(mrow[hr], mx * sl2) : mrow[hr];
        alpha[hr] = (valid[hr] && mrow[hr] != -INFINITY) ? exp2f(mrow[hr] - mnew) : 1.f;
        if (valid[hr] && mrow[hr] == -INFINITY) alpha[hr] = 0.f;
        mrow[hr] = mnew;
        float ls = 0.f;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float p = valid[hr] ? exp2f(s[nt][2 * hr + e] * sl2 - mnew) : 0.f;
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
      // P (16 x 32) as bf16 hi + lo A fragments, two 16-key chunks
      uint32_t ph[2][4], plo[2][4];
#pragma unroll
      for (int kc = 0; kc < 2; ++kc)
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            const float x0 = s[2 * kc + hf][2 * hr], x1 = s[2 * kc + hf][2 * hr + 1];
            const uint32_t hi = pack_bf16(x0, x1);
            ph[kc][hf * 2 + hr] = hi;
            plo[kc][hf * 2 + hr] = pack_bf16(x0 - bf16_lo(hi), x1 - bf16_hi(hi));
          }
#pragma unroll
      for (int kc = 0; kc < 2; ++kc)
#pragma unroll
        for (int dp = 0; dp < 4; ++dp) {
          uint32_t b0, b1, b2, b3;
          const int r = kc * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
          const int ch = 2 * dp + (lane >> 4);
          ldsm_x4_t(b0, b1, b2, b3, vb + swz128(r, ch));
          mma_bf16_16816(o[2 * dp], ph[kc], b0, b1);
          mma_bf16_16816(o[2 * dp + 1], ph[kc], b2, b3);
          mma_bf16_16816(o[2 * dp], plo[kc], b0, b1);
          mma_bf16_16816(o[2 * dp + 1], plo[kc], b2, b3);
        }
    }
    __syncthreads();
  }

  // ---- epilogue: normalise, RMSNorm, store fp32
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    lrow[hr] += __shfl_xor_sync(0xffffffffu, lrow[hr], 1);
    lrow[hr] += __shfl_xor_sync(0xffffffffu, lrow[hr], 2);
    const float inv = lrow[hr] > 0.f ? 1.f / lrow[hr] : 0.f;
    float ss = 0.f;
#pragma unroll
    for (int dt = 0; dt < 8; ++dt) {
      o[dt][2 * hr] *= inv;
      o[dt][2 * hr + 1] *= inv;
      ss = fmaf(o[dt][2 * hr], o[dt][2 * hr], ss);
      ss = fmaf(o[dt][2 * hr + 1], o[dt][2 * hr + 1], ss);
    }
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    const float rn = lrow[hr] > 0.f ? rsqrtf(ss / kD + rms_eps) : 0.f;
    const int n = b0 + warp * 16 + g + 8 * hr;
    float *dst = o_long + (head + n) * kD;
#pragma unroll
    for (int dt = 0; dt < 8; ++dt)
      *reinterpret_cast<float2 *>(dst + dt * 8 + 2 * t) =
          make_float2(o[dt][2 * hr] * rn, o[dt][2 * hr + 1] * rn);
  }
}

cudaError_t launch_readout(const void *q, const void *k, const void *v, const int32_t *sel,
                           const Shape &sh, int K, float rms_eps, float *o_long,
                           cudaStream_t st) {
  const size_t smem = sizeof(ReadoutSmem);
  cudaFuncSetAttribute(k4_readout_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  dim3 grid(sh.nblk(), sh.BH());
  k4_readout_kernel<<<grid, 256, smem, st>>>(
      static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
      static_cast<const __nv_bfloat16 *>(v), sel, sh.N, K, rms_eps, o_long);
  return cudaGetLastError();
}

}  // namespace fs
