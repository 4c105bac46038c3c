// fs_internal.h -- launchers shared between the kernel files and the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fs {

struct Shape {
  int batch, H, N, d;
  int BH() const { return batch * H; }
  int C() const { return N / 32; }
  int nblk() const { return N / 128; }
};

cudaError_t launch_round_bf16(const float *src, void *dst, size_t n, cudaStream_t st);
cudaError_t launch_cell_summary(const void *k, bool f32, const Shape &sh, float *kbar,
                                float *amax, cudaStream_t st);
size_t prune_workspace_bytes(const Shape &sh);
cudaError_t launch_prune(const float *amax, const Shape &sh, int P, int W, int32_t *pool,
                         int32_t *pool_count, void *ws, cudaStream_t st);
cudaError_t launch_select(const void *q, const float *kbar, const float *amax,
                          const int32_t *pool, const int32_t *pool_count, const float *lambda,
                          const float *sigma, const Shape &sh, int K, int cap, int W,
                          bool fs_mode, int32_t *sel, float *sel_score, int *err,
                          cudaStream_t st);
// RoPE angle table (rope_table_bytes(N) of device memory, written by
// launch_rope_table) and the window operands prepared from it: kt = rotated
// keys [rows, 128] bf16 (hi | lo), v16 = values [rows, 64] fp16.
size_t rope_table_bytes(int N);
cudaError_t launch_rope_table(void *tab, int N, float rope_base, cudaStream_t st,
                              int *clear = nullptr);
// k0_prep with the cell summaries of the same keys (one read of k).
cudaError_t launch_prep_summary(const void *k, const void *v, const void *tab, const Shape &sh,
                                void *kt, void *v16, float *kbar, float *amax, int *err,
                                cudaStream_t st);
cudaError_t launch_prep(const void *k, const void *v, const void *tab, const Shape &sh, void *kt,
                        void *v16, int *err, cudaStream_t st);
// Both attention branches (window RoPE branch, NoPE readout of the selected
// cells) in one persistent tcgen05 kernel.  window: run the window branch
// (reads kt, v16, tab); sel != nullptr: run the long branch (reads the raw
// k, v cells); write_long: write RMSNorm(o_long) to `out` instead of the
// mixed output; o_long_in (window only, nullable): a precomputed long branch
// to mix in.
struct AttnArgs {
  Shape sh;
  const void *q, *k, *v;
  const void *kt, *v16, *tab;
  const int32_t *sel;
  const float *o_long_in;
  const float *mix;
  int w, K;
  float rms_eps;
  bool window, write_long;
  float *out;
  int *err;
  int *sched;  // nullable: two ints, zero at launch, left zero (q-tile tickets)
  long long *timeline;  // nullable: per CTA, global-timer ns at its start and end
};
cudaError_t launch_attn_tc(const AttnArgs &a, cudaStream_t st);
// Per-CTA timeline of the calling host thread's next attention launches
// (fs_set_attention_timeline): buffer and its length in int64 entries.
void set_attention_timeline(long long *timeline, int entries);
// Bounded decode state (see k6_decode.cu): a global part (256-byte header
// whose first int is the error word, then the relative-angle tables), then
// one fixed-size block per (batch, head).  Offsets inside a head's block.
constexpr int kDecodeHeaderInts = 192;  // counts and slot lists of one head
constexpr int kDecodeTabRows = 64 + 16;  // (cos, sin)(o theta): o = r < 64, o = 64a, a < 16
struct DecodeLayout {
  int w, P, W, K, pend, nslots;
  size_t hdr, slot_cell, slot_amax, slot_kbar, slot_k, slot_v, ring_k, ring_v;
  size_t head_bytes;              // one (batch, head)
  size_t tab, global_bytes;       // angle tables inside the global part; its size
  size_t total(int BH) const { return global_bytes + (size_t)BH * head_bytes; }
};
DecodeLayout decode_layout(int w, int P, int W, int K);
size_t decode_smem_bytes(const DecodeLayout &L);
cudaError_t launch_decode_init(const void *k, const void *v, const float *kbar, const float *amax,
                               const int32_t *pool, const int32_t *pool_count, int BH, int N,
                               int N0, float rope_base, const DecodeLayout &L, void *state,
                               cudaStream_t st);
// One decode step for token t of every (batch, head).
struct DecodeArgs {
  const void *q_t, *k_t, *v_t;
  void *state;
  const float *lambda, *sigma, *mix;
  DecodeLayout L;
  int batch, H, t;
  float rms_eps;
  float *out;
  int32_t *sel_out;
};
cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t st);

// Shared q / k / v projection (k7_qkv.cu): RMSNorm row scale, gain folded
// into the weights, one tcgen05 GEMM writing q, k, v [batch, H, N, 64] bf16.
struct QkvArgs {
  const void *x;      // [batch, N, D] bf16
  const float *gain;  // [D] or null (ones)
  const void *w;      // [3*H*64, D] bf16
  int batch, N, D, H;
  float eps;
  void *q, *k, *v;
  void *ws;           // qkv_workspace_bytes
  int *err;
};
size_t qkv_workspace_bytes(int M, int D, int H);
// FS-B forests (k9_fsb.cu): per (batch, head) two leaf lists (all cells;
// cells with a_c > tau), the tau forest's prefix count, then per forest the
// node means [nodes, 64] and (radius, a_max, first cell, -) [nodes].
constexpr int kFsbMaxLevels = 24;
struct FsbLayout {
  int C, levels, nodes;
  int level_off[kFsbMaxLevels];
  size_t list, hcount, mean, meta, head_bytes;
};
FsbLayout fsb_layout(int C);
cudaError_t launch_fsb(const void *q, const void *k, const float *kbar, const float *amax,
                       const float *lambda, const float *sigma, const Shape &sh, int K, int beam,
                       float tau, void *ws, int32_t *sel, cudaStream_t st);
// Gradients of the forward (k8_backward.cu), from the forward's selection.
struct BwdArgs {
  Shape sh;
  const void *q, *k, *v;   // bf16
  const float *g;          // dL/dout
  const int32_t *sel;      // the forward's selection [BH, N, K]
  const float *mix;
  int w, K;
  float rope_base, rms_eps;
  float *dq, *dk, *dv, *dmix;
  void *ws;                // backward_workspace_bytes
  int *err;                // bounded-wait failures (FS_ERR_TIMEOUT)
};
size_t backward_workspace_bytes(const Shape &sh);
cudaError_t launch_backward(const BwdArgs &a, cudaStream_t st);
cudaError_t launch_qkv(const QkvArgs &a, cudaStream_t st);

}  // namespace fs
