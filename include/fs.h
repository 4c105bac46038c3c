/*
 * fs.h -- C ABI of the GB300 (sm_103a) FreeSolo FS-L attention forward.
 *
 * Method: "FreeSolo: Linear-time Sparse Attention with Zero-Shot Length
 * Extrapolation", as summarised on paper.rainbus.top (sections 核心方法 and
 * 方法步骤详情 ②-⑥) and ai.info (section "Methodology in Plain English").
 * Every head has a w-token sliding-window RoPE branch and a long-range NoPE
 * branch that reads the tokens of K selected s-token key cells; the two are
 * added with a per-head weight.
 *
 * Conventions shared by every entry point
 *  - Tensors are DEVICE pointers to contiguous row-major arrays owned by the
 *    caller.  q, k, v are [batch, H, N, d]; per-head parameter arrays are
 *    [H] float32 device arrays.
 *  - The library never allocates or frees memory.  Scratch comes from a
 *    caller-provided device workspace sized by fs_workspace_bytes().
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls only enqueue work on it and return without
 *    synchronising; a returned FS_OK means the arguments were valid and the
 *    launches were accepted.
 *  - Arguments are validated before anything is launched: a NULL pointer, a
 *    non-positive size, N not a multiple of Bq or Bq not a multiple of s
 *    give FS_ERR_INVALID_ARG; shapes the kernels are not built for (d != 64,
 *    s != 32, Bq != 128, P > 64, K > 8, w outside [1, 1024], N > 2^24 or
 *    batch*H*N >= 2^31) give
 *    FS_ERR_UNSUPPORTED.  A CUDA launch error gives FS_ERR_CUDA.  No call
 *    throws across the ABI.
 *  - Cell c covers tokens [c*s, (c+1)*s); C = N/s.  Query block beta covers
 *    queries [beta*Bq, (beta+1)*Bq); a cell is available to the block iff it
 *    ends at or before beta*Bq.
 */
#ifndef FS_H_
#define FS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FS_OK = 0,
  FS_ERR_INVALID_ARG = 1,
  FS_ERR_UNSUPPORTED = 2,
  FS_ERR_CUDA = 3,
  FS_ERR_TIMEOUT = 4,
  FS_ERR_RANGE = 5, /* a finite value of v read by the window branch has
                       |v| >= 65520: past the fp16 range of its P.V product */
  FS_ERR_SCRATCH_LIMIT = 6, /* fs_prune_cells_static: the shape needs more
                               than its fixed scratch array */
  FS_ERR_STATE = 7 /* fs_decode_step: the decode state is not at the step's
                      position t */
} fs_status;

typedef enum { FS_BF16 = 0, FS_FP32 = 1 } fs_dtype;

/* FS-L prunes the prefix to P + W cells per block; FS scores the whole
 * available prefix (quadratic); FS-B keeps every cell and selects by beam
 * search over two causal forests (paper.rainbus.top summary, 核心方法 and
 * 方法步骤详情 ⑤; ai.info "Methodology in Plain English"). */
typedef enum { FS_MODE_FSL = 0, FS_MODE_FS = 1, FS_MODE_FSB = 2 } fs_mode;

/* Method parameters.  Page values: w=512, s=32, K=4, P=64, W=8, Bq=128
 * (paper.rainbus.top summary, 核心方法); rope_base=10000 and rms_eps=1e-6 are
 * readings (the pages give neither). */
typedef struct {
  int w;           /* window keys, self included: [n-w+1, n]           */
  int s;           /* tokens per cell                                    */
  int K;           /* cells read per query                               */
  int P;           /* FS-L: older cells kept by largest max key norm     */
  int W;           /* FS-L: most recent available cells always kept      */
  int Bq;          /* query block sharing one availability set           */
  float rope_base; /* theta_i = rope_base^(-2i/d), half-split pairing    */
  float rms_eps;   /* RMSNorm epsilon of the long-branch output          */
  int mode;        /* fs_mode                                            */
  int beam;        /* FS-B: nodes kept per level of each forest (1..16)  */
  float tau;       /* FS-B: the second forest holds the cells a_c > tau  */
} fs_params;

/* Fills the page values above (FS-B: beam 16; tau 0, an input the pages
 * calibrate per model as a median cell norm). */
void fs_default_params(fs_params *p);

/* Human-readable name of a status code (static string). */
const char *fs_status_string(int status);

/* Description of the CUDA error behind the calling thread's most recent
 * FS_ERR_CUDA (static string; "no error" if there was none). */
const char *fs_last_cuda_error(void);

/* Diagnostics (no counterpart on the pages): each CTA of the attention
 * kernel launches that the calling host thread makes next (inside
 * fs_attention_fwd, fs_window_attn and fs_sparse_readout) writes the device's
 * global timer, in ns, at its start and at its end into timeline[2 * cta] and
 * timeline[2 * cta + 1]: the spread of the CTAs' finish times shows how well
 * the q-tiles were balanced.  timeline is device memory of `entries` int64,
 * owned by the caller, which must keep it allocated until it turns the
 * timeline off again (the library keeps only the pointer); a launch of more
 * than entries / 2 CTAs records nothing.  (NULL, 0) turns it off.  FS_ERR_INVALID_ARG when exactly one of
 * timeline and entries is zero, or entries < 0. */
int fs_set_attention_timeline(long long *timeline, int entries);

/* Device workspace bytes fs_attention_fwd needs for this shape (includes the
 * bf16 staging copies of q, k, v when dtype is FS_FP32).  0 on bad args. */
size_t fs_workspace_bytes(int batch, int H, int N, int d, const fs_params *p,
                          int dtype);

/* Workspace bytes fs_prune_cells needs (per-chunk running lists). */
size_t fs_prune_workspace_bytes(int batch, int H, int N, const fs_params *p);

/* Cell summaries (paper.rainbus.top summary, 方法步骤详情 ③; ai.info,
 * "Key Contributions" 2): for every cell of every (batch, head)
 *   kbar[c] = (1/s) * sum of the cell's s unrotated keys      [batch,H,C,d] f32
 *   amax[c] = max over the cell's tokens of ||k_t||_2          [batch,H,C]   f32
 * k is bf16 (dtype FS_BF16) or float32 (FS_FP32, rounded to bf16 first). */
int fs_cell_summarize(const void *k, int dtype, int batch, int H, int N, int d,
                      int s, float *kbar, float *amax, void *stream);

/* FS-L availability sets (paper.rainbus.top summary, 方法步骤详情 ④; ai.info,
 * "Methodology in Plain English": 8 recent plus the 64 highest-norm cells,
 * updated only at query-block boundaries).  For every query block beta with
 * A = beta*Bq/s available cells, the pool is the min(W, A) newest available
 * cells plus the top-P older cells ranked by (amax desc, index asc).
 *   amax        [batch,H,C] f32 (from fs_cell_summarize)
 *   pool        [batch,H,N/Bq,P+W] int32: recent cells ascending, then the
 *               kept older cells in rank order; unused slots are -1
 *   pool_count  [batch,H,N/Bq] int32
 *   ws          device scratch of fs_prune_workspace_bytes() bytes
 * Linear in N: per 64-cell chunk sorted lists and a prefix merge.
 * mode must be FS_MODE_FSL (FS needs no pool). */
int fs_prune_cells(const float *amax, int batch, int H, int N,
                   const fs_params *p, int32_t *pool, int32_t *pool_count,
                   void *ws, size_t ws_bytes, void *stream);

/* Decoding from a bounded state (paper.rainbus.top summary, 核心方法: linear
 * prefill, constant-size decode state; 实验结果: constant attention buffer
 * from 4k to 256k; ai.info "Methodology in Plain English": a bounded pool of
 * 8 recent plus 64 highest-norm cells, updated at block boundaries, and a
 * small streaming cache).  The state is one caller-owned device buffer of
 * fs_decode_state_bytes() bytes whose size does not depend on the position:
 *  - a 256-byte header whose first int is the error word (fs_check_status
 *    reads it), then theta_i / pi (fp64) for the rotations;
 *  - per (batch, head): a w-row ring of the last keys (fp32, rotated by
 *    their absolute position, so that a step rotates only its query) and
 *    values (bf16), P + W +
 *    Bq/s + 1 cell slots (raw keys and values of one cell, its mean key and
 *    largest key norm), and the lists that place the slots: the W recent
 *    cells, the running top-P older cells (a_c desc, c asc), the closed cells
 *    not yet available, the open cell, the free slots.
 * A cell stays in its slot from its first token until it leaves the pool; a
 * cell dropped from the top P is never needed again (the threshold only
 * rises), so its slot is reused.  Decoding supports w <= 512 (the window's
 * values are staged in shared memory), FS-L mode only, P + W <= 72, K <= 8. */
size_t fs_decode_state_bytes(int batch, int H, int d, const fs_params *p);

/* Layout of a decode state, for inspection: offs receives 7 values --
 * the global part's bytes, one (batch, head)'s bytes, then inside a head's
 * block the offsets of the slot cell ids (int32), slot a_c (f32), slot mean
 * keys (f32 x d), and the number of slots and of header ints.  Head bh's
 * block starts at offs[0] + bh * offs[1]. */
int fs_decode_state_view(int batch, int H, int d, const fs_params *p,
                         size_t *offs);

/* Fill `state` as it stands after the first N0 tokens of a sequence.
 *   k, v        [batch,H,N,d] bf16 DEVICE: rows < N0 are the prefix (N0 <= N,
 *               N a multiple of Bq); NULL when N0 == 0
 *   kbar, amax  fs_cell_summarize of k (cells < floor(N0/s) are read)
 *   pool, pool_count  fs_prune_cells of amax (the row of block
 *               floor((N0-1)/Bq) is read); NULL when N0 == 0
 * The next fs_decode_step must be for t = N0. */
int fs_decode_state_init(const void *k, const void *v, int dtype,
                         const float *kbar, const float *amax,
                         const int32_t *pool, const int32_t *pool_count,
                         int batch, int H, int N, int N0, int d,
                         const fs_params *p, void *state, size_t state_bytes,
                         void *stream);

/* One decode step of FS-L for token t of every (batch, head): row t of
 * fs_attention_fwd's output, from the bounded state alone (paper.rainbus.top
 * summary, 方法步骤详情 ②-⑥).  It also advances the state: at a block start
 * (t % Bq == 0, t > 0) the pool moves to block t/Bq; k_t, v_t enter the ring
 * and the open cell; a cell that row t closes gets its summary, bit-identical
 * to fs_cell_summarize.
 *   q_t, k_t, v_t   [batch,H,d] bf16: the new token
 *   lambda, sigma, mix [H] f32
 *   out_t           [batch,H,d] f32
 *   sel_t           [batch,H,K] int32 (nullable): the selected cells
 * The state must be at position t (after t tokens); otherwise the step
 * changes nothing and records FS_ERR_STATE in the state's error word.
 * A cluster of 8 CTAs per (batch, head); the state stays the same size at
 * any t. */
int fs_decode_step(const void *q_t, const void *k_t, const void *v_t, int dtype,
                   int batch, int H, int d, int t, const float *lambda,
                   const float *sigma, const float *mix, const fs_params *p,
                   void *state, size_t state_bytes, float *out_t,
                   int32_t *sel_t, void *stream);

/* fs_prune_cells for callers that can neither allocate device memory nor
 * lend a workspace (no counterpart on the pages: a library convenience).
 * Same arguments, same pools and counts, bit for bit, as fs_prune_cells; the
 * scratch is a fixed array inside the library instead of `ws`.
 *  - Limit: fs_prune_static_scratch_bytes() (4 MiB per device), enough for
 *    batch*H*ceil(N/2048) <= 4096; a larger shape returns
 *    FS_ERR_SCRATCH_LIMIT and launches nothing.
 *  - The array needs no initial contents (nothing in it must start at zero).
 *  - Every call on a device uses the same array: calls that overlap in time
 *    (other streams, or host threads without ordering) race on it.
 *  - The first call on each device looks up the array's address (for the
 *    device current at that call) and keeps it with the device's context; a
 *    device reset (cudaDeviceReset) changes the address, and the next call
 *    looks it up again.  Make the first call on a device, and the first
 *    after a reset, before any stream capture begins.
 * Allocates nothing: no device or host memory is obtained. */
size_t fs_prune_static_scratch_bytes(void);
int fs_prune_cells_static(const float *amax, int batch, int H, int N,
                          const fs_params *p, int32_t *pool,
                          int32_t *pool_count, void *stream);

/* Shared q / k / v projection (paper.rainbus.top summary, 方法步骤详情 ①:
 * the hidden state goes through RMSNorm and W_q, W_k, W_v, and both branches
 * of every head use the result):
 *   RMSNorm(x) = x / sqrt(mean(x^2) + eps) * gain      (per row of D)
 *   [q | k | v] = RMSNorm(x) . w_qkv^T, split into heads of d = 64
 *   x        [batch, N, D] bf16 DEVICE (N a multiple of 128, D of 64)
 *   gain     [D] f32, or NULL for ones; it is folded into the weights once
 *            per call as bf16(w * gain)
 *   w_qkv    [3*H*64, D] bf16: rows of q, then k, then v (head h of each
 *            holds rows h*64 .. h*64+63), the [out, in] layout
 *   q, k, v  [batch, H, N, 64] bf16 (the layout every attention call reads)
 *   ws       device workspace of fs_qkv_workspace_bytes() bytes (row
 *            scales, folded weights; the first 256 bytes are the error word)
 * One tcgen05 GEMM with the row scale in its epilogue, after a streaming
 * pass for the row scales. */
size_t fs_qkv_workspace_bytes(int batch, int N, int D, int H);
int fs_qkv_prologue(const void *x, const float *gain, const void *w_qkv,
                    int batch, int N, int D, int H, float eps, void *q,
                    void *k, void *v, void *ws, size_t ws_bytes,
                    void *stream);

/* FS-B selection (ai.info summary, "Methodology in Plain English", FS-B;
 * paper.rainbus.top summary, 方法步骤详情 ⑤ and 技术新颖性): two causal
 * forests per (batch, head) over the cells in position order -- all cells, and
 * the cells with amax > tau -- whose nodes (aligned runs of 2^j cells) keep
 * the mean of their mean keys, a radius bounding their children, the largest
 * amax and the first cell; for query n of block beta, a beam of p->beam nodes
 * per level descends the runs tiling each forest's cells below beta*Bq/s,
 * ranked by the bound
 *   q . mean + |q| radius + lambda amax erf(sigma (n - p_first) / s),
 * and the union of both beams' cells is reranked by the log-sum-exp of their
 * s token logits q . k_t / sqrt(d); the top K are kept (LSE desc, c asc).
 *   q, k        [batch,H,N,d] bf16 (k unrotated, for the rerank)
 *   kbar, amax  fs_cell_summarize of k
 *   sel         [batch,H,N,K] int32 ranked, -1 padded
 *   ws          device scratch of fs_fsb_workspace_bytes() bytes (forests) */
size_t fs_fsb_workspace_bytes(int batch, int H, int N, const fs_params *p);
int fs_fsb_select(const void *q, const void *k, const float *kbar,
                  const float *amax, const float *lambda, const float *sigma,
                  int batch, int H, int N, int d, const fs_params *p,
                  int32_t *sel, void *ws, size_t ws_bytes, void *stream);

/* Cell scoring and top-K (paper.rainbus.top summary, 核心方法 and
 * 方法步骤详情 ⑤; 局限与改进 for the erf factor; ai.info "Methodology in
 * Plain English").  For query n of block beta and candidate c
 *   u = q_n . kbar_c + lambda_h * amax_c * erf(sigma_h * (n - p_c) / s),
 *   p_c = c*s + s/2,
 * q unrotated.  Candidates: the block's pool (FS-L) or every available cell
 * (FS; pool and pool_count may then be NULL).  Keeps the top min(K, |cands|)
 * by (u desc, c asc).
 *   q            [batch,H,N,d] bf16
 *   lambda,sigma [H] f32
 *   sel          [batch,H,N,K] int32 ranked, -1 padded
 *   sel_score    [batch,H,N,K] f32 or NULL */
int fs_select_cells(const void *q, int dtype, const float *kbar,
                    const float *amax, const int32_t *pool,
                    const int32_t *pool_count, const float *lambda,
                    const float *sigma, int batch, int H, int N, int d,
                    const fs_params *p, int32_t *sel, float *sel_score,
                    void *stream);

/* NoPE readout (paper.rainbus.top summary, 方法步骤详情 ⑥ and 前置知识
 * NoPE): softmax(q_n . k_t / sqrt(d)) over the tokens of query n's selected
 * cells, unrotated, weighted sum of v, then RMSNorm without gain:
 *   o_long[n] = o / sqrt(mean(o^2) + rms_eps);  0 when no cell is selected.
 *   q, k, v   [batch,H,N,d] bf16;  sel [batch,H,N,K] int32 (-1 = none)
 *   o_long    [batch,H,N,d] f32 */
int fs_sparse_readout(const void *q, const void *k, const void *v, int dtype,
                      const int32_t *sel, int batch, int H, int N, int d,
                      const fs_params *p, float *o_long, void *stream);

/* Workspace bytes fs_window_attn needs: header, RoPE angle table, keys
 * rotated by their positions (bf16 hi | lo, 256 B per token-head) and fp16
 * values (128 B per token-head).  0 for invalid arguments. */
size_t fs_window_workspace_bytes(int batch, int H, int N, int d, const fs_params *p);

/* Sliding-window RoPE branch and branch mix (paper.rainbus.top summary,
 * 方法步骤详情 ② and ⑥; ai.info, "Methodology in Plain English"):
 *   o_win[n] = softmax over j in [max(0,n-w+1), n] of (R(n)q_n . R(j)k_j)/sqrt(d)
 *              applied to v_j, RoPE half-split with base rope_base;
 *   out[n]   = o_win[n] + mix_h * o_long[n]   (o_long NULL: out = o_win).
 *   out       [batch,H,N,d] f32
 *   ws        device scratch of fs_window_workspace_bytes() bytes */
int fs_window_attn(const void *q, const void *k, const void *v, int dtype,
                   const float *o_long, const float *mix, int batch, int H,
                   int N, int d, const fs_params *p, float *out, void *ws,
                   size_t ws_bytes, void *stream);

/* fs_window_attn that also records CUDA events on `stream` (no counterpart
 * on the pages: per-kernel timing).  stage_events: NULL, or an array of 3
 * cudaEvent_t (as void*) created by the caller; event 0 is recorded before
 * the operand preparation (angle table, rotated keys, fp16 values), event 1
 * before the attention kernel and event 2 after it.  Same arguments and
 * results otherwise. */
int fs_window_attn_traced(const void *q, const void *k, const void *v,
                          int dtype, const float *o_long, const float *mix,
                          int batch, int H, int N, int d, const fs_params *p,
                          float *out, void *ws, size_t ws_bytes, void *stream,
                          void *const *stage_events);

/* Whole FS-L (or FS) attention forward: cell summaries, pools, selection,
 * then both attention branches and the mix in one kernel, all on `stream`.
 *   q, k, v   [batch,H,N,d] bf16 or f32 (f32 is rounded to bf16 once)
 *   lambda, sigma, mix   [H] f32
 *   out       [batch,H,N,d] f32
 *   ws        device workspace of at least fs_workspace_bytes() bytes; after
 *             the call it holds the intermediates (see fs_workspace_view). */
int fs_attention_fwd(const void *q, const void *k, const void *v, int dtype,
                     int batch, int H, int N, int d, const fs_params *p,
                     const float *lambda, const float *sigma, const float *mix,
                     float *out, void *ws, size_t ws_bytes, void *stream);

/* Gradients of the forward (paper.rainbus.top summary, 方法步骤详情: the
 * hard top-P / top-K indices carry no gradient; sigma_h and lambda_h are
 * fixed, 局限与改进; ai.info "Methodology in Plain English", training).  For
 * L = sum(dout * out) with out = fs_attention_fwd(q, k, v, ...), the pools and
 * selections held at the forward's:
 *   dout        [batch,H,N,d] f32 DEVICE (dL/dout)
 *   dq, dk, dv  [batch,H,N,d] f32 (written)
 *   dmix        [H] f32 (written): summed over the batch
 * q, k, v bf16 (FS_BF16 only); the other arguments as fs_attention_fwd.
 *   ws          device workspace of fs_backward_workspace_bytes() bytes
 * The forward's selection stages run again inside the call (cell summaries,
 * pools, scores and top-K, bit-identical to the forward's).  dk and dv of the
 * long branch are accumulated with fp32 atomic additions, so their last bits
 * can differ between runs; everything else is deterministic.  The window
 * branch's kernels run on the tensor cores with bounded waits: a wait that
 * gives up records FS_ERR_TIMEOUT in the workspace's status word
 * (fs_check_status(ws)). */
size_t fs_backward_workspace_bytes(int batch, int H, int N, int d,
                                   const fs_params *p);
int fs_attention_bwd(const void *q, const void *k, const void *v, int dtype,
                     int batch, int H, int N, int d, const fs_params *p,
                     const float *lambda, const float *sigma, const float *mix,
                     const float *dout, float *dq, float *dk, float *dv,
                     float *dmix, void *ws, size_t ws_bytes, void *stream);

/* Number of timed stages of fs_attention_fwd_traced: cell summaries and
 * window-operand preparation (RoPE angle table, rotated keys, fp16 values),
 * pruning, selection, attention (window branch, NoPE readout of the selected
 * cells and the mix, in one kernel). */
#define FS_N_STAGES 4

/* fs_attention_fwd that also records CUDA events between its stages, for
 * per-kernel timing on the launch stream.  stage_events: NULL, or an array of
 * FS_N_STAGES + 1 cudaEvent_t (as void*) created by the caller; event i is
 * recorded before stage i and event FS_N_STAGES after the last stage (the
 * fp32-to-bf16 rounding of FS_FP32 inputs happens before event 0; the prune
 * stage is empty in FS mode).  Same arguments and results otherwise. */
int fs_attention_fwd_traced(const void *q, const void *k, const void *v,
                            int dtype, int batch, int H, int N, int d,
                            const fs_params *p, const float *lambda,
                            const float *sigma, const float *mix, float *out,
                            void *ws, size_t ws_bytes, void *stream,
                            void *const *stage_events);

/* Device workspace bytes fs_attention_fwd_host needs: two staging slots,
 * each with q, k, v and out of `heads_per_chunk` heads and a forward
 * workspace for them.  0 on bad args. */
size_t fs_host_workspace_bytes(int batch, int H, int N, int d,
                               const fs_params *p, int dtype,
                               int heads_per_chunk);

/* fs_attention_fwd on HOST buffers, with the copies inside the call.  This
 * entry point has no counterpart on the pages: it serves callers whose
 * activations live in host memory.  The op is independent per (batch,
 * head), so the call walks groups of `heads_per_chunk` heads of one batch
 * row through two device staging slots; the first group of the first and of
 * the last batch row takes half as many heads, since the call's first load
 * and last store overlap no compute.  The load of the next group, the
 * forward of this one and the store of the previous one overlap: loads on
 * one copy stream, forwards on `stream`, stores on a second copy stream,
 * ordered by events.  Results are bit-identical to fs_attention_fwd.
 *   q, k, v   [batch,H,N,d] HOST memory, dtype as in fs_attention_fwd
 *             (page-locked memory lets the copies overlap; pageable memory
 *             works, with copies that do not)
 *   lambda, sigma, mix   [H] f32 DEVICE memory
 *   out       [batch,H,N,d] f32 HOST memory
 *   ws        device workspace of at least fs_host_workspace_bytes() bytes;
 *             its header holds the error word of the whole call
 * `stream` completes only after every copy of the call, so a stream
 * synchronise makes `out` readable; the host buffers must stay valid until
 * then.  The two copy streams and their six events are created on the first
 * call of each host thread on each device and kept for the thread's life
 * (driver objects, not memory: the call allocates no memory).  A CUDA failure
 * while creating them gives FS_ERR_CUDA. */
int fs_attention_fwd_host(const void *q, const void *k, const void *v,
                          int dtype, int batch, int H, int N, int d,
                          const fs_params *p, const float *lambda,
                          const float *sigma, const float *mix, float *out,
                          int heads_per_chunk, void *ws, size_t ws_bytes,
                          void *stream);

/* Every workspace begins with a 256-byte header whose first int is a device
 * error word, cleared at the start of each call (the next two ints are the
 * attention kernel's q-tile tickets, cleared with it and left clear).  Kernels that wait on
 * mbarriers give up after a bounded number of polls (seconds) and record
 * FS_ERR_TIMEOUT there instead of hanging; the window branch records
 * FS_ERR_RANGE there when a value of v is outside the fp16 range (its
 * probabilities and values meet in an fp16 product, fp32 accumulation), and
 * the output is then not valid.  fs_check_status synchronises
 * `stream` and returns FS_OK or the recorded status (FS_ERR_CUDA if the copy
 * or the synchronisation fails). */
int fs_check_status(const void *ws, void *stream);

/* Self-test of the bounded device waits (no counterpart on the pages): one
 * CTA waits on an mbarrier that nothing completes; the wait gives up after
 * its limit (about two seconds of SM clock) and records FS_ERR_TIMEOUT in the
 * error word at the start of `ws` (cleared first), exactly as a stalled
 * pipeline stage of the attention kernels would.  fs_check_status(ws) then
 * returns FS_ERR_TIMEOUT.  No GPU fault is involved. */
int fs_selftest_wait_timeout(void *ws, void *stream);

/* Byte offsets of the intermediates inside an fs_attention_fwd workspace,
 * for inspection: kbar, amax, pool, pool_count, sel (any may be NULL).  The
 * long-branch output is never materialised: the attention kernel mixes it
 * into `out` directly.  Returns FS_OK or FS_ERR_INVALID_ARG. */
int fs_workspace_view(int batch, int H, int N, int d, const fs_params *p,
                      int dtype, size_t *off_kbar, size_t *off_amax,
                      size_t *off_pool, size_t *off_pool_count,
                      size_t *off_sel);

#ifdef __cplusplus
}
#endif
#endif /* FS_H_ */
