// fs_api.cu -- the extern "C" entry points declared in include/fs.h:
// argument validation, workspace carving and stream-ordered launches.
#include <stdio.h>

#include <functional>
#include <mutex>

#include "fs_common.cuh"
#include "fs_internal.h"
#include "tc05.cuh"

namespace fs {

__global__ void round_bf16_kernel(const float4 *__restrict__ src, uint2 *__restrict__ dst,
                                  size_t n4) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4;
       i += (size_t)gridDim.x * blockDim.x) {
    const float4 x = __ldg(src + i);
    dst[i] = make_uint2(pack_bf16(x.x, x.y), pack_bf16(x.z, x.w));
  }
}

cudaError_t launch_round_bf16(const float *src, void *dst, size_t n, cudaStream_t st) {
  const size_t n4 = n / 4;  // n is a multiple of 64 here
  const unsigned grid = (unsigned)((n4 + 255) / 256 < 152 * 16 ? (n4 + 255) / 256 : 152 * 16);
  round_bf16_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const float4 *>(src),
                                          static_cast<uint2 *>(dst), n4);
  return cudaGetLastError();
}

namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int check_params(const fs_params *p) {
  if (!p) return FS_ERR_INVALID_ARG;
  if (p->w < 1 || p->s < 1 || p->K < 1 || p->P < 0 || p->W < 0 || p->Bq < 1)
    return FS_ERR_INVALID_ARG;
  if (p->Bq % p->s) return FS_ERR_INVALID_ARG;
  if (!(p->rms_eps >= 0.f) || !(p->rope_base > 0.f)) return FS_ERR_INVALID_ARG;
  if (p->mode != FS_MODE_FSL && p->mode != FS_MODE_FS && p->mode != FS_MODE_FSB)
    return FS_ERR_INVALID_ARG;
  if (p->mode == FS_MODE_FSB && (p->beam < 1 || !(p->tau == p->tau))) return FS_ERR_INVALID_ARG;
  if (p->mode == FS_MODE_FSB && p->beam > 16) return FS_ERR_UNSUPPORTED;
  if (p->s != kS || p->Bq != kBq || p->P > kMaxP || p->K > kMaxK || p->w > 1024)
    return FS_ERR_UNSUPPORTED;
  return FS_OK;
}

int check_shape(int batch, int H, int N, int d) {
  if (batch < 1 || H < 1 || N < 1 || d < 1) return FS_ERR_INVALID_ARG;
  if (N % kBq) return FS_ERR_INVALID_ARG;
  if (d != kD) return FS_ERR_UNSUPPORTED;
  if ((long long)batch * H > 65535) return FS_ERR_UNSUPPORTED;
  if ((long long)N > (1ll << 24)) return FS_ERR_UNSUPPORTED;
  if ((long long)batch * H * N >= (1ll << 31)) return FS_ERR_UNSUPPORTED;  // 32-bit TMA rows
  return FS_OK;
}

int check_dtype(int dtype) {
  return (dtype == FS_BF16 || dtype == FS_FP32) ? FS_OK : FS_ERR_INVALID_ARG;
}

thread_local cudaError_t g_last_cuda_error = cudaSuccess;

int status_of(cudaError_t e) {
  if (e == cudaSuccess) return FS_OK;
  g_last_cuda_error = e;
  return FS_ERR_CUDA;
}

#define FS_TRY(x)                  \
  do {                             \
    int _rc = (x);                 \
    if (_rc != FS_OK) return _rc;  \
  } while (0)

// Every workspace starts with a 256-byte header whose first int is the device
// error word (0 = ok, else an fs_status set by a kernel's bounded wait).
constexpr size_t kHeader = 256;

// Window-branch operands: RoPE angle table, rotated keys (bf16 hi | lo),
// fp16 values.
struct WindowLayout {
  size_t tab, kt, v16;
};

WindowLayout take_window(const Shape &sh, const std::function<size_t(size_t)> &take) {
  WindowLayout W;
  const size_t rows = (size_t)sh.BH() * sh.N;
  W.tab = take(rope_table_bytes(sh.N));
  W.kt = take(rows * 2 * kD * 2);
  W.v16 = take(rows * kD * 2);
  return W;
}

// Layout of the fs_attention_fwd workspace.
struct Layout {
  size_t qb, kb, vb;       // bf16 copies (fp32 inputs only)
  size_t kbar, amax, pool, pool_count, sel, prune, fsb;
  WindowLayout win;
  size_t total;
};

Layout make_layout(const Shape &sh, const fs_params &p, int dtype) {
  Layout L{};
  size_t off = kHeader;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  const size_t elems = (size_t)sh.BH() * sh.N * sh.d;
  const size_t in_bytes = dtype == FS_FP32 ? elems * 2 : 0;
  L.qb = take(in_bytes);
  L.kb = take(in_bytes);
  L.vb = take(in_bytes);
  L.kbar = take((size_t)sh.BH() * sh.C() * kD * sizeof(float));
  L.amax = take((size_t)sh.BH() * sh.C() * sizeof(float));
  L.pool = take((size_t)sh.BH() * sh.nblk() * (p.P + p.W) * sizeof(int32_t));
  L.pool_count = take((size_t)sh.BH() * sh.nblk() * sizeof(int32_t));
  L.sel = take((size_t)sh.BH() * sh.N * p.K * sizeof(int32_t));
  L.prune = take(prune_workspace_bytes(sh));
  L.fsb = take(p.mode == FS_MODE_FSB ? (size_t)sh.BH() * fsb_layout(sh.C()).head_bytes : 0);
  L.win = take_window(sh, take);
  L.total = off;
  return L;
}

// Workspace of fs_window_attn: header, then the window operands.
size_t window_total(const Shape &sh, WindowLayout *W) {
  size_t off = kHeader;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  const WindowLayout L = take_window(sh, take);
  if (W) *W = L;
  return off;
}

// Angle table, then rotated keys and fp16 values, on `st`.
int prepare_window(const Shape &sh, const void *k, const void *v, float rope_base, char *base,
                   const WindowLayout &W, int *err, cudaStream_t st) {
  FS_TRY(status_of(launch_rope_table(base + W.tab, sh.N, rope_base, st)));
  return status_of(launch_prep(k, v, base + W.tab, sh, base + W.kt, base + W.v16, err, st));
}

int forward(const void *q, const void *k, const void *v, int dtype, const Shape &sh,
            const fs_params *p, const float *lambda, const float *sigma, const float *mix,
            float *out, char *base, const Layout &L, int *err, cudaStream_t st,
            void *const *stage_events, bool clear_status);

}  // namespace
}  // namespace fs

using namespace fs;

extern "C" {

void fs_default_params(fs_params *p) {
  if (!p) return;
  p->w = 512;
  p->s = 32;
  p->K = 4;
  p->P = 64;
  p->W = 8;
  p->Bq = 128;
  p->rope_base = 10000.f;
  p->rms_eps = 1e-6f;
  p->mode = FS_MODE_FSL;
  p->beam = 16;
  p->tau = 0.f;
}

const char *fs_status_string(int status) {
  switch (status) {
    case FS_OK: return "ok";
    case FS_ERR_INVALID_ARG: return "invalid argument";
    case FS_ERR_UNSUPPORTED: return "unsupported shape or parameter";
    case FS_ERR_CUDA: return "CUDA error";
    case FS_ERR_TIMEOUT: return "device wait timed out";
    case FS_ERR_RANGE: return "a value of v is outside the fp16 range of the window product";
    case FS_ERR_SCRATCH_LIMIT:
      return "shape needs more scratch than the static array holds "
             "(4 MiB: batch*H*ceil(N/2048) <= 4096)";
    case FS_ERR_STATE: return "the decode state is not at the step's position";
    default: return "unknown status";
  }
}

const char *fs_last_cuda_error(void) { return cudaGetErrorString(g_last_cuda_error); }

int fs_set_attention_timeline(long long *timeline, int entries) {
  if ((timeline == nullptr) != (entries == 0) || entries < 0) return FS_ERR_INVALID_ARG;
  fs::set_attention_timeline(timeline, entries);
  return FS_OK;
}

size_t fs_workspace_bytes(int batch, int H, int N, int d, const fs_params *p, int dtype) {
  if (check_params(p) || check_shape(batch, H, N, d) || check_dtype(dtype)) return 0;
  return make_layout(Shape{batch, H, N, d}, *p, dtype).total;
}

int fs_workspace_view(int batch, int H, int N, int d, const fs_params *p, int dtype,
                      size_t *off_kbar, size_t *off_amax, size_t *off_pool,
                      size_t *off_pool_count, size_t *off_sel) {
  FS_TRY(check_params(p));
  FS_TRY(check_shape(batch, H, N, d));
  FS_TRY(check_dtype(dtype));
  const Layout L = make_layout(Shape{batch, H, N, d}, *p, dtype);
  if (off_kbar) *off_kbar = L.kbar;
  if (off_amax) *off_amax = L.amax;
  if (off_pool) *off_pool = L.pool;
  if (off_pool_count) *off_pool_count = L.pool_count;
  if (off_sel) *off_sel = L.sel;
  return FS_OK;
}

size_t fs_prune_workspace_bytes(int batch, int H, int N, const fs_params *p) {
  if (check_params(p) || check_shape(batch, H, N, kD)) return 0;
  return prune_workspace_bytes(Shape{batch, H, N, kD});
}

size_t fs_window_workspace_bytes(int batch, int H, int N, int d, const fs_params *p) {
  if (check_params(p) || check_shape(batch, H, N, d)) return 0;
  return window_total(Shape{batch, H, N, d}, nullptr);
}

int fs_check_status(const void *ws, void *stream) {
  if (!ws) return FS_ERR_INVALID_ARG;
  int word = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&word, ws, sizeof(int), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return FS_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return FS_ERR_CUDA;
  return word == 0 ? FS_OK : word;
}

int fs_cell_summarize(const void *k, int dtype, int batch, int H, int N, int d, int s,
                      float *kbar, float *amax, void *stream) {
  FS_TRY(check_shape(batch, H, N, d));
  FS_TRY(check_dtype(dtype));
  if (!k || !kbar || !amax || s < 1) return FS_ERR_INVALID_ARG;
  if (N % s) return FS_ERR_INVALID_ARG;
  if (s != kS) return FS_ERR_UNSUPPORTED;
  return status_of(launch_cell_summary(k, dtype == FS_FP32, Shape{batch, H, N, d}, kbar, amax,
                                       static_cast<cudaStream_t>(stream)));
}

int fs_prune_cells(const float *amax, int batch, int H, int N, const fs_params *p,
                   int32_t *pool, int32_t *pool_count, void *ws, size_t ws_bytes,
                   void *stream) {
  FS_TRY(check_params(p));
  FS_TRY(check_shape(batch, H, N, kD));
  if (!amax || !pool || !pool_count || !ws) return FS_ERR_INVALID_ARG;
  if (p->mode != FS_MODE_FSL) return FS_ERR_INVALID_ARG;
  const Shape sh{batch, H, N, kD};
  if (ws_bytes < prune_workspace_bytes(sh)) return FS_ERR_INVALID_ARG;
  return status_of(launch_prune(amax, sh, p->P, p->W, pool, pool_count, ws,
                                static_cast<cudaStream_t>(stream)));
}

int fs_select_cells(const void *q, int dtype, const float *kbar, const float *amax,
                    const int32_t *pool, const int32_t *pool_count, const float *lambda,
                    const float *sigma, int batch, int H, int N, int d, const fs_params *p,
                    int32_t *sel, float *sel_score, void *stream) {
  FS_TRY(check_params(p));
  FS_TRY(check_shape(batch, H, N, d));
  FS_TRY(check_dtype(dtype));
  if (dtype != FS_BF16) return FS_ERR_UNSUPPORTED;
  if (!q || !kbar || !amax || !lambda || !sigma || !sel) return FS_ERR_INVALID_ARG;
  if (p->mode == FS_MODE_FSB) return FS_ERR_INVALID_ARG;  // fs_fsb_select
  const bool fs_mode = p->mode == FS_MODE_FS;
  if (!fs_mode && (!pool || !pool_count)) return FS_ERR_INVALID_ARG;
  return status_of(launch_select(q, kbar, amax, pool, pool_count, lambda, sigma,
                                 Shape{batch, H, N, d}, p->K, p->P + p->W, p->W, fs_mode, sel,
                                 sel_score, nullptr, static_cast<cudaStream_t>(stream)));
}

int fs_sparse_readout(const void *q, const void *k, const void *v, int dtype,
                      const int32_t *sel, int batch, int H, int N, int d, const fs_params *p,
                      float *o_long, void *stream) {
  FS_TRY(check_params(p));
  FS_TRY(check_shape(batch, H, N, d));
  FS_TRY(check_dtype(dtype));
  if (dtype != FS_BF16) return FS_ERR_UNSUPPORTED;
  if (!q || !k || !v || !sel || !o_long) return FS_ERR_INVALID_ARG;
  AttnArgs a{};
  a.sh = Shape{batch, H, N, d};
  a.q = q;
  a.k = k;
  a.v = v;
  a.sel = sel;
  a.w = p->w;
  a.K = p->K;
  a.rms_eps = p->rms_eps;
  a.window = false;
  a.write_long = true;
  a.out = o_long;
  return status_of(launch_attn_tc(a, static_cast<cudaStream_t>(stream)));
}

int fs_window_attn(const void *q, const void *k, const void *v, int dtype, const float *o_long,
                   const float *mix, int batch, int H, int N, int d, const fs_params *p,
                   float *out, void *ws, size_t ws_bytes, void *stream) {
  return fs_window_attn_traced(q, k, v, dtype, o_long, mix, batch, H, N, d, p, out, ws, ws_bytes,
                               stream, nullptr);
}

int fs_window_attn_traced(const void *q, const void *k, const void *v, int dtype,
                          const float *o_long, const float *mix, int batch, int H, int N, int d,
                          const fs_params *p, float *out, void *ws, size_t ws_bytes, void *stream,
                          void *const *stage_events) {
  FS_TRY(check_params(p));
  FS_TRY(check_shape(batch, H, N, d));
  FS_TRY(check_dtype(dtype));
  if (dtype != FS_BF16) return FS_ERR_UNSUPPORTED;
  if (!q || !k || !v || !out || !ws || (o_long && !mix)) return FS_ERR_INVALID_ARG;
  const Shape sh{batch, H, N, d};
  WindowLayout W;
  if (ws_bytes < window_total(sh, &W)) return FS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char *base = static_cast<char *>(ws);
  int *err = reinterpret_cast<int *>(base);
  auto mark = [&](int i) -> int {
    if (!stage_events || !stage_events[i]) return FS_OK;
    return status_of(cudaEventRecord(static_cast<cudaEvent_t>(stage_events[i]), st));
  };
  FS_TRY(status_of(cudaMemsetAsync(err, 0, 4 * sizeof(int), st)));
  FS_TRY(mark(0));
  FS_TRY(prepare_window(sh, k, v, p->rope_base, base, W, err, st));
  FS_TRY(mark(1));
  AttnArgs a{};
  a.sh = sh;
  a.q = q;
  a.k = k;
  a.v = v;
  a.kt = base + W.kt;
  a.v16 = base + W.v16;
  a.tab = base + W.tab;
  a.o_long_in = o_long;
  a.mix = mix;
  a.w = p->w;
  a.K = p->K;
  a.rms_eps = p->rms_eps;
  a.window = true;
  a.out = out;
  a.err = err;
  a.sched = err + 1;  // the header's second and third ints
  FS_TRY(status_of(launch_attn_tc(a, st)));
  return mark(2);
}

int fs_attention_fwd(const void *q, const void *k, const void *v, int dtype, int batch, int H,
                     int N, int d, const fs_params *p, const float *lambda, const float *sigma,
                     const float *mix, float *out, void *ws, size_t ws_bytes, void *stream) {
  return fs_attention_fwd_traced(q, k, v, dtype, batch, H, N, d, p, lambda, sigma, mix, out, ws,
                                 ws_bytes, stream, nullptr);
}

int fs_attention_fwd_traced(const void *q, const void *k, const void *v, int dtype, int batch,
                            int H, int N, int d, const fs_params *p, const float *lambda,
                            const float *sigma, const float *mix, float *out, void *ws,
                            size_t ws_bytes, void *stream, void *const *stage_events) {
  FS_TRY(check_params(p));
  FS_TRY(check_shape(batch, H, N, d));
  FS_TRY(check_dtype(dtype));
  if (!q || !k || !v || !lambda || !sigma || !mix || !out || !ws) return FS_ERR_INVALID_ARG;
  const Shape sh{batch, H, N, d};
  const Layout L = make_layout(sh, *p, dtype);
  if (ws_bytes < L.total) return FS_ERR_INVALID_ARG;
  int *err = reinterpret_cast<int *>(ws);
  // the status word and the q-tile tickets are zeroed by the forward's first
  // kernel (no separate memset)
  return forward(q, k, v, dtype, sh, p, lambda, sigma, mix, out, static_cast<char *>(ws), L, err,
                 static_cast<cudaStream_t>(stream), stage_events, true);
}

}  // extern "C"

namespace fs {
namespace {

// The forward on validated arguments: workspace `base` laid out as `L`;
// device errors are recorded in `err`, whose four ints the first kernel zeroes
// when `clear_status` (else the caller has).
int forward(const void *q, const void *k, const void *v, int dtype, const Shape &sh,
            const fs_params *p, const float *lambda, const float *sigma, const float *mix,
            float *out, char *base, const Layout &L, int *err, cudaStream_t st,
            void *const *stage_events, bool clear_status) {
  const int N = sh.N, d = sh.d;
  const void *qb = q, *kb = k, *vb = v;
  if (dtype == FS_FP32) {
    const size_t elems = (size_t)sh.BH() * N * d;
    FS_TRY(status_of(launch_round_bf16(static_cast<const float *>(q), base + L.qb, elems, st)));
    FS_TRY(status_of(launch_round_bf16(static_cast<const float *>(k), base + L.kb, elems, st)));
    FS_TRY(status_of(launch_round_bf16(static_cast<const float *>(v), base + L.vb, elems, st)));
    qb = base + L.qb;
    kb = base + L.kb;
    vb = base + L.vb;
  }
  float *kbar = reinterpret_cast<float *>(base + L.kbar);
  float *amax = reinterpret_cast<float *>(base + L.amax);
  int32_t *pool = reinterpret_cast<int32_t *>(base + L.pool);
  int32_t *pool_count = reinterpret_cast<int32_t *>(base + L.pool_count);
  int32_t *sel = reinterpret_cast<int32_t *>(base + L.sel);
  const bool fs_mode = p->mode == FS_MODE_FS;

  auto mark = [&](int i) -> int {
    if (!stage_events || !stage_events[i]) return FS_OK;
    return status_of(cudaEventRecord(static_cast<cudaEvent_t>(stage_events[i]), st));
  };
  FS_TRY(mark(0));
  // angle table, then rotated keys, fp16 values and cell summaries in one
  // pass over k and v
  FS_TRY(status_of(launch_rope_table(base + L.win.tab, sh.N, p->rope_base, st,
                                     clear_status ? err : nullptr)));
  FS_TRY(status_of(launch_prep_summary(kb, vb, base + L.win.tab, sh, base + L.win.kt,
                                       base + L.win.v16, kbar, amax, err, st)));
  FS_TRY(mark(1));
  const bool fsb = p->mode == FS_MODE_FSB;
  if (!fs_mode && !fsb)
    FS_TRY(status_of(launch_prune(amax, sh, p->P, p->W, pool, pool_count, base + L.prune, st)));
  FS_TRY(mark(2));
  if (fsb)
    FS_TRY(status_of(launch_fsb(qb, kb, kbar, amax, lambda, sigma, sh, p->K, p->beam, p->tau,
                                base + L.fsb, sel, st)));
  else
    FS_TRY(status_of(launch_select(qb, kbar, amax, pool, pool_count, lambda, sigma, sh, p->K,
                                   p->P + p->W, p->W, fs_mode, sel, nullptr, err, st)));
  FS_TRY(mark(3));
  AttnArgs a{};
  a.sh = sh;
  a.q = qb;
  a.k = kb;
  a.v = vb;
  a.kt = base + L.win.kt;
  a.v16 = base + L.win.v16;
  a.tab = base + L.win.tab;
  a.sel = sel;
  a.mix = mix;
  a.w = p->w;
  a.K = p->K;
  a.rms_eps = p->rms_eps;
  a.window = true;
  a.out = out;
  a.err = err;
  a.sched = err + 1;  // the header's second and third ints
  FS_TRY(status_of(launch_attn_tc(a, st)));
  return mark(4);
}

// Two copy streams and the events of the host-buffer pipeline, per (host
// thread, device): created on first use and kept for the thread's life.  Per
// host thread, so that two callers never share an event between its record
// and its wait.
constexpr int kPipeDevices = 64;
struct CopyPipe {
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t entry = nullptr;  // the caller's stream at the start of a call
  cudaEvent_t loaded[2] = {}, computed[2] = {}, stored[2] = {};
};

CopyPipe *copy_pipe() {
  thread_local CopyPipe per_device[kPipeDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kPipeDevices) return nullptr;
  CopyPipe &c = per_device[dev];
  if (!c.h2d) {
    CopyPipe n;
    bool ok = cudaStreamCreateWithFlags(&n.h2d, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&n.d2h, cudaStreamNonBlocking) == cudaSuccess;
    ok = ok && cudaEventCreateWithFlags(&n.entry, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < 2; ++i)
      ok = cudaEventCreateWithFlags(&n.loaded[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&n.computed[i], cudaEventDisableTiming) == cudaSuccess &&
           cudaEventCreateWithFlags(&n.stored[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      if (n.entry) cudaEventDestroy(n.entry);
      for (int i = 0; i < 2; ++i) {
        if (n.loaded[i]) cudaEventDestroy(n.loaded[i]);
        if (n.computed[i]) cudaEventDestroy(n.computed[i]);
        if (n.stored[i]) cudaEventDestroy(n.stored[i]);
      }
      if (n.h2d) cudaStreamDestroy(n.h2d);
      if (n.d2h) cudaStreamDestroy(n.d2h);
      return nullptr;
    }
    c = n;
  }
  return &c;
}

// Staging slot of the host-buffer pipeline: q, k, v and out of `hc` heads,
// then a forward workspace for them.
struct HostLayout {
  size_t qkv_bytes, out_bytes, fwd_bytes, slot_bytes, total;
};

HostLayout host_layout(int H, int N, int d, const fs_params &p, int dtype, int hc) {
  HostLayout h{};
  const size_t elem = dtype == FS_FP32 ? 4 : 2;
  const size_t n = (size_t)hc * N * d;
  h.qkv_bytes = align_up(n * elem);
  h.out_bytes = align_up(n * 4);
  h.fwd_bytes = align_up(make_layout(Shape{1, hc, N, d}, p, dtype).total);
  h.slot_bytes = 3 * h.qkv_bytes + h.out_bytes + h.fwd_bytes;
  h.total = kHeader + 2 * h.slot_bytes;
  return h;
}

}  // namespace
}  // namespace fs

extern "C" {

size_t fs_host_workspace_bytes(int batch, int H, int N, int d, const fs_params *p, int dtype,
                               int heads_per_chunk) {
  if (check_params(p) != FS_OK || check_shape(batch, H, N, d) != FS_OK ||
      check_dtype(dtype) != FS_OK || heads_per_chunk < 1)
    return 0;
  return host_layout(H, N, d, *p, dtype, heads_per_chunk < H ? heads_per_chunk : H).total;
}

int fs_attention_fwd_host(const void *q, const void *k, const void *v, int dtype, int batch,
                          int H, int N, int d, const fs_params *p, const float *lambda,
                          const float *sigma, const float *mix, float *out, int heads_per_chunk,
                          void *ws, size_t ws_bytes, void *stream) {
  FS_TRY(check_params(p));
  FS_TRY(check_shape(batch, H, N, d));
  FS_TRY(check_dtype(dtype));
  if (!q || !k || !v || !lambda || !sigma || !mix || !out || !ws || heads_per_chunk < 1)
    return FS_ERR_INVALID_ARG;
  const int hc = heads_per_chunk < H ? heads_per_chunk : H;
  const HostLayout HL = host_layout(H, N, d, *p, dtype, hc);
  if (ws_bytes < HL.total) return FS_ERR_INVALID_ARG;
  CopyPipe *cp = copy_pipe();
  if (!cp) return FS_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char *base = static_cast<char *>(ws);
  int *err = reinterpret_cast<int *>(base);
  FS_TRY(status_of(cudaMemsetAsync(err, 0, 4 * sizeof(int), st)));
  // The loads begin only after everything already on the caller's stream:
  // an earlier call's forwards and stores that still read the staging slots,
  // and any work that writes the host inputs.
  FS_TRY(status_of(cudaEventRecord(cp->entry, st)));
  FS_TRY(status_of(cudaStreamWaitEvent(cp->h2d, cp->entry, 0)));
  const size_t elem = dtype == FS_FP32 ? 4 : 2;
  int rc = FS_OK;
  int chunk = 0;
  // Groups of hc heads, except the first group of the call's first and last
  // (batch) rows, which takes half as many: the call's first load and its
  // last store overlap no compute, so both are kept short (with H a multiple
  // of hc the last group then has half the heads as well).
  const int hhalf = (hc + 1) / 2;
  for (int b = 0; b < batch && rc == FS_OK; ++b) {
    for (int h0 = 0, hn = 0; h0 < H && rc == FS_OK; h0 += hn, ++chunk) {
      const int hg = (h0 == 0 && (b == 0 || b == batch - 1)) ? hhalf : hc;
      hn = H - h0 < hg ? H - h0 : hg;
      const int s = chunk & 1;
      char *slot = base + kHeader + s * HL.slot_bytes;
      char *qd = slot, *kd = qd + HL.qkv_bytes, *vd = kd + HL.qkv_bytes;
      float *od = reinterpret_cast<float *>(vd + HL.qkv_bytes);
      char *fws = vd + HL.qkv_bytes + HL.out_bytes;
      const size_t first = ((size_t)b * H + h0) * N * d;  // first element of the chunk
      const size_t n = (size_t)hn * N * d;
      // load: the slot's previous forward must have finished reading it
      if (chunk >= 2) rc = status_of(cudaStreamWaitEvent(cp->h2d, cp->computed[s], 0));
      const char *srcs[3] = {static_cast<const char *>(q), static_cast<const char *>(k),
                             static_cast<const char *>(v)};
      char *dsts[3] = {qd, kd, vd};
      for (int i = 0; i < 3 && rc == FS_OK; ++i)
        rc = status_of(cudaMemcpyAsync(dsts[i], srcs[i] + first * elem, n * elem,
                                       cudaMemcpyHostToDevice, cp->h2d));
      if (rc == FS_OK) rc = status_of(cudaEventRecord(cp->loaded[s], cp->h2d));
      // compute on the caller's stream: after the load, and after the slot's
      // previous output has been stored
      if (rc == FS_OK) rc = status_of(cudaStreamWaitEvent(st, cp->loaded[s], 0));
      if (rc == FS_OK && chunk >= 2) rc = status_of(cudaStreamWaitEvent(st, cp->stored[s], 0));
      if (rc == FS_OK) {
        const Shape sh{1, hn, N, d};
        rc = forward(qd, kd, vd, dtype, sh, p, lambda + h0, sigma + h0, mix + h0, od, fws,
                     make_layout(sh, *p, dtype), err, st, nullptr, false);
      }
      if (rc == FS_OK) rc = status_of(cudaEventRecord(cp->computed[s], st));
      // store
      if (rc == FS_OK) rc = status_of(cudaStreamWaitEvent(cp->d2h, cp->computed[s], 0));
      if (rc == FS_OK)
        rc = status_of(cudaMemcpyAsync(out + first, od, n * 4, cudaMemcpyDeviceToHost, cp->d2h));
      if (rc == FS_OK) rc = status_of(cudaEventRecord(cp->stored[s], cp->d2h));
    }
  }
  // the caller's stream completes only after every copy this call issued (also
  // after a failure, so that no copy outlives the caller's view of the buffers)
  for (int s = 0; s < 2 && s < chunk; ++s) {
    cudaEventRecord(cp->loaded[s], cp->h2d);
    cudaStreamWaitEvent(st, cp->loaded[s], 0);
    cudaEventRecord(cp->stored[s], cp->d2h);
    cudaStreamWaitEvent(st, cp->stored[s], 0);
  }
  return rc;
}

}  // extern "C"

namespace fs {
namespace {
int check_decode(const fs_params *p, int d) {
  FS_TRY(check_params(p));
  if (d != kD) return FS_ERR_UNSUPPORTED;
  if (p->mode != FS_MODE_FSL) return FS_ERR_INVALID_ARG;
  if (p->P + p->W > kMaxP + 8 || p->W > 8 || p->w > 512) return FS_ERR_UNSUPPORTED;
  return FS_OK;
}
}  // namespace
}  // namespace fs

extern "C" size_t fs_decode_state_bytes(int batch, int H, int d, const fs_params *p) {
  if (check_decode(p, d) != FS_OK || check_shape(batch, H, kBq, d) != FS_OK) return 0;
  return decode_layout(p->w, p->P, p->W, p->K).total(batch * H);
}

namespace fs {
namespace {
int check_qkv(int batch, int N, int D, int H) {
  if (batch < 1 || N < 1 || D < 1 || H < 1) return FS_ERR_INVALID_ARG;
  if (N % kBq || D % 64) return FS_ERR_INVALID_ARG;
  if ((long long)batch * N >= (1ll << 31) || (long long)3 * H * kD >= (1ll << 20) ||
      D > (1 << 16))
    return FS_ERR_UNSUPPORTED;
  return FS_OK;
}
}  // namespace
}  // namespace fs

extern "C" size_t fs_fsb_workspace_bytes(int batch, int H, int N, const fs_params *p) {
  if (check_params(p) != FS_OK || check_shape(batch, H, N, kD) != FS_OK) return 0;
  if (p->mode != FS_MODE_FSB) return 0;
  return (size_t)batch * H * fsb_layout(N / kS).head_bytes;
}

extern "C" int fs_fsb_select(const void *q, const void *k, const float *kbar, const float *amax,
                             const float *lambda, const float *sigma, int batch, int H, int N,
                             int d, const fs_params *p, int32_t *sel, void *ws, size_t ws_bytes,
                             void *stream) {
  FS_TRY(check_params(p));
  FS_TRY(check_shape(batch, H, N, d));
  if (p->mode != FS_MODE_FSB) return FS_ERR_INVALID_ARG;
  if (!q || !k || !kbar || !amax || !lambda || !sigma || !sel || !ws) return FS_ERR_INVALID_ARG;
  if (ws_bytes < (size_t)batch * H * fsb_layout(N / kS).head_bytes) return FS_ERR_INVALID_ARG;
  return status_of(launch_fsb(q, k, kbar, amax, lambda, sigma, Shape{batch, H, N, d}, p->K,
                              p->beam, p->tau, ws, sel, static_cast<cudaStream_t>(stream)));
}

extern "C" size_t fs_backward_workspace_bytes(int batch, int H, int N, int d,
                                              const fs_params *p) {
  if (check_params(p) != FS_OK || check_shape(batch, H, N, d) != FS_OK) return 0;
  const Shape sh{batch, H, N, d};
  return make_layout(sh, *p, FS_BF16).total + backward_workspace_bytes(sh);
}

extern "C" int fs_attention_bwd(const void *q, const void *k, const void *v, int dtype, int batch,
                                int H, int N, int d, const fs_params *p, const float *lambda,
                                const float *sigma, const float *mix, const float *dout, float *dq,
                                float *dk, float *dv, float *dmix, void *ws, size_t ws_bytes,
                                void *stream) {
  FS_TRY(check_params(p));
  FS_TRY(check_shape(batch, H, N, d));
  FS_TRY(check_dtype(dtype));
  if (dtype != FS_BF16) return FS_ERR_UNSUPPORTED;
  if (!q || !k || !v || !lambda || !sigma || !mix || !dout || !dq || !dk || !dv || !dmix || !ws)
    return FS_ERR_INVALID_ARG;
  const Shape sh{batch, H, N, d};
  const Layout L = make_layout(sh, *p, FS_BF16);
  if (ws_bytes < L.total + backward_workspace_bytes(sh)) return FS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  char *base = static_cast<char *>(ws);
  int *err = reinterpret_cast<int *>(base);
  FS_TRY(status_of(cudaMemsetAsync(err, 0, sizeof(int), st)));
  float *kbar = reinterpret_cast<float *>(base + L.kbar);
  float *amax = reinterpret_cast<float *>(base + L.amax);
  int32_t *pool = reinterpret_cast<int32_t *>(base + L.pool);
  int32_t *pool_count = reinterpret_cast<int32_t *>(base + L.pool_count);
  int32_t *sel = reinterpret_cast<int32_t *>(base + L.sel);
  const bool fs_mode = p->mode == FS_MODE_FS;
  // the forward's selection, by the forward's kernels
  FS_TRY(status_of(launch_cell_summary(k, false, sh, kbar, amax, st)));
  if (!fs_mode)
    FS_TRY(status_of(launch_prune(amax, sh, p->P, p->W, pool, pool_count, base + L.prune, st)));
  FS_TRY(status_of(launch_select(q, kbar, amax, pool, pool_count, lambda, sigma, sh, p->K,
                                 p->P + p->W, p->W, fs_mode, sel, nullptr, err, st)));
  BwdArgs a{};
  a.sh = sh;
  a.q = q;
  a.k = k;
  a.v = v;
  a.g = dout;
  a.sel = sel;
  a.mix = mix;
  a.w = p->w;
  a.K = p->K;
  a.rope_base = p->rope_base;
  a.rms_eps = p->rms_eps;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.dmix = dmix;
  a.ws = base + L.total;
  a.err = err;
  return status_of(launch_backward(a, st));
}

extern "C" size_t fs_qkv_workspace_bytes(int batch, int N, int D, int H) {
  if (check_qkv(batch, N, D, H) != FS_OK) return 0;
  return kHeader + qkv_workspace_bytes(batch * N, D, H);
}

extern "C" int fs_qkv_prologue(const void *x, const float *gain, const void *w_qkv, int batch,
                               int N, int D, int H, float eps, void *q, void *k, void *v, void *ws,
                               size_t ws_bytes, void *stream) {
  FS_TRY(check_qkv(batch, N, D, H));
  if (!x || !w_qkv || !q || !k || !v || !ws || !(eps >= 0.f)) return FS_ERR_INVALID_ARG;
  if (ws_bytes < kHeader + qkv_workspace_bytes(batch * N, D, H)) return FS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int *err = static_cast<int *>(ws);
  FS_TRY(status_of(cudaMemsetAsync(err, 0, sizeof(int), st)));
  QkvArgs a{};
  a.x = x;
  a.gain = gain;
  a.w = w_qkv;
  a.batch = batch;
  a.N = N;
  a.D = D;
  a.H = H;
  a.eps = eps;
  a.q = q;
  a.k = k;
  a.v = v;
  a.ws = static_cast<char *>(ws) + kHeader;
  a.err = err;
  return status_of(launch_qkv(a, st));
}

extern "C" int fs_decode_state_view(int batch, int H, int d, const fs_params *p, size_t *offs) {
  FS_TRY(check_decode(p, d));
  FS_TRY(check_shape(batch, H, kBq, d));
  if (!offs) return FS_ERR_INVALID_ARG;
  const DecodeLayout L = decode_layout(p->w, p->P, p->W, p->K);
  offs[0] = L.global_bytes;
  offs[1] = L.head_bytes;
  offs[2] = L.slot_cell;
  offs[3] = L.slot_amax;
  offs[4] = L.slot_kbar;
  offs[5] = (size_t)L.nslots;
  offs[6] = (size_t)kDecodeHeaderInts;
  return FS_OK;
}

extern "C" int fs_decode_state_init(const void *k, const void *v, int dtype, const float *kbar,
                                    const float *amax, const int32_t *pool,
                                    const int32_t *pool_count, int batch, int H, int N, int N0,
                                    int d, const fs_params *p, void *state, size_t state_bytes,
                                    void *stream) {
  FS_TRY(check_decode(p, d));
  FS_TRY(check_dtype(dtype));
  if (dtype != FS_BF16) return FS_ERR_UNSUPPORTED;
  if (N0 < 0 || !state) return FS_ERR_INVALID_ARG;
  if (N0 > 0) {
    FS_TRY(check_shape(batch, H, N, d));
    if (N0 > N || !k || !v || !kbar || !amax || !pool || !pool_count) return FS_ERR_INVALID_ARG;
  } else {
    FS_TRY(check_shape(batch, H, kBq, d));
    N = kBq;
  }
  const DecodeLayout L = decode_layout(p->w, p->P, p->W, p->K);
  if (state_bytes < L.total(batch * H)) return FS_ERR_INVALID_ARG;
  return status_of(launch_decode_init(k, v, kbar, amax, pool, pool_count, batch * H, N, N0,
                                      p->rope_base, L, state, static_cast<cudaStream_t>(stream)));
}

extern "C" int fs_decode_step(const void *q_t, const void *k_t, const void *v_t, int dtype,
                              int batch, int H, int d, int t, const float *lambda,
                              const float *sigma, const float *mix, const fs_params *p,
                              void *state, size_t state_bytes, float *out_t, int32_t *sel_t,
                              void *stream) {
  FS_TRY(check_decode(p, d));
  FS_TRY(check_shape(batch, H, kBq, d));
  FS_TRY(check_dtype(dtype));
  if (dtype != FS_BF16) return FS_ERR_UNSUPPORTED;
  if (t < 0) return FS_ERR_INVALID_ARG;
  if (!q_t || !k_t || !v_t || !lambda || !sigma || !mix || !state || !out_t)
    return FS_ERR_INVALID_ARG;
  const DecodeLayout L = decode_layout(p->w, p->P, p->W, p->K);
  if (state_bytes < L.total(batch * H)) return FS_ERR_INVALID_ARG;
  DecodeArgs a{};
  a.q_t = q_t;
  a.k_t = k_t;
  a.v_t = v_t;
  a.state = state;
  a.lambda = lambda;
  a.sigma = sigma;
  a.mix = mix;
  a.L = L;
  a.batch = batch;
  a.H = H;
  a.t = t;
  a.rms_eps = p->rms_eps;
  a.out = out_t;
  a.sel_out = sel_t;
  return status_of(launch_decode(a, static_cast<cudaStream_t>(stream)));
}

namespace fs {
namespace {
// One CTA waits on an mbarrier that nothing ever completes: the bounded wait
// gives up after its limit and records FS_ERR_TIMEOUT, as a stalled pipeline
// stage would, and the kernel returns normally.
__global__ void selftest_timeout_kernel(int *err) {
  __shared__ __align__(8) uint64_t never;
  if (threadIdx.x == 0) {
    tc::mbar_init(&never, 1);
    tc::mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) tc::mbar_wait(&never, 0, err);
}
}  // namespace
}  // namespace fs

extern "C" int fs_selftest_wait_timeout(void *ws, void *stream) {
  if (!ws) return FS_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int *err = static_cast<int *>(ws);
  FS_TRY(status_of(cudaMemsetAsync(err, 0, sizeof(int), st)));
  selftest_timeout_kernel<<<1, 32, 0, st>>>(err);
  return status_of(cudaGetLastError());
}

// ---------------------------------------------------------------------------
// fs_prune_cells_static: the pool construction without a caller workspace.
//
// Some callers have no device memory to hand over and may not obtain any:
// code that runs where allocating is forbidden or impossible, such as a
// memory allocator's own callbacks or out-of-memory handling, or a serving
// loop whose device memory was fully reserved before it started, and that
// owns no spare buffer it could lend as scratch.  For them this entry point
// runs the same three pruning kernels on a fixed array compiled into the
// library, so the call allocates nothing.
//
// Limit: kStaticScratchBytes (4 MiB per device) holds the two banks of
// per-chunk lists the kernels ping-pong between, 2 * batch*H*ceil(C/64)
// lists of 64 eight-byte keys; it serves batch*H*ceil(N/2048) <= 4096 (for
// example 16 heads up to N = 512k).  Larger shapes are rejected with
// FS_ERR_SCRATCH_LIMIT before anything is launched.  No byte of the array
// needs to start at zero: every call writes each list before it reads it.
// All calls on a device share the one array, so calls that overlap in time
// (on different streams, or from host threads without ordering between
// them) race on it.
//
// Set-up: the first call on each device (the device current at that call)
// looks up the array's device address with cudaGetSymbolAddress and keeps it
// with the device's context; after a device reset the next call looks it up
// again.  Make the first call on a device (and the first after a reset)
// before any stream capture begins.
// ---------------------------------------------------------------------------
namespace fs {
namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;
static __device__ __align__(256) unsigned char g_prune_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
struct ScratchAddr {
  void *ctx = nullptr;   // the device's context when the address was taken
  void *addr = nullptr;
};
ScratchAddr g_scratch_addr[kMaxDevices];

// The current context (cuCtxGetCurrent through the runtime's driver entry
// point); null when it cannot be read.
void *current_context() {
  using GetCurrent = int (*)(void **);
  static GetCurrent fn = [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<GetCurrent>(ptr);
    return static_cast<GetCurrent>(nullptr);
  }();
  void *ctx = nullptr;
  if (!fn || fn(&ctx) != 0) return nullptr;
  return ctx;
}

// Device address of g_prune_scratch on the current device.  It is looked up
// once per device and context: a device reset (cudaDeviceReset) replaces the
// context and with it the array's address, so a changed context (or one that
// cannot be read) makes the lookup run again.
cudaError_t static_scratch(void **addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void *ctx = current_context();  // null before the runtime's first use of the device
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  ScratchAddr &c = g_scratch_addr[dev];
  if (!c.addr || !ctx || c.ctx != ctx) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_prune_scratch);  // also makes the context current
    if (e != cudaSuccess) return e;
    c.addr = p;
    c.ctx = current_context();
  }
  *addr = c.addr;
  return cudaSuccess;
}

}  // namespace
}  // namespace fs

extern "C" {

size_t fs_prune_static_scratch_bytes(void) { return kStaticScratchBytes; }

int fs_prune_cells_static(const float *amax, int batch, int H, int N, const fs_params *p,
                          int32_t *pool, int32_t *pool_count, void *stream) {
  FS_TRY(check_params(p));
  FS_TRY(check_shape(batch, H, N, kD));
  if (!amax || !pool || !pool_count) return FS_ERR_INVALID_ARG;
  if (p->mode != FS_MODE_FSL) return FS_ERR_INVALID_ARG;
  const Shape sh{batch, H, N, kD};
  if (prune_workspace_bytes(sh) > kStaticScratchBytes) return FS_ERR_SCRATCH_LIMIT;
  void *scratch = nullptr;
  FS_TRY(status_of(static_scratch(&scratch)));
  return status_of(launch_prune(amax, sh, p->P, p->W, pool, pool_count, scratch,
                                static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
