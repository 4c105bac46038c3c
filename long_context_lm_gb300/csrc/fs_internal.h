// fs_internal.h -- launchers shared between the kernel files and the C ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace fs {

struct Shape;

cudaError_t launch_round_bf16(const float *src, void *dst, size_t n, cudaStream_t st);
cudaError_t launch_cell_summary(const void *k, bool f32, const Shape &sh, float *kbar,
                                float *amax, cudaStream_t st);
size_t prune_workspace_bytes(const Shape &sh);
cudaError_t launch_prune(const float *amax, const Shape &sh, int P, int W, int32_t *pool,
                         int32_t *pool_count, void *ws, cudaStream_t st);
cudaError_t launch_select(const void *q, const float *kbar, const float *amax,
                          const int32_t *pool, const int32_t *pool_count, const float *lambda,
                          const float *sigma, const Shape &sh, int K, int cap, bool fs_mode,
                          int32_t *sel, float *sel_score, int *err, cudaStream_t st);
cudaError_t launch_readout(const void *q, const void *k, const void *v, const int32_t *sel,
                           const Shape &sh, int K, float rms_eps, float *o_long,
                           cudaStream_t st);
size_t window_table_bytes(int w);
cudaError_t launch_window_tc(const void *q, const void *k, const void *v, const float *o_long,
                             const float *mix, void *table, const Shape &sh, int w, float base,
                             float *out, int *err, cudaStream_t st);

}  // namespace fs
