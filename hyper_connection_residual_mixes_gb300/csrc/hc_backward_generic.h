// hc_backward_generic.h -- the side step's backward for the stream counts
// other than four (hc = 2 and 8).  Same contract as launch_block_step_backward
// (hc_launch.h); the workspace size depends on hc.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace hc {

// Bytes of workspace the generic backward needs for n tokens; 0 unless hc is 2 or 8.
size_t backward_generic_workspace_bytes(int64_t n, int hc, int d);

cudaError_t launch_block_step_backward_generic(int hc, const uint16_t *x, const float *pre_mix,
                                               const uint16_t *f, const float *hc_fn,
                                               const float *hc_scale, const float *hc_base,
                                               const float *norm_w, int64_t n, int d, int iters,
                                               float eps, float norm_eps, const float *g_hn,
                                               const float *g_y, const float *g_pre, float *g_x,
                                               float *g_pm, float *g_f, float *g_fn, float *g_scale,
                                               float *g_base, float *g_w, void *workspace,
                                               cudaStream_t s);

}  // namespace hc
