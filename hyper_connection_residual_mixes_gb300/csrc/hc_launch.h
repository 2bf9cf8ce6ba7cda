// hc_launch.h -- internal launcher prototypes (host side of libhc).
// Arguments have been validated by hc_api.cu before any of these is called:
// hc in {2, 4, 8} (4 only for the cluster and chain paths), d a multiple of 64 in
// [64, 16384], n >= 1, pointers 16-byte aligned.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace hc {

cudaError_t launch_split_sinkhorn(const float *mixes, const float *hc_scale, const float *hc_base,
                                  int64_t n, int hc, int iters, float eps, float *pre, float *post,
                                  float *comb, cudaStream_t s);

cudaError_t launch_pre_norm(const uint16_t *x, const float *pre_mix, const float *norm_w,
                            int64_t n, int hc, int d, float norm_eps, uint16_t *out, cudaStream_t s);

cudaError_t launch_mxfp8_cast(const uint16_t *in, int64_t rows, int d, uint8_t *codes,
                              uint8_t *scales, cudaStream_t s);
cudaError_t launch_pre_norm_mxfp8(const uint16_t *x, const float *pre_mix, const float *norm_w,
                                  int64_t n, int hc, int d, float norm_eps, uint16_t *out,
                                  uint8_t *codes, uint8_t *scales, cudaStream_t s);
cudaError_t launch_post(const uint16_t *f, const uint16_t *residual, const float *post,
                        const float *comb, int64_t n, int hc, int d, uint16_t *y, cudaStream_t s);

// The projection a = x hc_fn^T alone on the tcgen05 tensor cores
// (hc_proj_umma.cu): a[t][i] at out[t * out_stride + i].  `wsplit` is device
// scratch of proj_umma_wsplit_bytes(hc, hc * d) bytes (16-byte aligned) for the
// split weights; it is dead once the launch has completed.  With `scratch`
// (scratch_floats floats) K may be split over CTAs when the batch has fewer
// 128-token tiles than CTA slots, the slices' partial sums held there and
// added in slice order.
size_t proj_umma_wsplit_bytes(int hc, int64_t K);
cudaError_t launch_proj_umma(const uint16_t *x, const float *hc_fn, int64_t n, int hc, int d, uint16_t *wsplit,
                             float *out, int out_stride, cudaStream_t s, float *scratch = nullptr,
                             int64_t scratch_floats = 0);
// a1-a3 on the same kernel: the projection, the sum of squares of x, the RMS
// scale, split + Sinkhorn; pre / post / comb / mixes out (each may be null)
// and post + comb at the start of each token's row of `coef_rows` (the y
// output, row length hc * d bf16) for the a4-a6 pass.
cudaError_t launch_mixes_umma(const uint16_t *x, const float *hc_fn, const float *hc_scale, const float *hc_base,
                              int64_t n, int hc, int d, int iters, float eps, float norm_eps, uint16_t *wsplit,
                              float *pre_out, float *post_out, float *comb_out, float *mixes_out,
                              uint16_t *coef_rows, cudaStream_t s);

// a1-a3 (write pre/post/comb, optional mixes) or, when `f` is non-null, the
// whole side step a1-a6.  Simple path: a CTA owns a few whole tokens.
cudaError_t launch_tokens_simple(const uint16_t *x, const float *pre_mix, const uint16_t *f,
                                 const float *hc_fn, const float *hc_scale, const float *hc_base,
                                 const float *norm_w, int64_t n, int hc, int d, int iters, float eps,
                                 float norm_eps, uint16_t *h_norm, uint16_t *y, float *pre_out,
                                 float *post_out, float *comb_out, float *mixes_out,
                                 cudaStream_t s);

// The backward of one side step (hc_backward.cu), hc == 4.
size_t backward_workspace_bytes(int64_t n, int d);
size_t backward_static_scratch_bytes();
cudaError_t backward_static_scratch(void **ptr);
cudaError_t launch_block_step_backward(const uint16_t *x, const float *pre_mix, const uint16_t *f,
                                       const float *hc_fn, const float *hc_scale,
                                       const float *hc_base, const float *norm_w, int64_t n, int d,
                                       int iters, float eps, float norm_eps, const float *g_hn,
                                       const float *g_y, const float *g_pre, float *g_x,
                                       float *g_pm, float *g_f, float *g_fn, float *g_scale,
                                       float *g_base, float *g_w, void *workspace, cudaStream_t s);

// The fused persistent-cluster path (hc_block_cluster.cu).  Supported when d
// is a multiple of 1024 and one stream's weight fragments fit a tensor-memory
// quadrant (d <= 7168).  With f == nullptr it computes a1-a3 only.
bool cluster_path_supported(int d);

cudaError_t launch_block_cluster(const uint16_t *x, const float *pre_mix, const uint16_t *f,
                                 const float *hc_fn, const float *hc_scale, const float *hc_base,
                                 const float *norm_w, int64_t n, int d, int iters, float eps,
                                 float norm_eps, uint16_t *h_norm, uint16_t *y, float *pre_out,
                                 float *post_out, float *comb_out, float *mixes_out,
                                 cudaStream_t s);

// The chain kernel (hc_slices.cu): supported when d is a multiple of 1024 and
// one stream's weight fragments fit a tensor-memory quadrant (d <= 7168).
bool slices_supported(int d);

// The chain of side steps fused across sides (hc_slices.cu).  A state buffer
// holds the [n, 32] coefficient rows, then the kernel's scratch.
size_t chain_state_bytes(int64_t n);

cudaError_t launch_slices_begin(const uint16_t *x, const float *pre_mix, const float *hc_fn,
                                const float *hc_scale, const float *hc_base, int64_t n, int d,
                                int iters, float eps, float norm_eps, float *state_out,
                                float *pre_out, uint16_t *h_pre_out, cudaStream_t s);

// hc_fn_next == nullptr: the last side (no phase 1 of a next side).  At most one
// of h_norm (this side's) and h_pre_out (the next side's bf16 h) is given.
cudaError_t launch_slices_side(const uint16_t *x, const uint16_t *f, const float *state_in,
                               const float *norm_w, const float *hc_fn_next,
                               const float *hc_scale_next, const float *hc_base_next, int64_t n,
                               int d, int iters, float eps, float norm_eps, uint16_t *h_norm,
                               uint16_t *y, float *state_out, float *pre_out, uint16_t *h_pre_out,
                               cudaStream_t s);

// a5 of the chain in model order: h_norm (and / or its MXFP8 cast) from the
// bf16 h and the statistic in the coefficient rows (hc_kernels_simple.cu).
cudaError_t launch_chain_norm(const uint16_t *h_pre, const float *state, const float *norm_w,
                              int64_t n, int d, uint16_t *out, uint8_t *codes, uint8_t *scales,
                              cudaStream_t s);

// Synchronise `s`, then read and clear the device flag that bounded waits set
// when they time out (each kernel file keeps its own flag).
cudaError_t consume_device_error(cudaStream_t s, unsigned int *flag);
cudaError_t consume_slices_device_error(cudaStream_t s, unsigned int *flag);
cudaError_t consume_backward_device_error(cudaStream_t s, unsigned int *flag);
cudaError_t consume_proj_device_error(cudaStream_t s, unsigned int *flag);
// one warp waits on a barrier nothing arrives on (the bounded-wait self-test)
cudaError_t launch_selftest_wait(cudaStream_t s);

}  // namespace hc
