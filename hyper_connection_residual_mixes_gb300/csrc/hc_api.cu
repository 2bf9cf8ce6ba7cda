// hc_api.cu -- the C ABI of libhc: host-side validation, then dispatch to the
// kernels.  Nothing here allocates device memory; every launch goes on the
// caller's stream.  See include/hc.h for the contract of each entry point.
#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/hc.h"
#include "hc_backward_generic.h"
#include "hc_launch.h"

namespace {

thread_local int g_last_cuda_error = 0;

constexpr int kMaxD = 16384;

struct Span {
    uintptr_t lo, hi;  // [lo, hi); empty when lo == hi
};

Span span(const void *p, int64_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Span{a, a + (uintptr_t)(bytes > 0 ? bytes : 0)};
}

bool overlaps(Span a, Span b) {
    if (a.lo == a.hi || b.lo == b.hi) return false;
    return a.lo < b.hi && b.lo < a.hi;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool finite_nonneg(float v) { return std::isfinite(v) && v >= 0.0f; }

hc_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return HC_OK;
    g_last_cuda_error = (int)e;
    return HC_ERR_CUDA;
}

// Shape checks shared by the entry points.  n == 0 is valid (no work).
hc_status check_shape(int64_t n, int hc, int d, bool uses_d) {
    if (n < 0) return HC_ERR_INVALID_ARG;
    if (hc <= 0) return HC_ERR_INVALID_ARG;
    if (hc != 2 && hc != 4 && hc != 8) return HC_ERR_UNSUPPORTED;  // the compiled stream counts
    if (uses_d) {
        if (d <= 0) return HC_ERR_INVALID_ARG;
        if (d % 64 != 0 || d > kMaxD) return HC_ERR_UNSUPPORTED;
        // n * hc * d elements must be addressable with 64-bit byte offsets
        if (n > (INT64_MAX / 8) / ((int64_t)hc * d)) return HC_ERR_INVALID_ARG;
    } else if (n > INT64_MAX / 1024) {
        return HC_ERR_INVALID_ARG;
    }
    return HC_OK;
}

// Every output span must be disjoint from every input span and from the other outputs.
hc_status check_alias(const Span *outs, int n_out, const Span *ins, int n_in) {
    for (int i = 0; i < n_out; ++i) {
        for (int j = 0; j < n_in; ++j)
            if (overlaps(outs[i], ins[j])) return HC_ERR_ALIAS;
        for (int j = i + 1; j < n_out; ++j)
            if (overlaps(outs[i], outs[j])) return HC_ERR_ALIAS;
    }
    return HC_OK;
}

}  // namespace

extern "C" {

const char *hc_status_string(hc_status status) {
    switch (status) {
        case HC_OK: return "HC_OK";
        case HC_ERR_INVALID_ARG: return "HC_ERR_INVALID_ARG: null pointer, bad size or bad scalar";
        case HC_ERR_UNSUPPORTED: return "HC_ERR_UNSUPPORTED: needs hc == 4 and d a multiple of 64 in [64, 16384]";
        case HC_ERR_MISALIGNED: return "HC_ERR_MISALIGNED: every pointer must be 16-byte aligned";
        case HC_ERR_ALIAS: return "HC_ERR_ALIAS: an output overlaps an input or another output";
        case HC_ERR_CUDA: return "HC_ERR_CUDA: a CUDA call failed (see hc_last_cuda_error)";
        case HC_ERR_TIMEOUT: return "HC_ERR_TIMEOUT: a kernel gave up waiting on a barrier";
    }
    return "unknown hc_status";
}

int hc_last_cuda_error(void) { return g_last_cuda_error; }

int hc_version(void) { return 100; }

hc_status hc_consume_device_error(cudaStream_t stream) {
    unsigned int flag = 0, flag_chain = 0, flag_bwd = 0, flag_proj = 0;
    hc_status st = cuda_status(hc::consume_device_error(stream, &flag));
    if (st != HC_OK) return st;
    st = cuda_status(hc::consume_slices_device_error(stream, &flag_chain));
    if (st != HC_OK) return st;
    st = cuda_status(hc::consume_backward_device_error(stream, &flag_bwd));
    if (st != HC_OK) return st;
    st = cuda_status(hc::consume_proj_device_error(stream, &flag_proj));
    if (st != HC_OK) return st;
    return (flag | flag_chain | flag_bwd | flag_proj) ? HC_ERR_TIMEOUT : HC_OK;
}

hc_status hc_selftest_barrier_timeout(cudaStream_t stream) {
    return cuda_status(hc::launch_selftest_wait(stream));
}

hc_status hc_split_sinkhorn(const float *mixes, const float *hc_scale, const float *hc_base,
                            int64_t n, int hc, int sinkhorn_iters, float eps, float *pre,
                            float *post, float *comb, cudaStream_t stream) {
    hc_status st = check_shape(n, hc, 0, false);
    if (st != HC_OK) return st;
    if (sinkhorn_iters < 1 || !finite_nonneg(eps)) return HC_ERR_INVALID_ARG;
    if (n == 0) return HC_OK;
    if (!mixes || !hc_scale || !hc_base || !pre || !post || !comb) return HC_ERR_INVALID_ARG;
    const void *ptrs[] = {mixes, hc_scale, hc_base, pre, post, comb};
    for (const void *p : ptrs)
        if (!aligned16(p)) return HC_ERR_MISALIGNED;
    const int64_t mix = (int64_t)(2 + hc) * hc;
    const Span ins[] = {span(mixes, n * mix * 4), span(hc_scale, 12), span(hc_base, mix * 4)};
    const Span outs[] = {span(pre, n * hc * 4), span(post, n * hc * 4), span(comb, n * hc * hc * 4)};
    if ((st = check_alias(outs, 3, ins, 3)) != HC_OK) return st;
    return cuda_status(hc::launch_split_sinkhorn(mixes, hc_scale, hc_base, n, hc, sinkhorn_iters, eps,
                                                 pre, post, comb, stream));
}

hc_status hc_mixes(const uint16_t *x, const float *hc_fn, const float *hc_scale,
                   const float *hc_base, int64_t n, int hc, int d, int sinkhorn_iters,
                   float eps, float norm_eps, float *pre, float *post, float *comb,
                   float *mixes_out, cudaStream_t stream) {
    hc_status st = check_shape(n, hc, d, true);
    if (st != HC_OK) return st;
    if (sinkhorn_iters < 1 || !finite_nonneg(eps) || !finite_nonneg(norm_eps))
        return HC_ERR_INVALID_ARG;
    if (n == 0) return HC_OK;
    if (!x || !hc_fn || !hc_scale || !hc_base || !pre || !post || !comb) return HC_ERR_INVALID_ARG;
    const void *ptrs[] = {x, hc_fn, hc_scale, hc_base, pre, post, comb};
    for (const void *p : ptrs)
        if (!aligned16(p)) return HC_ERR_MISALIGNED;
    if (mixes_out && !aligned16(mixes_out)) return HC_ERR_MISALIGNED;
    const int64_t mix = (int64_t)(2 + hc) * hc, K = (int64_t)hc * d;
    const Span ins[] = {span(x, n * K * 2), span(hc_fn, mix * K * 4), span(hc_scale, 12),
                        span(hc_base, mix * 4)};
    const Span outs[] = {span(pre, n * hc * 4), span(post, n * hc * 4),
                         span(comb, n * hc * hc * 4), span(mixes_out, mixes_out ? n * mix * 4 : 0)};
    if ((st = check_alias(outs, 4, ins, 4)) != HC_OK) return st;
    if (hc == 4 && hc::cluster_path_supported(d))
        return cuda_status(hc::launch_block_cluster(x, nullptr, nullptr, hc_fn, hc_scale, hc_base,
                                                    nullptr, n, d, sinkhorn_iters, eps, norm_eps,
                                                    nullptr, nullptr, pre, post, comb, mixes_out,
                                                    stream));
    return cuda_status(hc::launch_tokens_simple(x, nullptr, nullptr, hc_fn, hc_scale, hc_base,
                                                nullptr, n, hc, d, sinkhorn_iters, eps, norm_eps,
                                                nullptr, nullptr, pre, post, comb, mixes_out,
                                                stream));
}

hc_status hc_pre_norm(const uint16_t *x, const float *pre_mix, const float *norm_w, int64_t n,
                      int hc, int d, float norm_eps, uint16_t *out, cudaStream_t stream) {
    hc_status st = check_shape(n, hc, d, true);
    if (st != HC_OK) return st;
    if (!finite_nonneg(norm_eps)) return HC_ERR_INVALID_ARG;
    if (n == 0) return HC_OK;
    if (!x || !pre_mix || !norm_w || !out) return HC_ERR_INVALID_ARG;
    const void *ptrs[] = {x, pre_mix, norm_w, out};
    for (const void *p : ptrs)
        if (!aligned16(p)) return HC_ERR_MISALIGNED;
    const Span ins[] = {span(x, n * hc * d * 2), span(pre_mix, n * hc * 4), span(norm_w, d * 4)};
    const Span outs[] = {span(out, n * d * 2)};
    if ((st = check_alias(outs, 1, ins, 3)) != HC_OK) return st;
    return cuda_status(hc::launch_pre_norm(x, pre_mix, norm_w, n, hc, d, norm_eps, out, stream));
}

size_t hc_block_step_backward_workspace_bytes(int64_t n, int hc, int d) {
    if (check_shape(n, hc, d, true) != HC_OK) return 0;
    return hc == 4 ? hc::backward_workspace_bytes(n, d) : hc::backward_generic_workspace_bytes(n, hc, d);
}

hc_status hc_block_step_backward(const uint16_t *x, const float *pre_mix, const uint16_t *f,
                                 const float *hc_fn, const float *hc_scale, const float *hc_base,
                                 const float *norm_w, int64_t n, int hc, int d, int sinkhorn_iters,
                                 float eps, float norm_eps, const float *g_h_norm, const float *g_y,
                                 const float *g_pre, float *g_x, float *g_pre_mix, float *g_f,
                                 float *g_hc_fn, float *g_hc_scale, float *g_hc_base,
                                 float *g_norm_w, void *workspace, size_t workspace_bytes,
                                 cudaStream_t stream) {
    hc_status st = check_shape(n, hc, d, true);
    if (st != HC_OK) return st;
    if (sinkhorn_iters < 1 || sinkhorn_iters > 128 || !finite_nonneg(eps) || !finite_nonneg(norm_eps))
        return HC_ERR_INVALID_ARG;
    if (n == 0) return HC_OK;
    if (!x || !pre_mix || !f || !hc_fn || !hc_scale || !hc_base || !norm_w || !g_h_norm || !g_y ||
        !g_x || !g_pre_mix || !g_f || !g_hc_fn || !g_hc_scale || !g_hc_base || !g_norm_w || !workspace)
        return HC_ERR_INVALID_ARG;
    if (workspace_bytes < hc_block_step_backward_workspace_bytes(n, hc, d)) return HC_ERR_INVALID_ARG;
    const void *ptrs[] = {x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, g_h_norm, g_y, g_x,
                          g_pre_mix, g_f, g_hc_fn, g_hc_scale, g_hc_base, g_norm_w, workspace};
    for (const void *p : ptrs)
        if (!aligned16(p)) return HC_ERR_MISALIGNED;
    if (g_pre && !aligned16(g_pre)) return HC_ERR_MISALIGNED;
    const int64_t mix = (int64_t)(2 + hc) * hc, K = (int64_t)hc * d;
    const Span ins[] = {span(x, n * K * 2), span(pre_mix, n * hc * 4), span(f, n * d * 2),
                        span(hc_fn, mix * K * 4), span(hc_scale, 12), span(hc_base, mix * 4),
                        span(norm_w, d * 4), span(g_h_norm, n * d * 4), span(g_y, n * K * 4),
                        span(g_pre, g_pre ? n * hc * 4 : 0)};
    const Span outs[] = {span(g_x, n * K * 4), span(g_pre_mix, n * hc * 4), span(g_f, n * d * 4),
                         span(g_hc_fn, mix * K * 4), span(g_hc_scale, 12), span(g_hc_base, mix * 4),
                         span(g_norm_w, d * 4), span(workspace, (int64_t)workspace_bytes)};
    if ((st = check_alias(outs, 8, ins, 10)) != HC_OK) return st;
    if (hc != 4)  // two or eight streams: the plain kernels of hc_backward_generic.cu
        return cuda_status(hc::launch_block_step_backward_generic(
            hc, x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, n, d, sinkhorn_iters, eps, norm_eps,
            g_h_norm, g_y, g_pre, g_x, g_pre_mix, g_f, g_hc_fn, g_hc_scale, g_hc_base, g_norm_w,
            workspace, stream));
    return cuda_status(hc::launch_block_step_backward(
        x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, n, d, sinkhorn_iters, eps, norm_eps,
        g_h_norm, g_y, g_pre, g_x, g_pre_mix, g_f, g_hc_fn, g_hc_scale, g_hc_base, g_norm_w,
        workspace, stream));
}

hc_status hc_block_step_backward_no_workspace(
    const uint16_t *x, const float *pre_mix, const uint16_t *f, const float *hc_fn,
    const float *hc_scale, const float *hc_base, const float *norm_w, int64_t n, int hc, int d,
    int sinkhorn_iters, float eps, float norm_eps, const float *g_h_norm, const float *g_y,
    const float *g_pre, float *g_x, float *g_pre_mix, float *g_f, float *g_hc_fn, float *g_hc_scale,
    float *g_hc_base, float *g_norm_w, cudaStream_t stream) {
    hc_status st = check_shape(n, hc, d, true);
    if (st != HC_OK) return st;
    if (hc != 4 || hc::backward_workspace_bytes(n, d) > hc::backward_static_scratch_bytes())
        return HC_ERR_UNSUPPORTED;
    if (n == 0) return HC_OK;
    void *scratch = nullptr;
    if ((st = cuda_status(hc::backward_static_scratch(&scratch))) != HC_OK) return st;
    return hc_block_step_backward(x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, n, hc, d,
                                  sinkhorn_iters, eps, norm_eps, g_h_norm, g_y, g_pre, g_x,
                                  g_pre_mix, g_f, g_hc_fn, g_hc_scale, g_hc_base, g_norm_w, scratch,
                                  hc::backward_static_scratch_bytes(), stream);
}

hc_status hc_mxfp8_cast(const uint16_t *in, int64_t rows, int d, uint8_t *codes, uint8_t *scales,
                        cudaStream_t stream) {
    if (rows < 0 || d <= 0) return HC_ERR_INVALID_ARG;
    if (d % 32 != 0) return HC_ERR_UNSUPPORTED;
    if (rows > (INT64_MAX / 8) / d) return HC_ERR_INVALID_ARG;
    if (rows == 0) return HC_OK;
    if (!in || !codes || !scales) return HC_ERR_INVALID_ARG;
    if (!aligned16(in) || !aligned16(codes)) return HC_ERR_MISALIGNED;
    const Span ins[] = {span(in, rows * d * 2)};
    const Span outs[] = {span(codes, rows * d), span(scales, rows * (d / 32))};
    hc_status st = check_alias(outs, 2, ins, 1);
    if (st != HC_OK) return st;
    return cuda_status(hc::launch_mxfp8_cast(in, rows, d, codes, scales, stream));
}

hc_status hc_pre_norm_mxfp8(const uint16_t *x, const float *pre_mix, const float *norm_w, int64_t n,
                            int hc, int d, float norm_eps, uint16_t *h_norm_out, uint8_t *codes,
                            uint8_t *scales, cudaStream_t stream) {
    hc_status st = check_shape(n, hc, d, true);
    if (st != HC_OK) return st;
    if (!finite_nonneg(norm_eps)) return HC_ERR_INVALID_ARG;
    if (n == 0) return HC_OK;
    if (!x || !pre_mix || !norm_w || !codes || !scales) return HC_ERR_INVALID_ARG;
    const void *ptrs[] = {x, pre_mix, norm_w, codes};
    for (const void *p : ptrs)
        if (!aligned16(p)) return HC_ERR_MISALIGNED;
    if (h_norm_out && !aligned16(h_norm_out)) return HC_ERR_MISALIGNED;
    const Span ins[] = {span(x, n * hc * d * 2), span(pre_mix, n * hc * 4), span(norm_w, d * 4)};
    const Span outs[] = {span(codes, n * d), span(scales, n * (d / 32)),
                         span(h_norm_out, h_norm_out ? n * d * 2 : 0)};
    if ((st = check_alias(outs, 3, ins, 3)) != HC_OK) return st;
    return cuda_status(hc::launch_pre_norm_mxfp8(x, pre_mix, norm_w, n, hc, d, norm_eps, h_norm_out,
                                                 codes, scales, stream));
}

hc_status hc_post(const uint16_t *f, const uint16_t *residual, const float *post,
                  const float *comb, int64_t n, int hc, int d, uint16_t *y,
                  cudaStream_t stream) {
    hc_status st = check_shape(n, hc, d, true);
    if (st != HC_OK) return st;
    if (n == 0) return HC_OK;
    if (!f || !residual || !post || !comb || !y) return HC_ERR_INVALID_ARG;
    const void *ptrs[] = {f, residual, post, comb, y};
    for (const void *p : ptrs)
        if (!aligned16(p)) return HC_ERR_MISALIGNED;
    const Span ins[] = {span(f, n * d * 2), span(residual, n * hc * d * 2), span(post, n * hc * 4),
                        span(comb, n * hc * hc * 4)};
    const Span outs[] = {span(y, n * hc * d * 2)};
    if ((st = check_alias(outs, 1, ins, 4)) != HC_OK) return st;
    return cuda_status(hc::launch_post(f, residual, post, comb, n, hc, d, y, stream));
}

hc_status hc_block_step(const uint16_t *x, const float *pre_mix, const uint16_t *f,
                        const float *hc_fn, const float *hc_scale, const float *hc_base,
                        const float *norm_w, int64_t n, int hc, int d, int sinkhorn_iters,
                        float eps, float norm_eps, uint16_t *h_norm, uint16_t *y,
                        float *pre_out, float *post_out, float *comb_out,
                        cudaStream_t stream) {
    hc_status st = check_shape(n, hc, d, true);
    if (st != HC_OK) return st;
    if (sinkhorn_iters < 1 || !finite_nonneg(eps) || !finite_nonneg(norm_eps))
        return HC_ERR_INVALID_ARG;
    if (n == 0) return HC_OK;
    if (!x || !pre_mix || !f || !hc_fn || !hc_scale || !hc_base || !norm_w || !h_norm || !y ||
        !pre_out)
        return HC_ERR_INVALID_ARG;
    const void *ptrs[] = {x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, h_norm, y, pre_out};
    for (const void *p : ptrs)
        if (!aligned16(p)) return HC_ERR_MISALIGNED;
    if ((post_out && !aligned16(post_out)) || (comb_out && !aligned16(comb_out)))
        return HC_ERR_MISALIGNED;
    const int64_t mix = (int64_t)(2 + hc) * hc, K = (int64_t)hc * d;
    const Span ins[] = {span(x, n * K * 2),        span(pre_mix, n * hc * 4), span(f, n * d * 2),
                        span(hc_fn, mix * K * 4),  span(hc_scale, 12),        span(hc_base, mix * 4),
                        span(norm_w, d * 4)};
    const Span outs[] = {span(h_norm, n * d * 2), span(y, n * K * 2), span(pre_out, n * hc * 4),
                         span(post_out, post_out ? n * hc * 4 : 0),
                         span(comb_out, comb_out ? n * hc * hc * 4 : 0)};
    if ((st = check_alias(outs, 5, ins, 7)) != HC_OK) return st;
    if (hc == 4 && hc::cluster_path_supported(d))
        return cuda_status(hc::launch_block_cluster(x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w,
                                                    n, d, sinkhorn_iters, eps, norm_eps, h_norm, y,
                                                    pre_out, post_out, comb_out, nullptr, stream));
    return cuda_status(hc::launch_tokens_simple(x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, n,
                                                hc, d, sinkhorn_iters, eps, norm_eps, h_norm, y,
                                                pre_out, post_out, comb_out, nullptr, stream));
}

size_t hc_chain_state_bytes(int64_t n, int hc, int d) {
    if (check_shape(n, hc, d, true) != HC_OK || hc != 4 || !hc::slices_supported(d)) return 0;
    return hc::chain_state_bytes(n);
}

hc_status hc_chain_begin(const uint16_t *x, const float *pre_mix, const float *hc_fn,
                         const float *hc_scale, const float *hc_base, int64_t n, int hc, int d,
                         int sinkhorn_iters, float eps, float norm_eps, float *state_out,
                         size_t state_bytes, float *pre_out, uint16_t *h_pre_out,
                         cudaStream_t stream) {
    hc_status st = check_shape(n, hc, d, true);
    if (st != HC_OK) return st;
    if (sinkhorn_iters < 1 || !finite_nonneg(eps) || !finite_nonneg(norm_eps))
        return HC_ERR_INVALID_ARG;
    if (hc != 4 || !hc::slices_supported(d)) return HC_ERR_UNSUPPORTED;
    if (n == 0) return HC_OK;
    if (!x || !pre_mix || !hc_fn || !hc_scale || !hc_base || !state_out) return HC_ERR_INVALID_ARG;
    if (state_bytes < hc::chain_state_bytes(n)) return HC_ERR_INVALID_ARG;
    const void *ptrs[] = {x, pre_mix, hc_fn, hc_scale, hc_base, state_out};
    for (const void *p : ptrs)
        if (!aligned16(p)) return HC_ERR_MISALIGNED;
    if ((pre_out && !aligned16(pre_out)) || (h_pre_out && !aligned16(h_pre_out))) return HC_ERR_MISALIGNED;
    const int64_t mix = (int64_t)(2 + hc) * hc, K = (int64_t)hc * d;
    const Span ins[] = {span(x, n * K * 2), span(pre_mix, n * hc * 4), span(hc_fn, mix * K * 4),
                        span(hc_scale, 12), span(hc_base, mix * 4)};
    const Span outs[] = {span(state_out, (int64_t)state_bytes), span(pre_out, pre_out ? n * hc * 4 : 0),
                         span(h_pre_out, h_pre_out ? n * d * 2 : 0)};
    if ((st = check_alias(outs, 3, ins, 5)) != HC_OK) return st;
    return cuda_status(hc::launch_slices_begin(x, pre_mix, hc_fn, hc_scale, hc_base, n, d,
                                               sinkhorn_iters, eps, norm_eps, state_out, pre_out,
                                               h_pre_out, stream));
}

hc_status hc_chain_side(const uint16_t *x, const uint16_t *f, const float *state_in,
                        const float *norm_w, const float *hc_fn_next, const float *hc_scale_next,
                        const float *hc_base_next, int64_t n, int hc, int d, int sinkhorn_iters,
                        float eps, float norm_eps, uint16_t *h_norm, uint16_t *y,
                        float *state_out, size_t state_bytes, float *pre_out, uint16_t *h_pre_out,
                        cudaStream_t stream) {
    hc_status st = check_shape(n, hc, d, true);
    if (st != HC_OK) return st;
    if (sinkhorn_iters < 1 || !finite_nonneg(eps) || !finite_nonneg(norm_eps))
        return HC_ERR_INVALID_ARG;
    if (hc != 4 || !hc::slices_supported(d)) return HC_ERR_UNSUPPORTED;
    if (n == 0) return HC_OK;
    const bool next = hc_fn_next != nullptr;
    if (!x || !f || !state_in || !norm_w || !y) return HC_ERR_INVALID_ARG;
    // the next side's weights come all together, with a state to write, or not at all
    if (next != (hc_scale_next != nullptr) || next != (hc_base_next != nullptr)) return HC_ERR_INVALID_ARG;
    if (next && (!state_out || state_bytes < hc::chain_state_bytes(n))) return HC_ERR_INVALID_ARG;
    // the next side's bf16 h needs a next side; it and this side's h_norm are one or the other
    if (h_pre_out && (!next || h_norm)) return HC_ERR_INVALID_ARG;
    const void *ptrs[] = {x, f, state_in, norm_w, y};
    for (const void *p : ptrs)
        if (!aligned16(p)) return HC_ERR_MISALIGNED;
    if ((h_norm && !aligned16(h_norm)) || (h_pre_out && !aligned16(h_pre_out))) return HC_ERR_MISALIGNED;
    if (next) {
        const void *nptrs[] = {hc_fn_next, hc_scale_next, hc_base_next, state_out};
        for (const void *p : nptrs)
            if (!aligned16(p)) return HC_ERR_MISALIGNED;
    }
    if (pre_out && !aligned16(pre_out)) return HC_ERR_MISALIGNED;
    const int64_t mix = (int64_t)(2 + hc) * hc, K = (int64_t)hc * d;
    const Span ins[] = {span(x, n * K * 2),
                        span(f, n * d * 2),
                        span(state_in, n * HC_STATE_FLOATS * 4),
                        span(norm_w, d * 4),
                        span(hc_fn_next, next ? mix * K * 4 : 0),
                        span(hc_scale_next, next ? 12 : 0),
                        span(hc_base_next, next ? mix * 4 : 0)};
    const Span outs[] = {span(h_norm, h_norm ? n * d * 2 : 0), span(y, n * K * 2),
                         span(state_out, next ? (int64_t)state_bytes : 0),
                         span(pre_out, (next && pre_out) ? n * hc * 4 : 0),
                         span(h_pre_out, h_pre_out ? n * d * 2 : 0)};
    if ((st = check_alias(outs, 5, ins, 7)) != HC_OK) return st;
    return cuda_status(hc::launch_slices_side(x, f, state_in, norm_w, hc_fn_next, hc_scale_next,
                                              hc_base_next, n, d, sinkhorn_iters, eps, norm_eps,
                                              h_norm, y, next ? state_out : nullptr,
                                              next ? pre_out : nullptr, h_pre_out, stream));
}

hc_status hc_chain_norm(const uint16_t *h_pre, const float *state, const float *norm_w, int64_t n,
                        int d, uint16_t *h_norm, uint8_t *codes, uint8_t *scales,
                        cudaStream_t stream) {
    if (n < 0 || d <= 0) return HC_ERR_INVALID_ARG;
    if (d % 64 != 0 || d > kMaxD) return HC_ERR_UNSUPPORTED;
    if (n > (INT64_MAX / 8) / d) return HC_ERR_INVALID_ARG;
    if (n == 0) return HC_OK;
    if (!h_pre || !state || !norm_w) return HC_ERR_INVALID_ARG;
    if ((codes == nullptr) != (scales == nullptr) || (!h_norm && !codes)) return HC_ERR_INVALID_ARG;
    const void *ptrs[] = {h_pre, state, norm_w};
    for (const void *p : ptrs)
        if (!aligned16(p)) return HC_ERR_MISALIGNED;
    if ((h_norm && !aligned16(h_norm)) || (codes && !aligned16(codes))) return HC_ERR_MISALIGNED;
    const Span ins[] = {span(h_pre, n * d * 2), span(state, n * HC_STATE_FLOATS * 4), span(norm_w, d * 4)};
    const Span outs[] = {span(h_norm, h_norm ? n * d * 2 : 0), span(codes, codes ? n * d : 0),
                         span(scales, scales ? n * (d / 32) : 0)};
    hc_status st = check_alias(outs, 3, ins, 3);
    if (st != HC_OK) return st;
    return cuda_status(hc::launch_chain_norm(h_pre, state, norm_w, n, d, h_norm, codes, scales, stream));
}

}  // extern "C"
