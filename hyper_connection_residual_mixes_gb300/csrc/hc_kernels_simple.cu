// hc_kernels_simple.cu -- straightforward kernels for every step of the
// hyper-connection side step (sm_103a).
//
//  k_split_sinkhorn  a2-a3, one thread per token row of 24 mix numbers
//                    ("Stream combination" page, hc_split_sinkhorn).
//  k_pre_norm        a4-a5, one CTA per token: collapse the streams under
//                    pre_mix, round to bf16, RMSNorm with gain (Block page,
//                    Block.hc_pre + attn_norm).
//  k_post            a6, one CTA per token (Block page, Block.hc_post).
//  k_mxfp8_cast      the MXFP8 cast of bf16 rows (Flash diagram, Cast to MXFP8).
//  k_pre_norm_mxfp8  a4-a5 with the cast in its epilogue.
//  k_tokens_simple   a1-a3 and optionally a4-a6 for TOK whole tokens per CTA
//                    (Block page, Block.hc_mixes and Block.forward); with
//                    kCoefIn, a4-a6 only, from coefficients computed before.
//  k_mixes_tiled     a1-a3 for 32 tokens per CTA with hc_fn streamed through
//                    shared memory (the projection on the tensor cores), for
//                    the stream counts and widths the fused kernel does not
//                    serve.
//
// The fused side step for hc = 4 and d a multiple of 1024 lives in
// hc_block_cluster.cu and hc_slices.cu.
#include <cuda.h>

#include "hc_device.cuh"
#include "hc_launch.h"
#include "hc_ptx.cuh"

namespace hc {

// ------------------------------------------------------------------ a2-a3
// HC streams: mix = (2 + HC) * HC numbers per row, a multiple of 4 for HC = 2, 4, 8.
template <int HC>
__global__ void __launch_bounds__(128)
k_split_sinkhorn(const float *__restrict__ mixes, const float *__restrict__ hc_scale,
                 const float *__restrict__ hc_base, int64_t n, int iters, float eps,
                 float *__restrict__ pre, float *__restrict__ post, float *__restrict__ comb) {
    constexpr int MIX = (2 + HC) * HC;
    const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (row >= n) return;
    float m[MIX];
    const float4 *src = reinterpret_cast<const float4 *>(mixes + row * MIX);
#pragma unroll
    for (int q = 0; q < MIX / 4; ++q) {
        const float4 v = __ldg(src + q);
        m[4 * q + 0] = v.x; m[4 * q + 1] = v.y; m[4 * q + 2] = v.z; m[4 * q + 3] = v.w;
    }
    float pr[HC], po[HC], c[HC * HC];
    // the fast reciprocal and exponential, as the fused kernels' owners use them
    split_sinkhorn_token_hc<HC, true>(m, __ldg(hc_scale), __ldg(hc_scale + 1), __ldg(hc_scale + 2),
                                      hc_base, iters, eps, pr, po, c);
    // 16-byte stores (hc = 2: pre and post are 8 bytes per row)
    if constexpr (HC % 4 == 0) {
#pragma unroll
        for (int k = 0; k < HC; k += 4) {
            reinterpret_cast<float4 *>(pre + row * HC + k)[0] = make_float4(pr[k], pr[k + 1], pr[k + 2], pr[k + 3]);
            reinterpret_cast<float4 *>(post + row * HC + k)[0] = make_float4(po[k], po[k + 1], po[k + 2], po[k + 3]);
        }
    } else {
        reinterpret_cast<float2 *>(pre + row * HC)[0] = make_float2(pr[0], pr[1]);
        reinterpret_cast<float2 *>(post + row * HC)[0] = make_float2(po[0], po[1]);
    }
#pragma unroll
    for (int i = 0; i < HC * HC; i += 4)
        reinterpret_cast<float4 *>(comb + row * HC * HC + i)[0] = make_float4(c[i], c[i + 1], c[i + 2], c[i + 3]);
}

cudaError_t launch_split_sinkhorn(const float *mixes, const float *hc_scale, const float *hc_base,
                                  int64_t n, int hc, int iters, float eps, float *pre, float *post,
                                  float *comb, cudaStream_t s) {
    const int threads = 128;
    const unsigned blocks = (unsigned)((n + threads - 1) / threads);
    switch (hc) {
        case 2: k_split_sinkhorn<2><<<blocks, threads, 0, s>>>(mixes, hc_scale, hc_base, n, iters, eps, pre, post, comb); break;
        case 4: k_split_sinkhorn<4><<<blocks, threads, 0, s>>>(mixes, hc_scale, hc_base, n, iters, eps, pre, post, comb); break;
        case 8: k_split_sinkhorn<8><<<blocks, threads, 0, s>>>(mixes, hc_scale, hc_base, n, iters, eps, pre, post, comb); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

// ------------------------------------------------------------------ block sum helper
template <int NT>
__device__ __forceinline__ float block_sum(float v, float *scratch /* NT/32 floats */) {
    v = warp_sum(v);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    float t = 0.0f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) t += scratch[w];
    return t;
}

// ------------------------------------------------------------------ a4-a5
// h[c] = bf16(sum_s pre_mix[s] * x[s][c]) in fp32 in stream order; then
// out[c] = bf16((h[c] * rsqrt(mean(h^2) + eps)) * w[c]).
constexpr int kRowThreads = 256;

// h_c = bf16(sum_s pre_mix[s] * x[s][c]): the product with stream 0, then a
// fused multiply-add per further stream, in stream order.
template <int HC>
__device__ __forceinline__ uint4 collapse8(const uint4 *xs, int d8, int c, const float (&p)[HC]) {
    float h[8], v[8];
    unpack8(__ldg(xs + c), v);
#pragma unroll
    for (int i = 0; i < 8; ++i) h[i] = p[0] * v[i];
#pragma unroll
    for (int s = 1; s < HC; ++s) {
        unpack8(__ldg(xs + s * d8 + c), v);
#pragma unroll
        for (int i = 0; i < 8; ++i) h[i] = fmaf(p[s], v[i], h[i]);
    }
    return pack8(h);
}

template <int HC>
__global__ void __launch_bounds__(kRowThreads)
k_pre_norm(const uint16_t *__restrict__ x, const float *__restrict__ pre_mix,
           const float *__restrict__ norm_w, int d, float norm_eps, uint16_t *__restrict__ out) {
    extern __shared__ uint4 hbuf[];  // d/8 chunks of 8 bf16
    __shared__ float red[kRowThreads / 32];
    const int64_t t = blockIdx.x;
    const int d8 = d >> 3;
    const uint4 *xs = reinterpret_cast<const uint4 *>(x + t * HC * d);
    float p[HC];
#pragma unroll
    for (int s = 0; s < HC; ++s) p[s] = __ldg(pre_mix + t * HC + s);
    float ss = 0.0f;
    for (int c = threadIdx.x; c < d8; c += kRowThreads) {
        const uint4 hb = collapse8<HC>(xs, d8, c, p);
        hbuf[c] = hb;
        float r[8];
        unpack8(hb, r);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(r[i], r[i], ss);
    }
    const float tot = block_sum<kRowThreads>(ss, red);
    const float rs = rsqrtf(tot / (float)d + norm_eps);
    uint4 *o = reinterpret_cast<uint4 *>(out + t * d);
    const float4 *w4 = reinterpret_cast<const float4 *>(norm_w);
    for (int c = threadIdx.x; c < d8; c += kRowThreads) {
        float h[8];
        unpack8(hbuf[c], h);
        const float4 wa = __ldg(w4 + 2 * c), wb = __ldg(w4 + 2 * c + 1);
        const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int i = 0; i < 8; ++i) h[i] = (h[i] * rs) * wv[i];
        o[c] = pack8(h);
    }
}

template <int HC>
cudaError_t launch_pre_norm_hc(const uint16_t *x, const float *pre_mix, const float *norm_w,
                               int64_t n, int d, float norm_eps, uint16_t *out, cudaStream_t s) {
    const size_t smem = (size_t)d * 2;
    cudaError_t e = cudaFuncSetAttribute(k_pre_norm<HC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    k_pre_norm<HC><<<(unsigned)n, kRowThreads, smem, s>>>(x, pre_mix, norm_w, d, norm_eps, out);
    return cudaGetLastError();
}

cudaError_t launch_pre_norm(const uint16_t *x, const float *pre_mix, const float *norm_w,
                            int64_t n, int hc, int d, float norm_eps, uint16_t *out, cudaStream_t s) {
    switch (hc) {
        case 2: return launch_pre_norm_hc<2>(x, pre_mix, norm_w, n, d, norm_eps, out, s);
        case 4: return launch_pre_norm_hc<4>(x, pre_mix, norm_w, n, d, norm_eps, out, s);
        case 8: return launch_pre_norm_hc<8>(x, pre_mix, norm_w, n, d, norm_eps, out, s);
        default: return cudaErrorInvalidValue;
    }
}

// ------------------------------------------------------------------ MXFP8 cast
// DeepSeek V4.1 Flash diagram, block "Cast to MXFP8".  The channels of a row
// are cut into groups of 32.  A group's scale is the smallest power of two at
// or above max(amax, 1e-4) / 448 (the division in fp32, correctly rounded),
// written as its biased exponent (UE8M0); every channel is written as the
// E4M3 number nearest to x / scale (ties to even) after clamping to
// [-448, 448].  Each thread holds one 8-channel chunk, so a group is four
// consecutive lanes; every loop below runs the same number of times in all
// lanes of a warp, so the group shuffles always see a full warp.
__device__ __forceinline__ int mx_scale_exp(float amax) {
    const float q = __fdiv_rn(fmaxf(amax, 1e-4f), 448.0f);  // a normal float here
    const uint32_t b = __float_as_uint(q);
    // ceil(log2(q)): the exponent, plus one unless q is a power of two
    return (int)((b >> 23) & 0xffu) - 127 + ((b & 0x7fffffu) ? 1 : 0);
}
// two fp32 values -> two E4M3 bytes (lo in the low byte), nearest even, saturating
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
// eight channels (exact bf16 values) of a group with scale 2^ex -> eight bytes
__device__ __forceinline__ uint2 mx_codes8(const float (&v)[8], int ex) {
    const float inv = __uint_as_float((uint32_t)(127 - ex) << 23);  // 2^-ex, exact
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        w[i] = e4m3x2(fminf(fmaxf(v[2 * i] * inv, -448.0f), 448.0f),
                      fminf(fmaxf(v[2 * i + 1] * inv, -448.0f), 448.0f));
    return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}
// the largest magnitude of the group (four lanes), then its scale exponent
__device__ __forceinline__ int mx_group_exp(const float (&v)[8]) {
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(v[i]));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
    return mx_scale_exp(am);
}

constexpr int kCastThreads = 256;

// bf16 rows -> E4M3 codes + UE8M0 scale bytes; chunks = rows * d / 8 (a multiple of 4)
__global__ void __launch_bounds__(kCastThreads)
k_mxfp8_cast(const uint16_t *__restrict__ in, int64_t chunks, uint8_t *__restrict__ codes,
             uint8_t *__restrict__ scales) {
    const uint4 *in8 = reinterpret_cast<const uint4 *>(in);
    uint2 *out8 = reinterpret_cast<uint2 *>(codes);
    for (int64_t base = (int64_t)blockIdx.x * kCastThreads; base < chunks;
         base += (int64_t)gridDim.x * kCastThreads) {
        const int64_t c = base + threadIdx.x;
        const bool live = c < chunks;
        float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (live) unpack8(__ldg(in8 + c), v);
        const int ex = mx_group_exp(v);
        if (live) {
            out8[c] = mx_codes8(v, ex);
            if ((c & 3) == 0) scales[c >> 2] = (uint8_t)(ex + 127);
        }
    }
}

cudaError_t launch_mxfp8_cast(const uint16_t *in, int64_t rows, int d, uint8_t *codes,
                              uint8_t *scales, cudaStream_t s) {
    const int64_t chunks = rows * (int64_t)(d / 8);
    int64_t blocks = (chunks + kCastThreads - 1) / kCastThreads;
    if (blocks > 152 * 16) blocks = 152 * 16;  // grid-stride beyond 16 CTAs per SM
    k_mxfp8_cast<<<(unsigned)blocks, kCastThreads, 0, s>>>(in, chunks, codes, scales);
    return cudaGetLastError();
}

// a5 for the chain in model order: the chain's launch for side i wrote side
// i + 1's bf16 h (hc_pre of y_i with side i's pre) and the RMSNorm statistic of
// that h into the coefficient rows; here h_norm = bf16((h * rs) * w), the
// products of the fused kernels, with rs read from the rows (index 20), and
// optionally its MXFP8 codes and scales (the cast above).  chunks = n * d / 8.
__global__ void __launch_bounds__(kCastThreads)
k_chain_norm(const uint16_t *__restrict__ h_pre, const float *__restrict__ state,
             const float *__restrict__ norm_w, int d8, int64_t chunks, uint16_t *__restrict__ out,
             uint8_t *__restrict__ codes, uint8_t *__restrict__ scales) {
    const uint4 *in8 = reinterpret_cast<const uint4 *>(h_pre);
    const float4 *w4 = reinterpret_cast<const float4 *>(norm_w);
    for (int64_t base = (int64_t)blockIdx.x * kCastThreads; base < chunks;
         base += (int64_t)gridDim.x * kCastThreads) {
        const int64_t c = base + threadIdx.x;
        const bool live = c < chunks;
        float h[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (live) {
            const int64_t t = c / d8;
            const int cc = (int)(c - t * d8);
            const float rs = __ldg(state + t * 32 + 20);
            unpack8(__ldg(in8 + c), h);
            const float4 wa = __ldg(w4 + 2 * cc), wb = __ldg(w4 + 2 * cc + 1);
            const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) h[i] = (h[i] * rs) * wv[i];
        }
        const uint4 hb = pack8(h);
        if (live && out) reinterpret_cast<uint4 *>(out)[c] = hb;
        if (codes) {  // uniform across the grid: the group shuffles see full warps
            float hn[8];
            unpack8(hb, hn);
            const int ex = mx_group_exp(hn);
            if (live) {
                reinterpret_cast<uint2 *>(codes)[c] = mx_codes8(hn, ex);
                if ((c & 3) == 0) scales[c >> 2] = (uint8_t)(ex + 127);
            }
        }
    }
}

cudaError_t launch_chain_norm(const uint16_t *h_pre, const float *state, const float *norm_w,
                              int64_t n, int d, uint16_t *out, uint8_t *codes, uint8_t *scales,
                              cudaStream_t s) {
    const int64_t chunks = n * (int64_t)(d / 8);
    int64_t blocks = (chunks + kCastThreads - 1) / kCastThreads;
    if (blocks > 152 * 16) blocks = 152 * 16;
    k_chain_norm<<<(unsigned)blocks, kCastThreads, 0, s>>>(h_pre, state, norm_w, d / 8, chunks, out,
                                                           codes, scales);
    return cudaGetLastError();
}

// a4-a5 and the cast in one pass: h_norm as k_pre_norm computes it, then its
// MXFP8 codes and scales; the bf16 h_norm is written too when out is given.
template <int HC>
__global__ void __launch_bounds__(kRowThreads)
k_pre_norm_mxfp8(const uint16_t *__restrict__ x, const float *__restrict__ pre_mix,
                 const float *__restrict__ norm_w, int d, float norm_eps,
                 uint16_t *__restrict__ out, uint8_t *__restrict__ codes,
                 uint8_t *__restrict__ scales) {
    extern __shared__ uint4 hbuf[];  // d/8 chunks of 8 bf16
    __shared__ float red[kRowThreads / 32];
    const int64_t t = blockIdx.x;
    const int d8 = d >> 3;
    const uint4 *xs = reinterpret_cast<const uint4 *>(x + t * HC * d);
    float p[HC];
#pragma unroll
    for (int s = 0; s < HC; ++s) p[s] = __ldg(pre_mix + t * HC + s);
    float ss = 0.0f;
    for (int c = threadIdx.x; c < d8; c += kRowThreads) {
        const uint4 hb = collapse8<HC>(xs, d8, c, p);
        hbuf[c] = hb;
        float r[8];
        unpack8(hb, r);
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(r[i], r[i], ss);
    }
    const float tot = block_sum<kRowThreads>(ss, red);
    const float rs = rsqrtf(tot / (float)d + norm_eps);
    const float4 *w4 = reinterpret_cast<const float4 *>(norm_w);
    for (int base = 0; base < d8; base += kRowThreads) {
        const int c = base + threadIdx.x;
        const bool live = c < d8;
        float h[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        if (live) {
            unpack8(hbuf[c], h);
            const float4 wa = __ldg(w4 + 2 * c), wb = __ldg(w4 + 2 * c + 1);
            const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) h[i] = (h[i] * rs) * wv[i];
        }
        const uint4 hb = pack8(h);  // h_norm, rounded to bf16
        float hn[8];
        unpack8(hb, hn);
        const int ex = mx_group_exp(hn);
        if (live) {
            if (out) reinterpret_cast<uint4 *>(out + t * d)[c] = hb;
            reinterpret_cast<uint2 *>(codes + t * d)[c] = mx_codes8(hn, ex);
            if ((c & 3) == 0) scales[t * (d >> 5) + (c >> 2)] = (uint8_t)(ex + 127);
        }
    }
}

template <int HC>
cudaError_t launch_pre_norm_mxfp8_hc(const uint16_t *x, const float *pre_mix, const float *norm_w,
                                     int64_t n, int d, float norm_eps, uint16_t *out, uint8_t *codes,
                                     uint8_t *scales, cudaStream_t s) {
    const size_t smem = (size_t)d * 2;
    cudaError_t e = cudaFuncSetAttribute(k_pre_norm_mxfp8<HC>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k_pre_norm_mxfp8<HC><<<(unsigned)n, kRowThreads, smem, s>>>(x, pre_mix, norm_w, d, norm_eps, out,
                                                                codes, scales);
    return cudaGetLastError();
}

cudaError_t launch_pre_norm_mxfp8(const uint16_t *x, const float *pre_mix, const float *norm_w,
                                  int64_t n, int hc, int d, float norm_eps, uint16_t *out,
                                  uint8_t *codes, uint8_t *scales, cudaStream_t s) {
    switch (hc) {
        case 2: return launch_pre_norm_mxfp8_hc<2>(x, pre_mix, norm_w, n, d, norm_eps, out, codes, scales, s);
        case 4: return launch_pre_norm_mxfp8_hc<4>(x, pre_mix, norm_w, n, d, norm_eps, out, codes, scales, s);
        case 8: return launch_pre_norm_mxfp8_hc<8>(x, pre_mix, norm_w, n, d, norm_eps, out, codes, scales, s);
        default: return cudaErrorInvalidValue;
    }
}

// ------------------------------------------------------------------ a6
// y[k][c] = bf16(post[k] * f[c] + sum_j comb[j][k] * x[j][c]), fp32, j in order.
template <int HC>
__global__ void __launch_bounds__(kRowThreads)
k_post(const uint16_t *__restrict__ f, const uint16_t *__restrict__ residual,
       const float *__restrict__ post, const float *__restrict__ comb, int d,
       uint16_t *__restrict__ y) {
    const int64_t t = blockIdx.x;
    const int d8 = d >> 3;
    float po[HC], cm[HC * HC];
#pragma unroll
    for (int k = 0; k < HC; ++k) po[k] = __ldg(post + t * HC + k);
#pragma unroll
    for (int i = 0; i < HC * HC; ++i) cm[i] = __ldg(comb + t * HC * HC + i);
    const uint4 *fs = reinterpret_cast<const uint4 *>(f + t * d);
    const uint4 *xs = reinterpret_cast<const uint4 *>(residual + t * HC * d);
    uint4 *ys = reinterpret_cast<uint4 *>(y + t * HC * d);
    for (int c = threadIdx.x; c < d8; c += kRowThreads) {
        float fv[8], xv[HC][8];
        unpack8(__ldg(fs + c), fv);
#pragma unroll
        for (int j = 0; j < HC; ++j) unpack8(__ldg(xs + j * d8 + c), xv[j]);
#pragma unroll
        for (int k = 0; k < HC; ++k) {
            float o[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float acc = po[k] * fv[i];
#pragma unroll
                for (int j = 0; j < HC; ++j) acc = fmaf(cm[j * HC + k], xv[j][i], acc);
                o[i] = acc;
            }
            ys[k * d8 + c] = pack8(o);
        }
    }
}

template <int HC>
cudaError_t launch_post_hc(const uint16_t *f, const uint16_t *residual, const float *post,
                           const float *comb, int64_t n, int d, uint16_t *y, cudaStream_t s) {
    k_post<HC><<<(unsigned)n, kRowThreads, 0, s>>>(f, residual, post, comb, d, y);
    return cudaGetLastError();
}

cudaError_t launch_post(const uint16_t *f, const uint16_t *residual, const float *post,
                        const float *comb, int64_t n, int hc, int d, uint16_t *y, cudaStream_t s) {
    switch (hc) {
        case 2: return launch_post_hc<2>(f, residual, post, comb, n, d, y, s);
        case 4: return launch_post_hc<4>(f, residual, post, comb, n, d, y, s);
        case 8: return launch_post_hc<8>(f, residual, post, comb, n, d, y, s);
        default: return cudaErrorInvalidValue;
    }
}

// ------------------------------------------------------------------ a1-a6, TOK tokens per CTA
// Phase 1: every thread walks 8-wide chunks of the flattened hc*d axis,
// accumulating the 24 partial dot products and the sum of squares of each of
// the CTA's tokens; block reduction; one thread per token computes
// r = rsqrt(mean(x^2) + norm_eps), mixes = dot * r, and the split + Sinkhorn.
// Phase 2 (side step only): y and h for every token (x re-read through L1/L2),
// sum of squares of the rounded h, then h_norm.
constexpr int kTokThreads = 256;
// threads per CTA of k_tokens_simple: the a4-a6 flavour at eight streams takes
// 128 (one token per CTA; d = 5120 is 640 chunks of 8 channels, 5 per thread
// rather than 2 or 3), the rest 256
template <int HC, bool kCoefIn>
__host__ __device__ constexpr int tok_threads() { return (kCoefIn && HC == 8) ? 128 : kTokThreads; }
// from this many tokens on, a1-a3 run on token tiles (k_mixes_tiled): below it the
// 32-token tiles would leave most SMs idle
constexpr int64_t kTiledMinTokens = 128;

// tokens per CTA: the accumulators are (2 + HC) * HC per token
template <int HC>
__host__ __device__ constexpr int tok_per_cta() { return HC <= 4 ? 4 : 1; }

// The a4-a6 flavour (kCoefIn) keeps its registers low enough for four CTAs of
// 128 threads per SM at eight streams (one CTA of 256 per SM left too few warps
// in flight), four of 256 at two streams.
template <bool kFull, int HC, bool kCoefIn = false>
__global__ void __launch_bounds__(tok_threads<HC, kCoefIn>(), kCoefIn ? (HC == 8 ? 4 : HC <= 2 ? 4 : 2) : 1)
k_tokens_simple(const uint16_t *__restrict__ x, const float *__restrict__ pre_mix,
                const uint16_t *__restrict__ f, const float *__restrict__ hc_fn,
                const float *__restrict__ hc_scale, const float *__restrict__ hc_base,
                const float *__restrict__ norm_w, int64_t n, int d, int iters, float eps,
                float norm_eps, uint16_t *__restrict__ h_norm, uint16_t *__restrict__ y,
                float *__restrict__ pre_out, float *__restrict__ post_out,
                float *__restrict__ comb_out, float *__restrict__ mixes_out) {
    constexpr int kTok = tok_per_cta<HC>();
    constexpr int NT = tok_threads<HC, kCoefIn>();
    constexpr int MIX = (2 + HC) * HC;
    constexpr int kVals = MIX * kTok + kTok;  // MIX dots per token + sum of squares per token
    extern __shared__ uint4 hbuf[];            // kTok * d/8 chunks (side step only)
    __shared__ float red[NT / 32][kVals];
    __shared__ float tot[kVals];
    __shared__ float coef[kTok][HC + HC * HC];
    __shared__ float ssh[NT / 32][kTok];

    const int64_t t0 = (int64_t)blockIdx.x * kTok;
    const int ntok = (n - t0 < kTok) ? (int)(n - t0) : kTok;
    const int K = HC * d, K8 = K >> 3;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if constexpr (kCoefIn) {
        // post and comb of each token, parked by k_mixes_tiled at the start of the
        // token's own y row (read here before this CTA writes that row)
        constexpr int C = HC + HC * HC;
        for (int q = threadIdx.x; q < ntok * C; q += NT)  // one load per thread
            coef[q / C][q % C] = reinterpret_cast<const float *>(y + (t0 + q / C) * K)[q % C];
    } else {

    float acc[MIX][kTok];
    float ss[kTok];
#pragma unroll
    for (int i = 0; i < MIX; ++i)
#pragma unroll
        for (int u = 0; u < kTok; ++u) acc[i][u] = 0.0f;
#pragma unroll
    for (int u = 0; u < kTok; ++u) ss[u] = 0.0f;

    for (int ch = threadIdx.x; ch < K8; ch += NT) {
        float xv[kTok][8];
#pragma unroll
        for (int u = 0; u < kTok; ++u) {
            if (u < ntok) {
                unpack8(__ldg(reinterpret_cast<const uint4 *>(x + (t0 + u) * K) + ch), xv[u]);
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) xv[u][e] = 0.0f;
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) ss[u] = fmaf(xv[u][e], xv[u][e], ss[u]);
        }
#pragma unroll
        for (int i = 0; i < MIX; ++i) {
            const float4 *wp = reinterpret_cast<const float4 *>(hc_fn + (int64_t)i * K) + 2 * ch;
            const float4 wa = __ldg(wp), wb = __ldg(wp + 1);
            const float w[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int u = 0; u < kTok; ++u)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[i][u] = fmaf(xv[u][e], w[e], acc[i][u]);
        }
    }
    // block reduction of the 24*kTok dots and kTok sums of squares
#pragma unroll
    for (int i = 0; i < MIX; ++i)
#pragma unroll
        for (int u = 0; u < kTok; ++u) {
            const float v = warp_sum(acc[i][u]);
            if (lane == 0) red[warp][i * kTok + u] = v;
        }
#pragma unroll
    for (int u = 0; u < kTok; ++u) {
        const float v = warp_sum(ss[u]);
        if (lane == 0) red[warp][MIX * kTok + u] = v;
    }
    __syncthreads();
    for (int v = threadIdx.x; v < kVals; v += NT) {
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) s += red[w][v];
        tot[v] = s;
    }
    __syncthreads();
    if (threadIdx.x < ntok) {
        const int u = threadIdx.x;
        const int64_t t = t0 + u;
        const float r = rsqrtf(tot[MIX * kTok + u] / (float)K + norm_eps);
        float m[MIX];
#pragma unroll
        for (int i = 0; i < MIX; ++i) m[i] = tot[i * kTok + u] * r;
        float pr[HC], po[HC], c[HC * HC];
        split_sinkhorn_token_hc<HC>(m, __ldg(hc_scale), __ldg(hc_scale + 1), __ldg(hc_scale + 2),
                                    hc_base, iters, eps, pr, po, c);
#pragma unroll
        for (int k = 0; k < HC; ++k) {
            if (pre_out) pre_out[t * HC + k] = pr[k];
            if (post_out) post_out[t * HC + k] = po[k];
        }
        if (comb_out) {
#pragma unroll
            for (int i = 0; i < HC * HC; ++i) comb_out[t * HC * HC + i] = c[i];
        }
        if (mixes_out) {
#pragma unroll
            for (int i = 0; i < MIX; ++i) mixes_out[t * MIX + i] = m[i];
        }
#pragma unroll
        for (int k = 0; k < HC; ++k) coef[u][k] = po[k];
#pragma unroll
        for (int i = 0; i < HC * HC; ++i) coef[u][HC + i] = c[i];
    }
    }  // kCoefIn
    if constexpr (!kFull) return;
    __syncthreads();

    // phase 2: y, h (kept in shared memory as bf16), sum of squares of h
    const int d8 = d >> 3;
    float hs[kTok];
#pragma unroll
    for (int u = 0; u < kTok; ++u) hs[u] = 0.0f;
#pragma unroll
    for (int u = 0; u < kTok; ++u) {
        if (u >= ntok) break;
        const int64_t t = t0 + u;
        // packed fp32 pairs (adjacent columns), each lane rounded as the scalar
        // instruction would be
        f32x2 pm2[HC];
#pragma unroll
        for (int s = 0; s < HC; ++s) pm2[s] = f2_dup(__ldg(pre_mix + t * HC + s));
        const uint4 *xs = reinterpret_cast<const uint4 *>(x + t * K);
        const uint4 *fs = reinterpret_cast<const uint4 *>(f + t * d);
        uint4 *ys = reinterpret_cast<uint4 *>(y + t * K);
        f32x2 hs2 = f2_dup(0.0f);
        for (int c = threadIdx.x; c < d8; c += NT) {
            f32x2 fv[4], xv[HC][4];
            {
                const uint4 fr = __ldg(fs + c);
                fv[0] = f2_from_bf16x2(fr.x); fv[1] = f2_from_bf16x2(fr.y);
                fv[2] = f2_from_bf16x2(fr.z); fv[3] = f2_from_bf16x2(fr.w);
            }
#pragma unroll
            for (int j = 0; j < HC; ++j) {
                const uint4 xr = __ldg(xs + j * d8 + c);
                xv[j][0] = f2_from_bf16x2(xr.x); xv[j][1] = f2_from_bf16x2(xr.y);
                xv[j][2] = f2_from_bf16x2(xr.z); xv[j][3] = f2_from_bf16x2(xr.w);
            }
#pragma unroll
            for (int k = 0; k < HC; ++k) {
                const f32x2 ck = f2_dup(coef[u][k]);
                f32x2 o[4];
#pragma unroll
                for (int p = 0; p < 4; ++p) o[p] = f2_mul(ck, fv[p]);
#pragma unroll
                for (int j = 0; j < HC; ++j) {
                    const f32x2 cjk = f2_dup(coef[u][HC + j * HC + k]);
#pragma unroll
                    for (int p = 0; p < 4; ++p) o[p] = f2_fma(cjk, xv[j][p], o[p]);
                }
                ys[k * d8 + c] = make_uint4(f2_to_bf16x2(o[0]), f2_to_bf16x2(o[1]), f2_to_bf16x2(o[2]),
                                            f2_to_bf16x2(o[3]));
            }
            f32x2 h[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                h[p] = f2_mul(pm2[0], xv[0][p]);
#pragma unroll
                for (int s2 = 1; s2 < HC; ++s2) h[p] = f2_fma(pm2[s2], xv[s2][p], h[p]);
            }
            const uint4 hb = make_uint4(f2_to_bf16x2(h[0]), f2_to_bf16x2(h[1]), f2_to_bf16x2(h[2]),
                                        f2_to_bf16x2(h[3]));
            hbuf[u * d8 + c] = hb;
            const uint32_t hw[4] = {hb.x, hb.y, hb.z, hb.w};
#pragma unroll
            for (int p = 0; p < 4; ++p) {
                const f32x2 r = f2_from_bf16x2(hw[p]);
                hs2 = f2_fma(r, r, hs2);
            }
        }
        hs[u] = f2_hsum(hs2);
    }
#pragma unroll
    for (int u = 0; u < kTok; ++u) {
        const float v = warp_sum(hs[u]);
        if (lane == 0) ssh[warp][u] = v;
    }
    __syncthreads();
    const float4 *w4 = reinterpret_cast<const float4 *>(norm_w);
    for (int u = 0; u < ntok; ++u) {
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < NT / 32; ++w) s += ssh[w][u];
        const float rs = rsqrtf(s / (float)d + norm_eps);
        uint4 *o = reinterpret_cast<uint4 *>(h_norm + (t0 + u) * d);
        for (int c = threadIdx.x; c < d8; c += NT) {
            float h[8];
            unpack8(hbuf[u * d8 + c], h);
            const float4 wa = __ldg(w4 + 2 * c), wb = __ldg(w4 + 2 * c + 1);
            const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) h[i] = (h[i] * rs) * wv[i];
            o[c] = pack8(h);
        }
    }
}

// ------------------------------------------------------------------ a1-a3, token tiles on the tensor cores
// m_i = r * sum_k x_k W_ik for 32 tokens per CTA (Block page, Block.hc_mixes),
// then the split + Sinkhorn ("Stream combination" page) per token.  Each stage
// stages COLS columns of x (the tile's tokens, bf16) and of W (all MIX rows,
// fp32) through a two-deep cp.async ring.  The warps form RG row groups x CG
// column groups: warp (rg, cg) takes rows rg*MIX/RG .. of W and 32 columns of
// every stage, in k-steps of 8 on mma.sync m16n8k8 tf32 (x is exact in tf32;
// W is split into tf32 hi + lo, two MMAs).  The tensor core's fp32
// accumulation is not rounded to nearest, and over the thousands of k-steps of
// a row of hc*d columns its error grows past the 1e-5 budget; so each stage's
// products go to a fresh accumulator (8 MMAs) that is then added to the
// running total with an ordinary fp32 add.  The sum of squares of x comes from
// the same A fragments (row group 0: every element once).  The column groups'
// totals are added in order through shared memory; then one thread per token
// finishes.  Columns past K and tokens past n are zero-filled.
constexpr int kMxTok = 32;
constexpr int kMxThreads = 256;

template <int HC>
struct Mx {
    static constexpr int MIX = (2 + HC) * HC;  // 8, 24, 80: whole 8-row n-tiles
    static constexpr int NT = MIX / 8;
    static constexpr int RG = HC == 8 ? 2 : 1;  // row groups of warps
    static constexpr int CG = 8 / RG;           // column groups of warps
    static constexpr int NTW = NT / RG;         // n-tiles per warp
    static constexpr int COLS = 32 * CG;        // columns per stage (32 per warp)
    static constexpr int KS = 4;                // k-steps of 8 per warp per stage
    static constexpr int XROW = COLS + 8;       // bf16 per staged row of x (bank spread)
    static constexpr int WROW = COLS + 4;       // floats per staged row of W
    struct Stage {
        uint16_t x[kMxTok][XROW];
        float w[MIX][WROW];
    };
    static constexpr size_t SMEM = 2 * sizeof(Stage);
    static_assert(MIX % 8 == 0 && NT % RG == 0, "whole n-tiles per row group");
    static_assert(sizeof(Stage) % 16 == 0 && (XROW * 2) % 16 == 0 && (WROW * 4) % 16 == 0, "16-byte rows");
    static_assert(SMEM >= sizeof(float) * CG * kMxTok * (MIX + 1), "the partial sums reuse the ring");
};

template <int HC>
__global__ void __launch_bounds__(kMxThreads, 2)
k_mixes_tiled(const uint16_t *__restrict__ x, const float *__restrict__ hc_fn,
              const float *__restrict__ hc_scale, const float *__restrict__ hc_base, int64_t n, int d,
              int iters, float eps, float norm_eps, float *__restrict__ pre_out,
              float *__restrict__ post_out, float *__restrict__ comb_out, float *__restrict__ mixes_out,
              uint16_t *__restrict__ coef_rows) {
    using M = Mx<HC>;
    constexpr int MIX = M::MIX, NTW = M::NTW, COLS = M::COLS, CG = M::CG;
    extern __shared__ uint4 smem_u4[];
    typename M::Stage *stg = reinterpret_cast<typename M::Stage *>(smem_u4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int rg = warp / CG, cg = warp % CG;
    const int r0 = rg * NTW * 8;  // this warp's first row of W
    const int64_t t0 = (int64_t)blockIdx.x * kMxTok;
    const int K = HC * d;
    const int nst = (K + COLS - 1) / COLS;
    auto issue = [&](int st) {
        if (st < nst) {
            typename M::Stage &S = stg[st & 1];
            const int c0 = st * COLS;
            for (int k = threadIdx.x; k < kMxTok * (COLS / 8); k += kMxThreads) {
                const int tt = k / (COLS / 8), kc = k % (COLS / 8);
                const bool ok = t0 + tt < n && c0 + kc * 8 < K;
                cp_async16(&S.x[tt][kc * 8], ok ? x + (t0 + tt) * K + c0 + kc * 8 : x, ok ? 16 : 0);
            }
            for (int k = threadIdx.x; k < MIX * (COLS / 4); k += kMxThreads) {
                const int i = k / (COLS / 4), kc = k % (COLS / 4);
                const bool ok = c0 + kc * 4 < K;
                cp_async16(&S.w[i][4 * kc], ok ? hc_fn + (int64_t)i * K + c0 + 4 * kc : hc_fn, ok ? 16 : 0);
            }
        }
        cp_async_commit();  // an empty group past the end keeps the count uniform
    };
    float tot[2][NTW][4];  // tokens 16mt + g (+8), rows r0 + 8nt + 2q (+1)
    float ss[2][2];        // sum of squares of tokens 16mt + g, 16mt + g + 8 (this lane's columns)
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
        ss[mt][0] = ss[mt][1] = 0.0f;
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) tot[mt][nt][e] = 0.0f;
    }
    issue(0);
    for (int st = 0; st < nst; ++st) {
        cp_async_wait<0>();
        __syncthreads();  // stage st landed for every thread; the other slot is free
        issue(st + 1);
        const typename M::Stage &S = stg[st & 1];
        float acc[2][NTW][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.0f;
#pragma unroll
        for (int ks = 0; ks < M::KS; ++ks) {
            const int k0 = 32 * cg + 8 * ks;
            uint32_t a[2][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt) {
                a[mt][0] = (uint32_t)S.x[16 * mt + g][k0 + q] << 16;
                a[mt][1] = (uint32_t)S.x[16 * mt + g + 8][k0 + q] << 16;
                a[mt][2] = (uint32_t)S.x[16 * mt + g][k0 + q + 4] << 16;
                a[mt][3] = (uint32_t)S.x[16 * mt + g + 8][k0 + q + 4] << 16;
                if (rg == 0) {
                    const float v0 = __uint_as_float(a[mt][0]), v1 = __uint_as_float(a[mt][1]);
                    const float v2 = __uint_as_float(a[mt][2]), v3 = __uint_as_float(a[mt][3]);
                    ss[mt][0] = fmaf(v2, v2, fmaf(v0, v0, ss[mt][0]));
                    ss[mt][1] = fmaf(v3, v3, fmaf(v1, v1, ss[mt][1]));
                }
            }
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt) {
                uint32_t bh0, bl0, bh1, bl1;
                tf32_split(S.w[r0 + 8 * nt + g][k0 + q], bh0, bl0);
                tf32_split(S.w[r0 + 8 * nt + g][k0 + q + 4], bh1, bl1);
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    mma_tf32(acc[mt][nt], a[mt], bl0, bl1);
                    mma_tf32(acc[mt][nt], a[mt], bh0, bh1);
                }
            }
        }
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) tot[mt][nt][e] += acc[mt][nt][e];
    }
    cp_async_wait<0>();
    __syncthreads();  // every warp is done with the ring: reuse it for the partial sums
    float *red = reinterpret_cast<float *>(smem_u4);  // [column group][token][MIX + 1]
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
#pragma unroll
        for (int nt = 0; nt < NTW; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int tt = 16 * mt + g + 8 * (e >> 1), i = r0 + 8 * nt + 2 * q + (e & 1);
                red[(cg * kMxTok + tt) * (MIX + 1) + i] = tot[mt][nt][e];
            }
        if (rg == 0) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                float v = ss[mt][h];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                if (q == 0) red[(cg * kMxTok + 16 * mt + g + 8 * h) * (MIX + 1) + MIX] = v;
            }
        }
    }
    __syncthreads();
    if (threadIdx.x < kMxTok && t0 + threadIdx.x < n) {
        const int tt = threadIdx.x;
        const int64_t t = t0 + tt;
        float m[MIX];
        float s2 = 0.0f;
#pragma unroll
        for (int w = 0; w < CG; ++w) s2 += red[(w * kMxTok + tt) * (MIX + 1) + MIX];
        const float r = rsqrtf(s2 / (float)K + norm_eps);
#pragma unroll
        for (int i = 0; i < MIX; ++i) {
            float v = 0.0f;
#pragma unroll
            for (int w = 0; w < CG; ++w) v += red[(w * kMxTok + tt) * (MIX + 1) + i];
            m[i] = v * r;
        }
        float pr[HC], po[HC], c[HC * HC];
        split_sinkhorn_token_hc<HC>(m, __ldg(hc_scale), __ldg(hc_scale + 1), __ldg(hc_scale + 2), hc_base,
                                    iters, eps, pr, po, c);
#pragma unroll
        for (int k = 0; k < HC; ++k) {
            if (pre_out) pre_out[t * HC + k] = pr[k];
            if (post_out) post_out[t * HC + k] = po[k];
        }
        if (comb_out) {
#pragma unroll
            for (int i = 0; i < HC * HC; ++i) comb_out[t * HC * HC + i] = c[i];
        }
        if (mixes_out) {
#pragma unroll
            for (int i = 0; i < MIX; ++i) mixes_out[t * MIX + i] = m[i];
        }
        if (coef_rows) {  // post and comb for the a4-a6 pass, at the start of the token's y row
            float *dst = reinterpret_cast<float *>(coef_rows + t * K);
#pragma unroll
            for (int k = 0; k < HC; ++k) dst[k] = po[k];
#pragma unroll
            for (int i = 0; i < HC * HC; ++i) dst[HC + i] = c[i];
        }
    }
}

template <int HC>
cudaError_t launch_mixes_tiled_hc(const uint16_t *x, const float *hc_fn, const float *hc_scale,
                                  const float *hc_base, int64_t n, int d, int iters, float eps,
                                  float norm_eps, float *pre_out, float *post_out, float *comb_out,
                                  float *mixes_out, uint16_t *coef_rows, cudaStream_t s) {
    const int smem = (int)Mx<HC>::SMEM;
    cudaError_t e = cudaFuncSetAttribute(k_mixes_tiled<HC>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t blocks = (n + kMxTok - 1) / kMxTok;
    k_mixes_tiled<HC><<<(unsigned)blocks, kMxThreads, smem, s>>>(x, hc_fn, hc_scale, hc_base, n, d, iters, eps,
                                                                 norm_eps, pre_out, post_out, comb_out, mixes_out,
                                                                 coef_rows);
    return cudaGetLastError();
}


template <int HC>
cudaError_t launch_tokens_simple_hc(const uint16_t *x, const float *pre_mix, const uint16_t *f,
                                    const float *hc_fn, const float *hc_scale, const float *hc_base,
                                    const float *norm_w, int64_t n, int d, int iters, float eps,
                                    float norm_eps, uint16_t *h_norm, uint16_t *y, float *pre_out,
                                    float *post_out, float *comb_out, float *mixes_out,
                                    cudaStream_t s) {
    constexpr int kTok = tok_per_cta<HC>();
    const int64_t blocks = (n + kTok - 1) / kTok;
    cudaError_t e;
    if (n >= kTiledMinTokens) {
        // a1-a3 on token tiles, then a4-a6 per token from the coefficients parked in
        // the y rows.  For the side step, the tcgen05 kernel when its split weights
        // fit the h_norm output (written only by the a4-a6 pass, after it); else
        // the mma.sync kernel (hc_fn read once per 32 tokens).
        if (f && (size_t)n * (size_t)d * 2 >= proj_umma_wsplit_bytes(HC, (int64_t)HC * d))
            e = launch_mixes_umma(x, hc_fn, hc_scale, hc_base, n, HC, d, iters, eps, norm_eps, h_norm, pre_out,
                                  post_out, comb_out, mixes_out, y, s);
        else
            e = launch_mixes_tiled_hc<HC>(x, hc_fn, hc_scale, hc_base, n, d, iters, eps, norm_eps, pre_out,
                                          post_out, comb_out, mixes_out, f ? y : nullptr, s);
        if (e != cudaSuccess || !f) return e;
        const size_t smem = (size_t)kTok * d * 2;
        e = cudaFuncSetAttribute(k_tokens_simple<true, HC, true>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        k_tokens_simple<true, HC, true><<<(unsigned)blocks, tok_threads<HC, true>(), smem, s>>>(
            x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, n, d, iters, eps, norm_eps, h_norm, y,
            nullptr, nullptr, nullptr, nullptr);
        return cudaGetLastError();
    }
    if (f) {
        const size_t smem = (size_t)kTok * d * 2;
        e = cudaFuncSetAttribute(k_tokens_simple<true, HC>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        k_tokens_simple<true, HC><<<(unsigned)blocks, kTokThreads, smem, s>>>(
            x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, n, d, iters, eps, norm_eps, h_norm, y,
            pre_out, post_out, comb_out, mixes_out);
    } else {
        k_tokens_simple<false, HC><<<(unsigned)blocks, kTokThreads, 0, s>>>(
            x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, n, d, iters, eps, norm_eps, h_norm, y,
            pre_out, post_out, comb_out, mixes_out);
    }
    return cudaGetLastError();
}

cudaError_t launch_tokens_simple(const uint16_t *x, const float *pre_mix, const uint16_t *f,
                                 const float *hc_fn, const float *hc_scale, const float *hc_base,
                                 const float *norm_w, int64_t n, int hc, int d, int iters, float eps,
                                 float norm_eps, uint16_t *h_norm, uint16_t *y, float *pre_out,
                                 float *post_out, float *comb_out, float *mixes_out,
                                 cudaStream_t s) {
#define HC_TOKENS(H) launch_tokens_simple_hc<H>(x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, n, d, \
                                                 iters, eps, norm_eps, h_norm, y, pre_out, post_out,   \
                                                 comb_out, mixes_out, s)
    switch (hc) {
        case 2: return HC_TOKENS(2);
        case 4: return HC_TOKENS(4);
        case 8: return HC_TOKENS(8);
        default: return cudaErrorInvalidValue;
    }
#undef HC_TOKENS
}

}  // namespace hc
