// hc_backward_generic.cu -- the backward of one hyper-connection side step
// (a1-a6) for two and eight streams.
//
// The same derivative as hc_backward.cu (DeepSeek-V4.1 Block page, Code
// section: Block.hc_mixes, Block.hc_pre, attn_norm / ffn_norm,
// Block.hc_post; "Stream combination" page: hc_split_sinkhorn, whose kernel
// takes the stream count hc as a parameter): the bf16 casts pass gradients
// through unchanged, the forward's rounded h is used where the forward used
// it, and Sinkhorn is differentiated step by step through its iterates.
//
// These kernels favour plainness over speed; the four-stream model runs the
// tensor-core kernels of hc_backward.cu.  The projection a = x W^T runs on the
// fifth-generation tensor cores (launch_proj_umma, hc_proj_umma.cu); then one
// CTA per token:
//   kg_token  the token's sums in one pass, the split, Sinkhorn forward with
//             its iterates and backward (one thread), g_pre_mix and the
//             per-token record;
//   kg_gx     g_x and g_f;
// then partial sums of the parameter gradients over blocks of 1,024 tokens,
// added block by block in a fixed order (deterministic, no atomics).
#include <cuda.h>

#include "hc_backward_generic.h"
#include "hc_launch.h"
#include "hc_device.cuh"
#include "hc_ptx.cuh"

namespace hc {
namespace bwg {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTokBlock = 1024;  // tokens per partial sum of a parameter gradient
constexpr int kFnTile = 16;      // tokens per staged tile in kg_fn_tc

// The per-token record in the workspace (floats).
template <int HC>
struct Lay {
    static constexpr int kMix = (2 + HC) * HC;
    static constexpr int kA = 0;                // a[mix]: the projection
    static constexpr int kGa = kMix;            // g_a[mix]: the gradient of a
    static constexpr int kGz = 2 * kMix;        // g_z[mix]: the g_hc_base terms
    static constexpr int kGzm = 3 * kMix;       // gzm[3]: the g_hc_scale terms
    static constexpr int kPost = 3 * kMix + 4;  // post[HC]
    static constexpr int kComb = kPost + HC;    // comb[HC * HC]
    static constexpr int kPm = kComb + HC * HC; // pre_mix[HC]
    static constexpr int kRs = kPm + HC;        // 1 / RMS(h)
    static constexpr int kCr = kRs + 1;         // the statistic's coefficient of x in g_x
    static constexpr int kK3 = kRs + 2;         // rs^3 / d * sum(h w g_hn)
    // g_a as three bf16 parts hi, mid, lo (part-major, 3 * mix bf16) for the
    // tensor cores of kg_fn_tc; 16-byte aligned
    static constexpr int kGaP = (kK3 + 1 + 3) / 4 * 4;
    static constexpr int kWs = kGaP + (3 * kMix / 2 + 3) / 4 * 4;
    static constexpr int kSmall = (kMix + 3 + 3) / 4 * 4;  // per-run partials of g_hc_base, g_hc_scale
    // token sums of kg_token: sum h^2, T = sum h w g_hn, sum x^2, g_post[HC],
    // g_comb[HC*HC], A[HC] = sum x_s w g_hn, B[HC] = sum x_s h
    static constexpr int kSH2 = 0, kST = 1, kSX2 = 2, kSPost = 3, kSComb = 3 + HC,
                         kSA = 3 + HC + HC * HC, kSB = kSA + HC, kSums = kSB + HC;
};

__device__ __forceinline__ float sigm(float z) { return 1.0f / (1.0f + expf(-z)); }

__device__ __forceinline__ void ld4bf(const uint16_t *p, float (&o)[4]) {
    const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
    o[0] = bf16lo(v.x);
    o[1] = __uint_as_float(v.x & 0xffff0000u);
    o[2] = bf16lo(v.y);
    o[3] = __uint_as_float(v.y & 0xffff0000u);
}
__device__ __forceinline__ void ld4f(const float *p, float (&o)[4]) {
    const float4 v = __ldg(reinterpret_cast<const float4 *>(p));
    o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
}
__device__ __forceinline__ float round_bf16(float v) { return bf16lo(pack_bf16x2(v, 0.0f)); }

// One warp per token (no CTA barrier): one pass over the token for its sums
// (every lane ends with the totals), then the split and Sinkhorn forward and
// backward with the comb matrix spread over the lanes (element e = lane +
// 32 r, r < max(1, HC*HC / 32); at HC*HC < 32 the lanes repeat it), the
// gradients of the mix numbers (mix row i = lane + 32 r), g_pre_mix and the
// record.  Row sums reduce over lanes ^1 .. ^HC/2, column sums over lanes
// ^HC .. ^16 and, at HC = 8, over the two elements a lane holds.  Dynamic
// shared memory per warp: the row softmax S, the iterates P_0 ..
// P_{2 iters - 1} (the backward recomputes each step's 1 / (sum + eps) from
// them, with the same sums the forward took), then the token's sums.
template <int HC>
__device__ __forceinline__ float row_sum(float v) {
#pragma unroll
    for (int m = 1; m < HC; m <<= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}
template <int HC>
__device__ __forceinline__ float row_max(float v) {
#pragma unroll
    for (int m = 1; m < HC; m <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}
template <int HC>
__device__ __forceinline__ float col_sum_lanes(float v) {
#pragma unroll
    for (int m = HC; m < 32 && m < HC * HC; m <<= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

template <int HC>
__global__ void __launch_bounds__(128, HC >= 8 ? 3 : 1)
kg_token(const uint16_t *__restrict__ x, const float *__restrict__ pre_mix,
         const uint16_t *__restrict__ f, const float *__restrict__ hc_scale,
         const float *__restrict__ hc_base, const float *__restrict__ norm_w, int64_t n, int d, int iters,
         float eps, float norm_eps, const float *__restrict__ g_hn, const float *__restrict__ g_y,
         const float *__restrict__ g_pre, float *__restrict__ g_pm, float *__restrict__ ws) {
    using L = Lay<HC>;
    constexpr int M = L::kMix, H2 = HC * HC;
    constexpr int EPL = H2 > 32 ? H2 / 32 : 1;  // comb elements per lane
    constexpr int MPL = (M + 31) / 32;          // mix rows per lane
    extern __shared__ float sdyn[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp;
    if (t >= n) return;  // warp-uniform
    const int K = HC * d;
    const uint16_t *xt = x + t * K;
    float *wt = ws + t * L::kWs;
    float *sS = sdyn + (size_t)warp * ((2 * iters + 1) * H2 + L::kSums);
    float *sP = sS + H2;
    float *sT = sP + 2 * iters * H2;
    float pm[HC];
#pragma unroll
    for (int s = 0; s < HC; ++s) pm[s] = __ldg(pre_mix + t * HC + s);
    float v[L::kSums];
#pragma unroll
    for (int i = 0; i < L::kSums; ++i) v[i] = 0.0f;
    if constexpr (HC >= 8) {
        // lane l: columns 4c .. 4c + 3 for c = l, l + 32, ..., taken as two halves of
        // two columns in column order (fewer loaded values live at a time: the
        // same sums in the same order)
        for (int c = lane; c < d / 4; c += 32) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const int c2 = 4 * c + 2 * hf;
                float xv[HC][2], fv[2], gh[2], w[2], h[2];
#pragma unroll
                for (int s = 0; s < HC; ++s) {
                    const uint32_t xb = __ldg(reinterpret_cast<const uint32_t *>(xt + (int64_t)s * d + c2));
                    xv[s][0] = bf16lo(xb);
                    xv[s][1] = __uint_as_float(xb & 0xffff0000u);
                }
                {
                    const uint32_t fb = __ldg(reinterpret_cast<const uint32_t *>(f + t * d + c2));
                    fv[0] = bf16lo(fb);
                    fv[1] = __uint_as_float(fb & 0xffff0000u);
                    const float2 g2 = __ldg(reinterpret_cast<const float2 *>(g_hn + t * d + c2));
                    const float2 w2 = __ldg(reinterpret_cast<const float2 *>(norm_w + c2));
                    gh[0] = g2.x; gh[1] = g2.y; w[0] = w2.x; w[1] = w2.y;
                }
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float hv = pm[0] * xv[0][e];
#pragma unroll
                    for (int s = 1; s < HC; ++s) hv = fmaf(pm[s], xv[s][e], hv);
                    h[e] = round_bf16(hv);  // the forward's bf16 h
                    const float wg = w[e] * gh[e];
                    v[L::kSH2] = fmaf(h[e], h[e], v[L::kSH2]);
                    v[L::kST] = fmaf(h[e], wg, v[L::kST]);
#pragma unroll
                    for (int j = 0; j < HC; ++j) {
                        v[L::kSX2] = fmaf(xv[j][e], xv[j][e], v[L::kSX2]);
                        v[L::kSA + j] = fmaf(xv[j][e], wg, v[L::kSA + j]);
                        v[L::kSB + j] = fmaf(xv[j][e], h[e], v[L::kSB + j]);
                    }
                }
#pragma unroll
                for (int k = 0; k < HC; ++k) {
                    const float2 g2 = __ldg(reinterpret_cast<const float2 *>(g_y + (t * HC + k) * d + c2));
                    const float gy[2] = {g2.x, g2.y};
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        v[L::kSPost + k] = fmaf(fv[e], gy[e], v[L::kSPost + k]);
#pragma unroll
                        for (int j = 0; j < HC; ++j)
                            v[L::kSComb + j * HC + k] = fmaf(xv[j][e], gy[e], v[L::kSComb + j * HC + k]);
                    }
                }
            }
        }
    } else {
        for (int c = lane; c < d / 4; c += 32) {
            float xv[HC][4], fv[4], gh[4], w[4], h[4];
    #pragma unroll
            for (int s = 0; s < HC; ++s) ld4bf(xt + (int64_t)s * d + 4 * c, xv[s]);
            ld4bf(f + t * d + 4 * c, fv);
            ld4f(g_hn + t * d + 4 * c, gh);
            ld4f(norm_w + 4 * c, w);
    #pragma unroll
            for (int e = 0; e < 4; ++e) {
                float hv = pm[0] * xv[0][e];
    #pragma unroll
                for (int s = 1; s < HC; ++s) hv = fmaf(pm[s], xv[s][e], hv);
                h[e] = round_bf16(hv);  // the forward's bf16 h
                const float wg = w[e] * gh[e];
                v[L::kSH2] = fmaf(h[e], h[e], v[L::kSH2]);
                v[L::kST] = fmaf(h[e], wg, v[L::kST]);
    #pragma unroll
                for (int j = 0; j < HC; ++j) {
                    v[L::kSX2] = fmaf(xv[j][e], xv[j][e], v[L::kSX2]);
                    v[L::kSA + j] = fmaf(xv[j][e], wg, v[L::kSA + j]);
                    v[L::kSB + j] = fmaf(xv[j][e], h[e], v[L::kSB + j]);
                }
            }
    #pragma unroll
            for (int k = 0; k < HC; ++k) {
                float gy[4];
                ld4f(g_y + (t * HC + k) * d + 4 * c, gy);
    #pragma unroll
                for (int e = 0; e < 4; ++e) {
                    v[L::kSPost + k] = fmaf(fv[e], gy[e], v[L::kSPost + k]);
    #pragma unroll
                    for (int j = 0; j < HC; ++j)
                        v[L::kSComb + j * HC + k] = fmaf(xv[j][e], gy[e], v[L::kSComb + j * HC + k]);
                }
            }
        }
    }
#pragma unroll
    for (int i = 0; i < L::kSums; ++i) {
        const float tv = warp_sum(v[i]);
        if (lane == 0) sT[i] = tv;
    }
    __syncwarp();

    const float r = rsqrtf(sT[L::kSX2] / (float)K + norm_eps);
    const float rs = rsqrtf(sT[L::kSH2] / (float)d + norm_eps);
    const float k3 = rs * rs * rs / (float)d * sT[L::kST];
    const float s0 = __ldg(hc_scale), s1 = __ldg(hc_scale + 1), s2 = __ldg(hc_scale + 2);

    // the row softmax S of the comb logits and P_0 = S + eps
    float S[EPL], P[EPL];
    int el[EPL];
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
        el[q] = (lane + 32 * q) % H2;
        const float lg = fmaf(wt[L::kA + 2 * HC + el[q]] * r, s2, __ldg(hc_base + 2 * HC + el[q]));
        const float ex = expf(lg - row_max<HC>(lg));
        S[q] = ex / row_sum<HC>(ex);
        P[q] = S[q] + eps;
        if (lane + 32 * q < H2) {
            sS[el[q]] = S[q];
            sP[el[q]] = P[q];
        }
    }
    auto axis_sum = [&](const float (&a)[EPL], int st, float (&o)[EPL]) {
        if (st & 1) {  // a column step: over the rows
            float cs = 0.0f;
#pragma unroll
            for (int q = 0; q < EPL; ++q) cs += col_sum_lanes<HC>(a[q]);
#pragma unroll
            for (int q = 0; q < EPL; ++q) o[q] = cs;
        } else {
#pragma unroll
            for (int q = 0; q < EPL; ++q) o[q] = row_sum<HC>(a[q]);
        }
    };
    // steps 1 .. 2*iters-1: a column step for odd, a row step for even steps
    for (int st = 1; st < 2 * iters; ++st) {
        float sm[EPL];
        axis_sum(P, st, sm);
#pragma unroll
        for (int q = 0; q < EPL; ++q) {
            P[q] *= 1.0f / (sm[q] + eps);
            if (lane + 32 * q < H2) sP[st * H2 + el[q]] = P[q];
        }
    }
#pragma unroll
    for (int q = 0; q < EPL; ++q)
        if (lane + 32 * q < H2) wt[L::kComb + el[q]] = P[q];
    // back through the steps: g, the gradient of the current iterate
    float g[EPL];
#pragma unroll
    for (int q = 0; q < EPL; ++q) g[q] = sT[L::kSComb + el[q]];
    __syncwarp();
    for (int st = 2 * iters - 1; st >= 1; --st) {
        float pa[EPL], pb[EPL], gp[EPL], sm[EPL], dot[EPL];
#pragma unroll
        for (int q = 0; q < EPL; ++q) {
            pa[q] = sP[(st - 1) * H2 + el[q]];
            pb[q] = sP[st * H2 + el[q]];
            gp[q] = g[q] * pb[q];
        }
        axis_sum(pa, st, sm);
        axis_sum(gp, st, dot);
#pragma unroll
        for (int q = 0; q < EPL; ++q) g[q] = (g[q] - dot[q]) * (1.0f / (sm[q] + eps));
    }
    // through the row softmax
    float gzc[EPL];
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
        const float dt = row_sum<HC>(g[q] * S[q]);
        gzc[q] = S[q] * (g[q] - dt);
    }

    // pre and post (sigmoids), then the gradient of the projection; mix row
    // i = lane + 32 u (pre 0 .. HC-1, post HC .. 2HC-1, comb the rest)
    float z0 = 0.0f, z1 = 0.0f, z2 = 0.0f, gr = 0.0f;
    uint16_t *gpart = reinterpret_cast<uint16_t *>(wt + L::kGaP);
#pragma unroll
    for (int u = 0; u < MPL; ++u) {
        const int i = lane + 32 * u;
        const int ic = i < M ? i : 0;
        const float a = wt[L::kA + ic];
        const float m = a * r;
        // the comb gradient of element i - 2HC sits in lane (i - 2HC) % 32, slot (i - 2HC) / 32
        const int ec = (ic >= 2 * HC ? ic - 2 * HC : 0);
        float gzc_i = 0.0f;
#pragma unroll
        for (int q = 0; q < EPL; ++q) {
            const float vq = __shfl_sync(0xffffffffu, gzc[q], ec & 31);
            if (ec / 32 == q) gzc_i = vq;
        }
        if (i >= M) continue;
        float gz, gm;
        if (i < HC) {
            const float sp = sigm(fmaf(m, s0, __ldg(hc_base + i)));
            gz = (g_pre ? __ldg(g_pre + t * HC + i) : 0.0f) * sp * (1.0f - sp);
            gm = gz * s0;
            z0 = fmaf(gz, m, z0);
        } else if (i < 2 * HC) {
            const float sq = sigm(fmaf(m, s1, __ldg(hc_base + i)));
            gz = sT[L::kSPost + i - HC] * 2.0f * sq * (1.0f - sq);
            gm = gz * s1;
            z1 = fmaf(gz, m, z1);
            wt[L::kPost + i - HC] = 2.0f * sq;
        } else {
            gz = gzc_i;
            gm = gz * s2;
            z2 = fmaf(gz, m, z2);
        }
        gr = fmaf(gm, a, gr);
        const float ga = gm * r;
        wt[L::kGa + i] = ga;
        wt[L::kGz + i] = gz;
        // ga = hi + mid + lo in bf16, to about 2^-24 of itself
        const uint32_t hi = pack_bf16x2(ga, 0.0f) & 0xffffu;
        const float r1 = ga - bf16lo(hi);
        const uint32_t mid = pack_bf16x2(r1, 0.0f) & 0xffffu;
        gpart[i] = (uint16_t)hi;
        gpart[M + i] = (uint16_t)mid;
        gpart[2 * M + i] = (uint16_t)(pack_bf16x2(r1 - bf16lo(mid), 0.0f) & 0xffffu);
    }
    z0 = warp_sum(z0);
    z1 = warp_sum(z1);
    z2 = warp_sum(z2);
    gr = warp_sum(gr);
    if (lane < HC) {
        wt[L::kPm + lane] = pm[lane];
        // g_pre_mix_s = sum_c x_s (rs w g_hn - k3 h) = rs A_s - k3 B_s
        g_pm[t * HC + lane] = rs * sT[L::kSA + lane] - k3 * sT[L::kSB + lane];
    }
    if (lane == 0) {
        wt[L::kGzm] = z0;
        wt[L::kGzm + 1] = z1;
        wt[L::kGzm + 2] = z2;
        wt[L::kRs] = rs;
        wt[L::kCr] = -gr * r * r * r / (float)K;  // the statistic's term: cr * x_k
        wt[L::kK3] = k3;
    }
}

// g_x[s][c] = pm_s g_h + cr x_s + sum_k comb_sk g_y_k + sum_i g_a_i W[i][s*d + c],
// g_h = rs w g_hn - k3 h; g_f[c] = sum_k post_k g_y_k.  Four channels per step,
// TOK tokens per CTA (the W columns of a step loaded once for all of them).
template <int HC, int TOK>
__global__ void __launch_bounds__(kThreads)
kg_gx(const uint16_t *__restrict__ x, const float *__restrict__ hc_fn, const float *__restrict__ norm_w,
      const float *__restrict__ g_hn, const float *__restrict__ g_y, const float *__restrict__ ws, int64_t n,
      int d, float *__restrict__ g_x, float *__restrict__ g_f) {
    using L = Lay<HC>;
    constexpr int M = L::kMix;
    __shared__ float rec[TOK][L::kWs];
    const int64_t t0 = (int64_t)blockIdx.x * TOK;
    const int ntok = (n - t0 < TOK) ? (int)(n - t0) : TOK;
    const int64_t K = (int64_t)HC * d;
    for (int i = threadIdx.x; i < ntok * L::kWs; i += kThreads) rec[i / L::kWs][i % L::kWs] = ws[t0 * L::kWs + i];
    __syncthreads();
    for (int c = threadIdx.x; c < d / 4; c += kThreads) {
        // the W columns of these 4 channels, read once for the CTA's TOK tokens
        float wv[M][HC][4];
#pragma unroll
        for (int i = 0; i < M; ++i)
#pragma unroll
            for (int s = 0; s < HC; ++s) ld4f(hc_fn + i * K + (int64_t)s * d + 4 * c, wv[i][s]);
        float w[4];
        ld4f(norm_w + 4 * c, w);
        for (int u = 0; u < ntok; ++u) {
            const int64_t t = t0 + u;
            const float *r = rec[u];
            const float rs = r[L::kRs], cr = r[L::kCr], k3 = r[L::kK3];
            float xv[HC][4], gy[HC][4], gh[4], ghh[4], gf[4];
#pragma unroll
            for (int s = 0; s < HC; ++s) {
                ld4bf(x + t * K + (int64_t)s * d + 4 * c, xv[s]);
                ld4f(g_y + (t * HC + s) * d + 4 * c, gy[s]);
            }
            ld4f(g_hn + t * d + 4 * c, gh);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float hv = r[L::kPm] * xv[0][e];
#pragma unroll
                for (int s = 1; s < HC; ++s) hv = fmaf(r[L::kPm + s], xv[s][e], hv);
                ghh[e] = rs * (w[e] * gh[e]) - k3 * round_bf16(hv);
                float fvv = r[L::kPost] * gy[0][e];
#pragma unroll
                for (int k = 1; k < HC; ++k) fvv = fmaf(r[L::kPost + k], gy[k][e], fvv);
                gf[e] = fvv;
            }
            *reinterpret_cast<float4 *>(g_f + t * d + 4 * c) = make_float4(gf[0], gf[1], gf[2], gf[3]);
#pragma unroll
            for (int s = 0; s < HC; ++s) {
                float gx[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float a = fmaf(r[L::kPm + s], ghh[e], cr * xv[s][e]);
#pragma unroll
                    for (int k = 0; k < HC; ++k) a = fmaf(r[L::kComb + s * HC + k], gy[k][e], a);
                    gx[e] = a;
                }
#pragma unroll
                for (int i = 0; i < M; ++i) {
                    const float ga = r[L::kGa + i];
#pragma unroll
                    for (int e = 0; e < 4; ++e) gx[e] = fmaf(ga, wv[i][s][e], gx[e]);
                }
                *reinterpret_cast<float4 *>(g_x + (t * HC + s) * d + 4 * c) = make_float4(gx[0], gx[1], gx[2], gx[3]);
            }
        }
    }
}

// The same g_x and g_f for 16 tokens per CTA (hc >= 8), so that hc_fn is read
// once per 16 tokens (kg_gx reads all of it per token: 13 MB at eight
// streams).  The CTA walks d in chunks of 64 columns: first the projection
// term D[t][s][c] = sum_i g_a[t][i] W[i][s*d + c] for its tokens into shared
// memory (each thread HC * 64 / 256 (stream, column) pairs, W read from L2
// once per chunk, g_a kept mix-major so that one i gives the 16 tokens' values
// in four 16-byte loads); then the rest per (token, column) as kg_gx computes
// it, plus D, with two adjacent columns per thread (8-byte loads and stores of
// the fp32 streams) in two passes of eight tokens.  Only the record fields
// that part reads are staged.  Sums are fp32 in index order (i, then the
// terms in kg_gx's order), as kg_gx.  At most 64 registers: four CTAs per SM,
// so that 8,192 tokens (512 CTAs) fit in one wave.
constexpr int kGxT = 16;     // tokens per CTA
constexpr int kGxTokSmall = 4;  // tokens per CTA of kg_gx (hc = 2): hc_fn read once per 4 tokens
constexpr int kGxC = 64;     // columns of d per chunk
template <int HC>
__global__ void __launch_bounds__(kThreads, 4)
kg_gx_tiled(const uint16_t *__restrict__ x, const float *__restrict__ hc_fn, const float *__restrict__ norm_w,
            const float *__restrict__ g_hn, const float *__restrict__ g_y, const float *__restrict__ ws,
            int64_t n, int d, float *__restrict__ g_x, float *__restrict__ g_f) {
    using L = Lay<HC>;
    constexpr int M = L::kMix;
    constexpr int kPairs = HC * kGxC / kThreads;
    constexpr int kF = L::kK3 + 1 - L::kPost;
    static_assert(HC * kGxC % kThreads == 0 && kGxT == 16 && kGxT * kGxC / 2 == 2 * kThreads, "thread maps");
    __shared__ __align__(16) float gaT[M][kGxT];
    __shared__ float fld[kGxT][kF];
    __shared__ __align__(16) float dsum[kGxT][HC][kGxC];
    const int64_t t0 = (int64_t)blockIdx.x * kGxT;
    const int cnt = (int)((n - t0 < kGxT) ? n - t0 : kGxT);
    const int64_t K = (int64_t)HC * d;
    for (int q = threadIdx.x; q < kGxT * M; q += kThreads) {
        const int u = q / M, i = q % M;
        gaT[i][u] = u < cnt ? ws[(t0 + u) * L::kWs + L::kGa + i] : 0.0f;
    }
    for (int q = threadIdx.x; q < kGxT * kF; q += kThreads) {
        const int u = q / kF, j = q % kF;
        fld[u][j] = u < cnt ? ws[(t0 + u) * L::kWs + L::kPost + j] : 0.0f;
    }
    for (int c0 = 0; c0 < d; c0 += kGxC) {
        __syncthreads();
        {
            // (1) D for (stream, column) pairs p = threadIdx.x + kThreads * j
            float acc[kPairs][kGxT];
            const float *wcol[kPairs];
#pragma unroll
            for (int j = 0; j < kPairs; ++j) {
                const int pr = threadIdx.x + kThreads * j;
                wcol[j] = hc_fn + (int64_t)(pr / kGxC) * d + c0 + pr % kGxC;
#pragma unroll
                for (int u = 0; u < kGxT; ++u) acc[j][u] = 0.0f;
            }
            for (int i = 0; i < M; ++i) {
                float w[kPairs];
#pragma unroll
                for (int j = 0; j < kPairs; ++j) w[j] = __ldg(wcol[j] + (int64_t)i * K);
                const float4 *g4 = reinterpret_cast<const float4 *>(gaT[i]);
#pragma unroll
                for (int v = 0; v < kGxT / 4; ++v) {
                    const float4 a = g4[v];
#pragma unroll
                    for (int j = 0; j < kPairs; ++j) {
                        acc[j][4 * v + 0] = fmaf(a.x, w[j], acc[j][4 * v + 0]);
                        acc[j][4 * v + 1] = fmaf(a.y, w[j], acc[j][4 * v + 1]);
                        acc[j][4 * v + 2] = fmaf(a.z, w[j], acc[j][4 * v + 2]);
                        acc[j][4 * v + 3] = fmaf(a.w, w[j], acc[j][4 * v + 3]);
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < kPairs; ++j) {
                const int pr = threadIdx.x + kThreads * j;
#pragma unroll
                for (int u = 0; u < kGxT; ++u) dsum[u][pr / kGxC][pr % kGxC] = acc[j][u];
            }
        }
        __syncthreads();
        // (2) thread: tokens u = tid / 32 and u + 8, columns c0 + 2 (tid % 32), + 1
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
            const int u = threadIdx.x / (kGxC / 2) + half * (kThreads / (kGxC / 2)), cc = 2 * (threadIdx.x % (kGxC / 2));
            if (u < cnt) {
                const int c = c0 + cc;
                const int64_t t = t0 + u;
                const float *r = fld[u];
                float xv[HC][2], gy[HC][2];
#pragma unroll
                for (int sI = 0; sI < HC; ++sI) {
                    const uint32_t xb = __ldg(reinterpret_cast<const uint32_t *>(x + t * K + (int64_t)sI * d + c));
                    xv[sI][0] = bf16lo(xb);
                    xv[sI][1] = __uint_as_float(xb & 0xffff0000u);
                    const float2 g2 = __ldg(reinterpret_cast<const float2 *>(g_y + (t * HC + sI) * d + c));
                    gy[sI][0] = g2.x;
                    gy[sI][1] = g2.y;
                }
                const float2 gh2 = __ldg(reinterpret_cast<const float2 *>(g_hn + t * d + c));
                const float2 wn2 = __ldg(reinterpret_cast<const float2 *>(norm_w + c));
                const float gh[2] = {gh2.x, gh2.y}, wn[2] = {wn2.x, wn2.y};
                float gf[2], gx[HC][2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float hv = r[L::kPm - L::kPost] * xv[0][e];
#pragma unroll
                    for (int sI = 1; sI < HC; ++sI) hv = fmaf(r[L::kPm - L::kPost + sI], xv[sI][e], hv);
                    const float ghh = r[L::kRs - L::kPost] * (wn[e] * gh[e]) - r[L::kK3 - L::kPost] * round_bf16(hv);
                    float fvv = r[L::kPost - L::kPost] * gy[0][e];
#pragma unroll
                    for (int k = 1; k < HC; ++k) fvv = fmaf(r[L::kPost - L::kPost + k], gy[k][e], fvv);
                    gf[e] = fvv;
#pragma unroll
                    for (int sI = 0; sI < HC; ++sI) {
                        float a = fmaf(r[L::kPm - L::kPost + sI], ghh, r[L::kCr - L::kPost] * xv[sI][e]);
#pragma unroll
                        for (int k = 0; k < HC; ++k) a = fmaf(r[L::kComb - L::kPost + sI * HC + k], gy[k][e], a);
                        gx[sI][e] = a + dsum[u][sI][cc + e];
                    }
                }
                *reinterpret_cast<float2 *>(g_f + t * d + c) = make_float2(gf[0], gf[1]);
#pragma unroll
                for (int sI = 0; sI < HC; ++sI)
                    *reinterpret_cast<float2 *>(g_x + (t * HC + sI) * d + c) = make_float2(gx[sI][0], gx[sI][1]);
            }
        }
    }
}

// g_hc_fn partial sums on the tensor cores: part[b][i][k] = sum_t g_a[t][i]
// x[t][k] over block b, as bf16 mma.sync m16n8k16 with x exact and g_a in
// three bf16 parts (from the record).  A CTA takes 256 columns k of one
// block; tiles of 16 tokens (x and the parts) are double-buffered through
// cp.async (rows past the block are zero-filled).  Warp w owns columns
// 32w .. 32w + 31 (two m-tiles of 16; A = x^T by ldmatrix.trans), all mix
// rows (n-tiles of 8; B = the parts by ldmatrix.trans).
constexpr int kFnCols = 256;
template <int HC>
struct FnTc {
    static constexpr int M = (2 + HC) * HC;
    static constexpr int NT = M / 8;                        // n-tiles
    static constexpr int XROW = kFnCols + 8;                // bf16 per staged x row (528 B: odd 16-byte units)
    static constexpr int PB = 3 * M;                        // bf16 of parts per token
    static constexpr int PROW = (PB * 2 / 16) % 2 ? PB : PB + 8;  // padded to an odd number of 16-byte units
    struct Stage {
        uint16_t x[kFnTile][XROW];
        uint16_t p[kFnTile][PROW];
    };
    static_assert(M % 8 == 0 && (PB * 2) % 16 == 0, "whole n-tiles, 16-byte part rows");
    static_assert(sizeof(Stage) % 16 == 0, "16-byte stage size");
};

template <int HC>
__global__ void __launch_bounds__(kThreads, 2)
kg_fn_tc(const uint16_t *__restrict__ x, const float *__restrict__ ws, int64_t n, int K,
         float *__restrict__ part) {
    using L = Lay<HC>;
    using F = FnTc<HC>;
    constexpr int M = F::M, NT = F::NT;
    __shared__ __align__(16) typename F::Stage stg[2];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int k0 = blockIdx.x * kFnCols;
    const int64_t t0 = (int64_t)blockIdx.y * kTokBlock;
    const int64_t t1 = (t0 + kTokBlock < n) ? t0 + kTokBlock : n;
    const int ntiles = (int)((t1 - t0 + kFnTile - 1) / kFnTile);
    auto issue = [&](int it) {
        if (it < ntiles) {
            typename F::Stage &S = stg[it & 1];
            const int64_t tb = t0 + (int64_t)it * kFnTile;
            for (int c = threadIdx.x; c < kFnTile * (kFnCols / 8); c += kThreads) {
                const int u = c / (kFnCols / 8), j = c % (kFnCols / 8);
                const bool ok = tb + u < t1 && k0 + 8 * j < K;
                cp_async16(&S.x[u][8 * j], ok ? x + (tb + u) * K + k0 + 8 * j : x, ok ? 16 : 0);
            }
            for (int c = threadIdx.x; c < kFnTile * (F::PB / 8); c += kThreads) {
                const int u = c / (F::PB / 8), j = c % (F::PB / 8);
                const bool ok = tb + u < t1;
                const uint16_t *src = reinterpret_cast<const uint16_t *>(ws + (tb + u) * L::kWs + L::kGaP) + 8 * j;
                cp_async16(&S.p[u][8 * j], ok ? src : reinterpret_cast<const uint16_t *>(ws), ok ? 16 : 0);
            }
        }
        cp_async_commit();
    };
    float acc[2][NT][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.0f;
    // ldmatrix rows: x^T (A): token (l & 7) + 8 (l >> 4), columns 8 ((l >> 3) & 1) of the m-tile;
    // parts (B): matrix 2 (3p + nt) + h = tokens 8h .. 8h + 7, mixes 8nt .. of part p
    const uint32_t xa_off = (uint32_t)((((lane & 7) + 8 * (lane >> 4)) * F::XROW + 32 * warp + 8 * ((lane >> 3) & 1)) * 2);
    issue(0);
    for (int it = 0; it < ntiles; ++it) {
        issue(it + 1);
        cp_async_wait<1>();
        __syncthreads();
        const typename F::Stage &S = stg[it & 1];
        const uint32_t xs = smem_u32(&S.x[0][0]) + xa_off, ps = smem_u32(&S.p[0][0]);
        uint32_t xa[2][4];
#pragma unroll
        for (int mt = 0; mt < 2; ++mt) ldmatrix_x4_trans(xs + 32 * mt, xa[mt][0], xa[mt][1], xa[mt][2], xa[mt][3]);
#pragma unroll
        for (int p = 2; p >= 0; --p)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                // b0: tokens 0-7, b1: tokens 8-15, mixes 8nt .. 8nt + 7 of part p (two 8x8 matrices)
                const int lrow = (lane & 7) + 8 * ((lane >> 3) & 1);
                uint32_t b0, b1;
                ldmatrix_x2_trans(ps + (uint32_t)((lrow * F::PROW + p * M + 8 * nt) * 2), b0, b1);
#pragma unroll
                for (int mt = 0; mt < 2; ++mt)
                    mma_bf16_16816(acc[mt][nt], xa[mt][0], xa[mt][1], xa[mt][2], xa[mt][3], b0, b1);
            }
        __syncthreads();  // every warp is done with this stage before it is refilled
    }
    cp_async_wait<0>();
    // accumulator (mt, nt, e): column k0 + 32 w + 16 mt + g + 8 (e >> 1), mix 8 nt + 2q + (e & 1)
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int k = k0 + 32 * warp + 16 * mt + g + 8 * (e >> 1), i = 8 * nt + 2 * q + (e & 1);
                if (k < K) part[((int64_t)blockIdx.y * M + i) * K + k] = acc[mt][nt][e];
            }
}

// g_norm_w partial sums over runs of kWRun tokens: part[b][c] = sum_t h[t][c]
// rs_h[t] g_hn[t][c], h as the forward rounds it.  A thread takes eight
// columns (16-byte loads of each stream's x, two of g_hn) and walks the run's
// tokens in order; 64-thread CTAs, enough of them to keep the loads in flight.
constexpr int kWRun = 64;
constexpr int kWThreads = 64;
template <int HC>
__global__ void __launch_bounds__(kWThreads)
kg_w_partial(const uint16_t *__restrict__ x, const float *__restrict__ g_hn, const float *__restrict__ ws,
             int64_t n, int d, float *__restrict__ part) {
    using L = Lay<HC>;
    const int c = 8 * (blockIdx.x * kWThreads + threadIdx.x);  // columns c .. c + 7
    const int64_t t0 = (int64_t)blockIdx.y * kWRun;
    const int64_t t1 = (t0 + kWRun < n) ? t0 + kWRun : n;
    if (c >= d) return;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
#pragma unroll 4
    for (int64_t t = t0; t < t1; ++t) {
        const float *rec = ws + t * L::kWs;
        const uint16_t *xt = x + t * HC * d + c;
        float hv[8], xv[8];
        unpack8(__ldg(reinterpret_cast<const uint4 *>(xt)), xv);
        const float pm0 = __ldg(rec + L::kPm);
#pragma unroll
        for (int e = 0; e < 8; ++e) hv[e] = pm0 * xv[e];
#pragma unroll
        for (int s = 1; s < HC; ++s) {
            unpack8(__ldg(reinterpret_cast<const uint4 *>(xt + (int64_t)s * d)), xv);
            const float pm = __ldg(rec + L::kPm + s);
#pragma unroll
            for (int e = 0; e < 8; ++e) hv[e] = fmaf(pm, xv[e], hv[e]);
        }
        const float rs = __ldg(rec + L::kRs);
        const float4 g0 = __ldg(reinterpret_cast<const float4 *>(g_hn + t * d + c));
        const float4 g1 = __ldg(reinterpret_cast<const float4 *>(g_hn + t * d + c + 4));
        const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = fmaf(round_bf16(hv[e]) * rs, g[e], acc[e]);
    }
    float4 *o = reinterpret_cast<float4 *>(part + (int64_t)blockIdx.y * d + c);
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

// per run of kSRun tokens: the sums over its tokens of g_z (g_hc_base terms)
// and gzm (g_hc_scale terms).  Short runs, so that the launch has enough CTAs
// to keep the record loads in flight.
constexpr int kSRun = 128;
template <int HC>
__global__ void __launch_bounds__(kThreads)
kg_small_partial(const float *__restrict__ ws, int64_t n, float *__restrict__ part) {
    // field j (g_z, then gzm: kGz + kMix = kGzm) = 32 fc + lane; warp w sums
    // tokens 16 w .. 16 w + 15 of the run, then the warp sums in warp order
    using L = Lay<HC>;
    constexpr int F = L::kMix + 3;
    __shared__ float red[kWarps][32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t tw = (int64_t)blockIdx.x * kSRun + (int64_t)warp * (kSRun / kWarps);
    for (int fc = 0; fc < (F + 31) / 32; ++fc) {
        const int j = 32 * fc + lane;
        float acc = 0.0f;
        if (j < F) {
#pragma unroll 8
            for (int u = 0; u < kSRun / kWarps; ++u)
                if (tw + u < n) acc += ws[(tw + u) * L::kWs + L::kGz + j];
        }
        red[warp][lane] = acc;
        __syncthreads();
        if (warp == 0 && j < F) {
            float v = red[0][lane];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) v += red[w][lane];
            part[(int64_t)blockIdx.x * L::kSmall + j] = v;
        }
        __syncthreads();
    }
}

// out[j] = sum_b part[b][j], blocks (or runs) in order.
__global__ void kg_sum_blocks(const float *__restrict__ part, int blocks, int64_t len, float *__restrict__ out) {
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= len) return;
    float s = 0.0f;
    for (int b = 0; b < blocks; ++b) s += part[(int64_t)b * len + j];
    out[j] = s;
}

// out[c] = sum_r part[r][c] over many runs: a CTA takes 32 columns, its eight
// warps each add an eighth of the runs in order, then the warp sums are added
// in warp order (enough CTAs for the loads to be in flight together).
__global__ void __launch_bounds__(kThreads)
kg_sum_runs(const float *__restrict__ part, int runs, int d, float *__restrict__ out) {
    __shared__ float red[kWarps][32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x * 32 + lane;
    const int per = (runs + kWarps - 1) / kWarps;
    const int r0 = warp * per, r1 = (r0 + per < runs) ? r0 + per : runs;
    float acc = 0.0f;
    if (c < d)
#pragma unroll 4
        for (int r = r0; r < r1; ++r) acc += part[(int64_t)r * d + c];
    red[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && c < d) {
        float v = red[0][lane];
#pragma unroll
        for (int w = 1; w < kWarps; ++w) v += red[w][lane];
        out[c] = v;
    }
}

template <int HC>
__global__ void kg_small_final(const float *__restrict__ part, int runs, float *__restrict__ g_base,
                               float *__restrict__ g_scale) {
    using L = Lay<HC>;
    const int j = threadIdx.x;
    if (j >= L::kMix + 3) return;
    float s = 0.0f;
    for (int b = 0; b < runs; ++b) s += part[(int64_t)b * L::kSmall + j];
    if (j < L::kMix) g_base[j] = s;
    else g_scale[j - L::kMix] = s;
}

template <int HC>
size_t ws_bytes(int64_t n, int d) {
    using L = Lay<HC>;
    const int64_t blocks = (n + kTokBlock - 1) / kTokBlock;
    const int64_t wruns = (n + kWRun - 1) / kWRun;
    const int64_t sruns = (n + kSRun - 1) / kSRun;
    const int64_t K = (int64_t)HC * d;
    return (size_t)(n * L::kWs + blocks * L::kMix * K + sruns * L::kSmall + wruns * d) * sizeof(float) +
           proj_umma_wsplit_bytes(HC, K);
}

template <int HC>
cudaError_t launch(const uint16_t *x, const float *pre_mix, const uint16_t *f, const float *hc_fn,
                   const float *hc_scale, const float *hc_base, const float *norm_w, int64_t n, int d,
                   int iters, float eps, float norm_eps, const float *g_hn, const float *g_y,
                   const float *g_pre, float *g_x, float *g_pm, float *g_f, float *g_fn, float *g_scale,
                   float *g_base, float *g_w, void *workspace, cudaStream_t s) {
    using L = Lay<HC>;
    constexpr int M = L::kMix;
    const int64_t K = (int64_t)HC * d;
    const int blocks = (int)((n + kTokBlock - 1) / kTokBlock);
    float *ws = reinterpret_cast<float *>(workspace);
    float *part_fn = ws + n * L::kWs;
    const int wruns = (int)((n + kWRun - 1) / kWRun);
    float *part_w = part_fn + (int64_t)blocks * M * K;
    float *part_s = part_w + (int64_t)wruns * d;
    const int sruns = (int)((n + kSRun - 1) / kSRun);
    uint16_t *wsplit = reinterpret_cast<uint16_t *>(part_s + (int64_t)sruns * L::kSmall);
    // kg_token: one warp per token, up to four per CTA within 200 KB of iterates
    const size_t per_warp = ((size_t)(2 * iters + 1) * HC * HC + L::kSums) * sizeof(float);
    int tok_warps = (int)((200u << 10) / per_warp);
    tok_warps = tok_warps < 1 ? 1 : (tok_warps > 4 ? 4 : tok_warps);
    const size_t smem = per_warp * tok_warps;
    cudaError_t e = cudaFuncSetAttribute(kg_token<HC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // tcgen05 (hc_proj_umma.cu); part_fn, written later by kg_fn_tc, holds its K slices meanwhile
    e = launch_proj_umma(x, hc_fn, n, HC, d, wsplit, ws + L::kA, L::kWs, s, part_fn, (int64_t)blocks * M * K);
    if (e != cudaSuccess) return e;
    kg_token<HC><<<(unsigned)((n + tok_warps - 1) / tok_warps), 32 * tok_warps, smem, s>>>(
        x, pre_mix, f, hc_scale, hc_base, norm_w, n, d, iters, eps, norm_eps, g_hn, g_y, g_pre, g_pm, ws);
    if constexpr (HC >= 8)  // hc_fn of 13 MB: read once per 16 tokens, the projection term in shared memory
        kg_gx_tiled<HC><<<(unsigned)((n + kGxT - 1) / kGxT), kThreads, 0, s>>>(x, hc_fn, norm_w, g_hn, g_y, ws,
                                                                             n, d, g_x, g_f);
    else  // hc_fn of 330 KB: its columns in registers, read once per kGxTokSmall tokens
        kg_gx<HC, kGxTokSmall><<<(unsigned)((n + kGxTokSmall - 1) / kGxTokSmall), kThreads, 0, s>>>(
            x, hc_fn, norm_w, g_hn, g_y, ws, n, d, g_x, g_f);
    kg_fn_tc<HC><<<dim3((unsigned)((K + kFnCols - 1) / kFnCols), (unsigned)blocks), kThreads, 0, s>>>(
        x, ws, n, (int)K, part_fn);
    kg_sum_blocks<<<(unsigned)((M * K + 255) / 256), 256, 0, s>>>(part_fn, blocks, M * K, g_fn);
    kg_w_partial<HC><<<dim3((unsigned)((d / 8 + kWThreads - 1) / kWThreads), (unsigned)wruns), kWThreads, 0, s>>>(
        x, g_hn, ws, n, d, part_w);
    kg_sum_runs<<<(unsigned)((d + 31) / 32), kThreads, 0, s>>>(part_w, wruns, d, g_w);
    kg_small_partial<HC><<<(unsigned)sruns, kThreads, 0, s>>>(ws, n, part_s);
    kg_small_final<HC><<<1, 128, 0, s>>>(part_s, sruns, g_base, g_scale);
    return cudaGetLastError();
}

}  // namespace bwg

size_t backward_generic_workspace_bytes(int64_t n, int hc, int d) {
    if (hc == 2) return bwg::ws_bytes<2>(n, d);
    if (hc == 8) return bwg::ws_bytes<8>(n, d);
    return 0;
}

cudaError_t launch_block_step_backward_generic(int hc, const uint16_t *x, const float *pre_mix,
                                               const uint16_t *f, const float *hc_fn,
                                               const float *hc_scale, const float *hc_base,
                                               const float *norm_w, int64_t n, int d, int iters,
                                               float eps, float norm_eps, const float *g_hn,
                                               const float *g_y, const float *g_pre, float *g_x,
                                               float *g_pm, float *g_f, float *g_fn, float *g_scale,
                                               float *g_base, float *g_w, void *workspace,
                                               cudaStream_t s) {
    if (hc == 2)
        return bwg::launch<2>(x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, n, d, iters, eps, norm_eps, g_hn,
                              g_y, g_pre, g_x, g_pm, g_f, g_fn, g_scale, g_base, g_w, workspace, s);
    if (hc == 8)
        return bwg::launch<8>(x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, n, d, iters, eps, norm_eps, g_hn,
                              g_y, g_pre, g_x, g_pm, g_f, g_fn, g_scale, g_base, g_w, workspace, s);
    return cudaErrorInvalidValue;
}

}  // namespace hc
