// hc_backward.cu -- the backward of one hyper-connection side step (a1-a6),
// for GB300.
//
// What it computes: the derivative of the side step that hc_block_step
// computes (DeepSeek-V4.1 Block page, Code section: Block.hc_mixes,
// Block.hc_pre, attn_norm / ffn_norm, Block.hc_post; "Stream combination"
// page: hc_split_sinkhorn).  The pages give no backward pass: this is the
// plain derivative of those definitions.  The three bf16 casts (h, h_norm,
// y) pass gradients through unchanged, as a dtype cast does in autograd, and
// the backward reads the forward's bf16-rounded h where the forward did.
// Sinkhorn is differentiated step by step through its stored intermediates.
//
// How: k_bwd_token, one CTA per token, recomputes the forward quantities it
// needs (the projection, the statistics, h, the split and the Sinkhorn
// iterates), runs the Sinkhorn backward on one thread, and writes the
// token's gradients (x, pre_mix, f) plus, into the workspace, the per-token
// terms of the parameter gradients.  The parameter gradients are then summed
// over fixed token blocks and the blocks added in a fixed order, so every
// result is deterministic (no atomics).
#include "hc_device.cuh"
#include "hc_launch.h"

namespace hc {

namespace bw {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kWs = 64;          // workspace floats per token: g_a[24], g_z[24], gzm[3], rs_h
constexpr int kTokBlock = 1024;  // tokens per partial sum of a parameter gradient
constexpr int kMaxIters = 128;

// Sum of V per-thread values over the CTA; the totals land in tot[0..V).
template <int V>
__device__ __forceinline__ void block_sums(const float (&v)[V], float (*red)[32], float *tot) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const float s = warp_sum(v[i]);
        if (lane == 0) red[warp][i] = s;
    }
    __syncthreads();
    if (threadIdx.x < V) {
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) s += red[w][threadIdx.x];
        tot[threadIdx.x] = s;
    }
    __syncthreads();
}

__device__ __forceinline__ float sigm(float z) { return 1.0f / (1.0f + expf(-z)); }

__device__ __forceinline__ void load8f(const float *p, float (&o)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w; o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
__device__ __forceinline__ void store8f(float *p, const float (&o)[8]) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(o[0], o[1], o[2], o[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(o[4], o[5], o[6], o[7]);
}

// Shared memory: h of the token (d bf16), then the Sinkhorn iterates
// (2 * iters matrices of 16) and the row softmax (16).
__global__ void __launch_bounds__(kThreads)
k_bwd_token(const uint16_t *__restrict__ x, const float *__restrict__ pre_mix,
            const uint16_t *__restrict__ f, const float *__restrict__ hc_fn,
            const float *__restrict__ hc_scale, const float *__restrict__ hc_base,
            const float *__restrict__ norm_w, int d, int iters, float eps, float norm_eps,
            const float *__restrict__ g_hn, const float *__restrict__ g_y,
            const float *__restrict__ g_pre, float *__restrict__ g_x, float *__restrict__ g_pm,
            float *__restrict__ g_f, float *__restrict__ ws) {
    extern __shared__ uint4 smem_u4[];
    uint4 *sh = smem_u4;                                             // d/8 chunks of h
    float *sP = reinterpret_cast<float *>(smem_u4 + (d >> 3));      // 2*iters*16 iterates
    float *sS = sP + 2 * iters * kHC * kHC;                         // row softmax
    __shared__ float red[kWarps][32];
    __shared__ float tot[32];
    __shared__ float sa[32];  // the projection a[24] and sum x^2
    // g_a[24], the statistic's term cr, rs_h, post[4], comb[16]
    __shared__ float sc[48];
    const int64_t t = blockIdx.x;
    const int K = kHC * d, K8 = K >> 3, d8 = d >> 3;
    const uint16_t *xt = x + t * K;

    // (a) the projection a_i = sum_k x_k W_ik and the statistic sum x^2
    {
        float v[kMix + 1];
#pragma unroll
        for (int i = 0; i <= kMix; ++i) v[i] = 0.0f;
        for (int ch = threadIdx.x; ch < K8; ch += kThreads) {
            float xv[8];
            unpack8(__ldg(reinterpret_cast<const uint4 *>(xt) + ch), xv);
#pragma unroll
            for (int e = 0; e < 8; ++e) v[kMix] = fmaf(xv[e], xv[e], v[kMix]);
#pragma unroll
            for (int i = 0; i < kMix; ++i) {
                float w[8];
                load8f(hc_fn + (int64_t)i * K + 8 * ch, w);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[i] = fmaf(xv[e], w[e], v[i]);
            }
        }
        block_sums<kMix + 1>(v, red, tot);
        if (threadIdx.x <= kMix) sa[threadIdx.x] = tot[threadIdx.x];
        __syncthreads();
    }
    float pm[kHC];
#pragma unroll
    for (int s = 0; s < kHC; ++s) pm[s] = __ldg(pre_mix + t * kHC + s);

    // (b) h (kept), sum h^2, T = sum h w g_hn, g_post_k, g_comb_jk
    {
        float v[2 + kHC + kHC * kHC];
#pragma unroll
        for (int i = 0; i < 2 + kHC + kHC * kHC; ++i) v[i] = 0.0f;
        for (int c = threadIdx.x; c < d8; c += kThreads) {
            float xv[kHC][8], fv[8], gy[kHC][8], gh[8], w[8], h[8];
#pragma unroll
            for (int s = 0; s < kHC; ++s) unpack8(__ldg(reinterpret_cast<const uint4 *>(xt + s * d) + c), xv[s]);
            unpack8(__ldg(reinterpret_cast<const uint4 *>(f + t * d) + c), fv);
#pragma unroll
            for (int k = 0; k < kHC; ++k) load8f(g_y + (t * kHC + k) * d + 8 * c, gy[k]);
            load8f(g_hn + t * d + 8 * c, gh);
            load8f(norm_w + 8 * c, w);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                h[e] = pm[0] * xv[0][e];
#pragma unroll
                for (int s = 1; s < kHC; ++s) h[e] = fmaf(pm[s], xv[s][e], h[e]);
            }
            const uint4 hb = pack8(h);
            sh[c] = hb;
            unpack8(hb, h);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                v[0] = fmaf(h[e], h[e], v[0]);
                v[1] = fmaf(h[e] * w[e], gh[e], v[1]);
#pragma unroll
                for (int k = 0; k < kHC; ++k) v[2 + k] = fmaf(fv[e], gy[k][e], v[2 + k]);
#pragma unroll
                for (int j = 0; j < kHC; ++j)
#pragma unroll
                    for (int k = 0; k < kHC; ++k)
                        v[2 + kHC + j * kHC + k] = fmaf(xv[j][e], gy[k][e], v[2 + kHC + j * kHC + k]);
            }
        }
        block_sums<2 + kHC + kHC * kHC>(v, red, tot);
    }

    // (c) one thread: split + Sinkhorn forward with its iterates, then back
    if (threadIdx.x == 0) {
        const float *a = sa;
        const float r = rsqrtf(sa[kMix] / (float)K + norm_eps);
        const float rs = rsqrtf(tot[0] / (float)d + norm_eps);
        const float s0 = __ldg(hc_scale), s1 = __ldg(hc_scale + 1), s2 = __ldg(hc_scale + 2);
        float m[kMix];
#pragma unroll
        for (int i = 0; i < kMix; ++i) m[i] = a[i] * r;
        // the row softmax S and P[0] = S + eps
        for (int j = 0; j < kHC; ++j) {
            float L[kHC], mx = -INFINITY, s = 0.0f;
            for (int k = 0; k < kHC; ++k) {
                L[k] = fmaf(m[2 * kHC + j * kHC + k], s2, __ldg(hc_base + 2 * kHC + j * kHC + k));
                mx = fmaxf(mx, L[k]);
            }
            for (int k = 0; k < kHC; ++k) {
                L[k] = expf(L[k] - mx);
                s += L[k];
            }
            for (int k = 0; k < kHC; ++k) {
                sS[j * kHC + k] = L[k] / s;
                sP[j * kHC + k] = sS[j * kHC + k] + eps;
            }
        }
        // steps 1 .. 2*iters-1: a column step for odd, a row step for even steps
        for (int st = 1; st < 2 * iters; ++st) {
            const float *pa = sP + (st - 1) * 16;
            float *pb = sP + st * 16;
            for (int i = 0; i < kHC; ++i) {
                float s = 0.0f;
                for (int o = 0; o < kHC; ++o) s += (st & 1) ? pa[o * kHC + i] : pa[i * kHC + o];
                const float inv = 1.0f / (s + eps);
                for (int o = 0; o < kHC; ++o) {
                    const int idx = (st & 1) ? o * kHC + i : i * kHC + o;
                    pb[idx] = pa[idx] * inv;
                }
            }
        }
        const float *comb = sP + (2 * iters - 1) * 16;
        // back through the steps: g (the gradient of the current iterate)
        float g[kHC * kHC];
        for (int i = 0; i < kHC * kHC; ++i) g[i] = tot[2 + kHC + i];
        for (int st = 2 * iters - 1; st >= 1; --st) {
            const float *pa = sP + (st - 1) * 16, *pb = sP + st * 16;
            for (int i = 0; i < kHC; ++i) {
                float s = 0.0f, dot = 0.0f;
                for (int o = 0; o < kHC; ++o) {
                    const int idx = (st & 1) ? o * kHC + i : i * kHC + o;
                    s += pa[idx];
                    dot = fmaf(g[idx], pb[idx], dot);
                }
                const float inv = 1.0f / (s + eps);
                for (int o = 0; o < kHC; ++o) {
                    const int idx = (st & 1) ? o * kHC + i : i * kHC + o;
                    g[idx] = (g[idx] - dot) * inv;
                }
            }
        }
        float gm[kMix], gz[kMix];
        for (int j = 0; j < kHC; ++j) {
            float dot = 0.0f;
            for (int k = 0; k < kHC; ++k) dot = fmaf(g[j * kHC + k], sS[j * kHC + k], dot);
            for (int k = 0; k < kHC; ++k) gz[2 * kHC + j * kHC + k] = sS[j * kHC + k] * (g[j * kHC + k] - dot);
        }
        float gzm0 = 0.0f, gzm1 = 0.0f, gzm2 = 0.0f;
        for (int j = 0; j < kHC; ++j) {
            const float sp = sigm(fmaf(m[j], s0, __ldg(hc_base + j)));
            gz[j] = (g_pre ? __ldg(g_pre + t * kHC + j) : 0.0f) * sp * (1.0f - sp);
            const float sq = sigm(fmaf(m[kHC + j], s1, __ldg(hc_base + kHC + j)));
            gz[kHC + j] = tot[2 + j] * 2.0f * sq * (1.0f - sq);
            sc[26 + j] = 2.0f * sq;  // post
            gm[j] = gz[j] * s0;
            gm[kHC + j] = gz[kHC + j] * s1;
            gzm0 = fmaf(gz[j], m[j], gzm0);
            gzm1 = fmaf(gz[kHC + j], m[kHC + j], gzm1);
        }
        for (int i = 2 * kHC; i < kMix; ++i) {
            gm[i] = gz[i] * s2;
            gzm2 = fmaf(gz[i], m[i], gzm2);
        }
        float gr = 0.0f;
        for (int i = 0; i < kMix; ++i) gr = fmaf(gm[i], a[i], gr);
        float *wt = ws + t * kWs;
        for (int i = 0; i < kMix; ++i) {
            wt[i] = gm[i] * r;       // g_a
            wt[kMix + i] = gz[i];    // g_z
            sc[i] = gm[i] * r;
        }
        wt[2 * kMix] = gzm0;
        wt[2 * kMix + 1] = gzm1;
        wt[2 * kMix + 2] = gzm2;
        wt[2 * kMix + 3] = rs;
        sc[24] = -gr * r * r * r / (float)K;  // the statistic's term: cr * x_k
        sc[25] = rs;
        for (int i = 0; i < kHC * kHC; ++i) sc[30 + i] = comb[i];
    }
    __syncthreads();

    // (d) g_h, g_x, g_f; g_pre_mix partial sums
    {
        const float rs = sc[25], cr = sc[24], T = tot[1];
        const float k3 = rs * rs * rs / (float)d * T;
        float ga[kMix], post[kHC], comb[kHC * kHC];
#pragma unroll
        for (int i = 0; i < kMix; ++i) ga[i] = sc[i];
#pragma unroll
        for (int k = 0; k < kHC; ++k) post[k] = sc[26 + k];
#pragma unroll
        for (int i = 0; i < kHC * kHC; ++i) comb[i] = sc[30 + i];
        float gp[kHC] = {0.0f, 0.0f, 0.0f, 0.0f};
        for (int c = threadIdx.x; c < d8; c += kThreads) {
            float h[8], w[8], gh[8], gy[kHC][8], gu[8];
            unpack8(sh[c], h);
            load8f(norm_w + 8 * c, w);
            load8f(g_hn + t * d + 8 * c, gh);
#pragma unroll
            for (int k = 0; k < kHC; ++k) load8f(g_y + (t * kHC + k) * d + 8 * c, gy[k]);
#pragma unroll
            for (int e = 0; e < 8; ++e) gu[e] = rs * (w[e] * gh[e]) - k3 * h[e];  // g_h
            float gf[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float acc = post[0] * gy[0][e];
#pragma unroll
                for (int k = 1; k < kHC; ++k) acc = fmaf(post[k], gy[k][e], acc);
                gf[e] = acc;
            }
            store8f(g_f + t * d + 8 * c, gf);
#pragma unroll
            for (int s = 0; s < kHC; ++s) {
                float xv[8], gx[8];
                unpack8(__ldg(reinterpret_cast<const uint4 *>(xt + s * d) + c), xv);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    gp[s] = fmaf(xv[e], gu[e], gp[s]);
                    float acc = fmaf(pm[s], gu[e], cr * xv[e]);
#pragma unroll
                    for (int k = 0; k < kHC; ++k) acc = fmaf(comb[s * kHC + k], gy[k][e], acc);
                    gx[e] = acc;
                }
#pragma unroll
                for (int i = 0; i < kMix; ++i) {
                    float wv[8];
                    load8f(hc_fn + (int64_t)i * K + (int64_t)s * d + 8 * c, wv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) gx[e] = fmaf(ga[i], wv[e], gx[e]);
                }
                store8f(g_x + t * K + (int64_t)s * d + 8 * c, gx);
            }
        }
        block_sums<kHC>(gp, red, tot);
        if (threadIdx.x < kHC) g_pm[t * kHC + threadIdx.x] = tot[threadIdx.x];
    }
}

// g_hc_fn partial sums over a block of kTokBlock tokens: partial[b][i][k] =
// sum over the block's tokens of g_a[t][i] * x[t][k]; one thread per column k.
__global__ void __launch_bounds__(kThreads)
k_bwd_fn_partial(const uint16_t *__restrict__ x, const float *__restrict__ ws, int64_t n, int K,
                 float *__restrict__ part) {
    __shared__ float sga[32][kMix];
    const int k = blockIdx.x * kThreads + threadIdx.x;
    const int64_t t0 = (int64_t)blockIdx.y * kTokBlock;
    const int64_t t1 = (t0 + kTokBlock < n) ? t0 + kTokBlock : n;
    float acc[kMix];
#pragma unroll
    for (int i = 0; i < kMix; ++i) acc[i] = 0.0f;
    for (int64_t tb = t0; tb < t1; tb += 32) {
        const int cnt = (int)((t1 - tb < 32) ? t1 - tb : 32);
        __syncthreads();
        for (int q = threadIdx.x; q < cnt * kMix; q += kThreads)
            sga[q / kMix][q % kMix] = ws[(tb + q / kMix) * kWs + q % kMix];
        __syncthreads();
        if (k < K) {
            for (int u = 0; u < cnt; ++u) {
                const float xv = __uint_as_float((uint32_t)x[(tb + u) * K + k] << 16);
#pragma unroll
                for (int i = 0; i < kMix; ++i) acc[i] = fmaf(sga[u][i], xv, acc[i]);
            }
        }
    }
    if (k < K)
#pragma unroll
        for (int i = 0; i < kMix; ++i) part[((int64_t)blockIdx.y * kMix + i) * K + k] = acc[i];
}

// g_norm_w partial sums: partial[b][c] = sum over the block's tokens of
// h[t][c] * rs_h[t] * g_hn[t][c], h recomputed exactly as k_bwd_token does.
__global__ void __launch_bounds__(kThreads)
k_bwd_w_partial(const uint16_t *__restrict__ x, const float *__restrict__ pre_mix,
                const float *__restrict__ g_hn, const float *__restrict__ ws, int64_t n, int d,
                float *__restrict__ part) {
    const int c = blockIdx.x * kThreads + threadIdx.x;
    const int64_t t0 = (int64_t)blockIdx.y * kTokBlock;
    const int64_t t1 = (t0 + kTokBlock < n) ? t0 + kTokBlock : n;
    if (c >= d) return;
    float acc = 0.0f;
    for (int64_t t = t0; t < t1; ++t) {
        const uint16_t *xt = x + t * kHC * d;
        float h = __ldg(pre_mix + t * kHC) * __uint_as_float((uint32_t)xt[c] << 16);
#pragma unroll
        for (int s = 1; s < kHC; ++s)
            h = fmaf(__ldg(pre_mix + t * kHC + s), __uint_as_float((uint32_t)xt[s * d + c] << 16), h);
        h = bf16lo(pack_bf16x2(h, 0.0f));  // the forward's bf16 h
        acc = fmaf(h * __ldg(ws + t * kWs + 2 * kMix + 3), __ldg(g_hn + t * d + c), acc);
    }
    part[(int64_t)blockIdx.y * d + c] = acc;
}

// out[j] = sum_b part[b][j], blocks in order.
__global__ void k_bwd_sum_blocks(const float *__restrict__ part, int blocks, int64_t len,
                                 float *__restrict__ out) {
    const int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= len) return;
    float s = 0.0f;
    for (int b = 0; b < blocks; ++b) s += part[(int64_t)b * len + j];
    out[j] = s;
}

// g_hc_base[i] = sum_t g_z[t][i], g_hc_scale[j] = sum_t gzm[t][j]: one CTA,
// each thread a fixed stride of tokens, then a fixed tree.
__global__ void __launch_bounds__(kThreads)
k_bwd_small(const float *__restrict__ ws, int64_t n, float *__restrict__ g_base,
            float *__restrict__ g_scale) {
    __shared__ float red[kWarps][32];
    __shared__ float tot[32];
    float v[kMix + 3];
#pragma unroll
    for (int i = 0; i < kMix + 3; ++i) v[i] = 0.0f;
    for (int64_t t = threadIdx.x; t < n; t += kThreads)
#pragma unroll
        for (int i = 0; i < kMix + 3; ++i) v[i] += ws[t * kWs + kMix + i];
    block_sums<kMix + 3>(v, red, tot);
    if (threadIdx.x < kMix) g_base[threadIdx.x] = tot[threadIdx.x];
    else if (threadIdx.x < kMix + 3) g_scale[threadIdx.x - kMix] = tot[threadIdx.x];
}

}  // namespace bw

// Scratch for the backward without a caller workspace: a fixed array in
// device memory, part of the module image, so a call allocates nothing.
// One array per process and device: such calls must not run concurrently.
constexpr size_t kStaticScratchBytes = size_t(64) << 20;
static __device__ __align__(256) unsigned char g_bwd_scratch[kStaticScratchBytes];

size_t backward_static_scratch_bytes() { return kStaticScratchBytes; }

cudaError_t backward_static_scratch(void **ptr) { return cudaGetSymbolAddress(ptr, g_bwd_scratch); }

size_t backward_workspace_bytes(int64_t n, int d) {
    const int64_t blocks = (n + bw::kTokBlock - 1) / bw::kTokBlock;
    const int64_t K = (int64_t)kHC * d;
    return (size_t)(n * bw::kWs + blocks * kMix * K + blocks * d) * sizeof(float);
}

cudaError_t launch_block_step_backward(const uint16_t *x, const float *pre_mix, const uint16_t *f,
                                       const float *hc_fn, const float *hc_scale,
                                       const float *hc_base, const float *norm_w, int64_t n, int d,
                                       int iters, float eps, float norm_eps, const float *g_hn,
                                       const float *g_y, const float *g_pre, float *g_x,
                                       float *g_pm, float *g_f, float *g_fn, float *g_scale,
                                       float *g_base, float *g_w, void *workspace, cudaStream_t s) {
    using namespace bw;
    const int64_t K = (int64_t)kHC * d;
    const int blocks = (int)((n + kTokBlock - 1) / kTokBlock);
    float *ws = reinterpret_cast<float *>(workspace);
    float *part_fn = ws + n * kWs;
    float *part_w = part_fn + (int64_t)blocks * kMix * K;
    const size_t smem = (size_t)d * 2 + (size_t)(2 * iters + 1) * kHC * kHC * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(k_bwd_token, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    k_bwd_token<<<(unsigned)n, kThreads, smem, s>>>(x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w,
                                                   d, iters, eps, norm_eps, g_hn, g_y, g_pre, g_x,
                                                   g_pm, g_f, ws);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    k_bwd_fn_partial<<<dim3((unsigned)((K + kThreads - 1) / kThreads), (unsigned)blocks), kThreads, 0, s>>>(
        x, ws, n, (int)K, part_fn);
    k_bwd_sum_blocks<<<(unsigned)((kMix * K + 255) / 256), 256, 0, s>>>(part_fn, blocks, kMix * K, g_fn);
    k_bwd_w_partial<<<dim3((unsigned)((d + kThreads - 1) / kThreads), (unsigned)blocks), kThreads, 0, s>>>(
        x, pre_mix, g_hn, ws, n, d, part_w);
    k_bwd_sum_blocks<<<(unsigned)((d + 255) / 256), 256, 0, s>>>(part_w, blocks, d, g_w);
    k_bwd_small<<<1, kThreads, 0, s>>>(ws, n, g_base, g_scale);
    return cudaGetLastError();
}

}  // namespace hc
