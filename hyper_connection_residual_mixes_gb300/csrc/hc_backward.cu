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
// How, in three passes over the batch:
//   k_bwd_proj   16 tokens per CTA: the projection a = x W^T and sum x^2,
//                x staged through shared memory with cp.async, each weight
//                row read once per tile (W is the 24 x hc*d matrix hc_fn);
//   k_bwd_token  one CTA per token: h, the statistics, the split and
//                Sinkhorn forward with its iterates, the Sinkhorn backward on
//                one thread, g_pre_mix; writes a per-token record;
//   k_bwd_gx     one CTA per (64 columns of d, all four streams) x (block of
//                1,024 tokens), the column's 24 weights in registers: g_x,
//                g_f, and the block's partial sums of g_hc_fn, g_norm_w and
//                the per-token terms of g_hc_base / g_hc_scale.
// The partial sums are then added over the blocks in a fixed order, so every
// result is deterministic (no atomics).
#include "hc_device.cuh"
#include "hc_launch.h"

namespace hc {

namespace bw {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kTokBlock = 1024;  // tokens per partial sum of a parameter gradient

// The per-token record in the workspace (floats).  [0, kRec) is what k_bwd_gx
// stages for each token; the rest feeds the hc_base / hc_scale sums or comes
// from k_bwd_proj.
constexpr int kWs = 112;
constexpr int kGa = 0;      // g_a[24]: the gradient of the projection a
constexpr int kPost = 24;   // post[4]
constexpr int kComb = 28;   // comb[16]
constexpr int kPm = 44;     // pre_mix[4]
constexpr int kRs = 48;     // rs_h = 1 / RMS(h)
constexpr int kCr = 49;     // the statistic's coefficient of x in g_x
constexpr int kK3 = 50;     // rs_h^3 / d * sum(h w g_hn)
constexpr int kRec = 52;
constexpr int kGz = 52;     // g_z[24]: the gradient of the pre-activations (= g_hc_base terms)
constexpr int kGzm = 76;    // gzm[3]: the g_hc_scale terms
constexpr int kA = 80;      // a[24] (k_bwd_proj)
constexpr int kSS = 104;    // sum x^2 (k_bwd_proj)
constexpr int kSmall = 32;  // partial sums per block for hc_base (24) and hc_scale (3)

constexpr int kProjTok = 16;    // tokens per CTA of k_bwd_proj
constexpr int kProjCols = 256;  // columns of x per stage
constexpr int kProjStages = 4;
constexpr int kGxCols = 64;     // columns of d per CTA of k_bwd_gx
constexpr int kGxTile = 16;     // tokens per staged tile of k_bwd_gx
constexpr int kGxStages = 3;
static_assert(kProjTok == 2 * kWarps, "each warp sums x^2 of two tokens");
static_assert(kThreads == kHC * kGxCols, "k_bwd_gx: one thread per (stream, column)");

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
// 16-byte asynchronous copy global -> shared; src_bytes = 0 fills zeros
// (the source address is not read then).
__device__ __forceinline__ void cp_async16(void *sdst, const void *gsrc, int src_bytes) {
    const uint32_t sa = (uint32_t)__cvta_generic_to_shared(sdst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(sa), "l"(gsrc), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// a_i = sum_k x_k W_ik and sum_k x_k^2 for kProjTok tokens.  Warp w owns the
// weight rows 3w .. 3w+2; lane l the columns 8l .. 8l+7 of each 256-column
// stage.  Tokens past n are zero-filled and not written.
__global__ void __launch_bounds__(kThreads, 2)
k_bwd_proj(const uint16_t *__restrict__ x, const float *__restrict__ hc_fn, int64_t n, int K,
           float *__restrict__ ws) {
    constexpr int kChunks = kProjTok * kProjCols / 8;  // 16-byte chunks per stage
    __shared__ __align__(16) uint4 sx[kProjStages][kChunks];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t0 = (int64_t)blockIdx.x * kProjTok;
    const int nst = K / kProjCols;
    auto issue = [&](int st) {
        if (st < nst) {
            uint4 *dst = sx[st % kProjStages];
            for (int q = threadIdx.x; q < kChunks; q += kThreads) {
                const int tt = q / (kProjCols / 8), kc = q % (kProjCols / 8);
                const bool ok = t0 + tt < n;
                const uint16_t *src = ok ? x + (t0 + tt) * K + (int64_t)st * kProjCols + kc * 8 : x;
                cp_async16(dst + q, src, ok ? 16 : 0);
            }
        }
        cp_async_commit();  // an empty group past the end keeps the count uniform
    };
    float acc[kProjTok][3], ss[2] = {0.0f, 0.0f};
#pragma unroll
    for (int tt = 0; tt < kProjTok; ++tt)
#pragma unroll
        for (int j = 0; j < 3; ++j) acc[tt][j] = 0.0f;
#pragma unroll
    for (int st = 0; st < kProjStages - 1; ++st) issue(st);
    for (int st = 0; st < nst; ++st) {
        cp_async_wait<kProjStages - 2>();
        __syncthreads();  // stage st landed for every thread; slot (st - 1) is free
        issue(st + kProjStages - 1);
        const uint4 *tile = sx[st % kProjStages];
        float w[3][8];
#pragma unroll
        for (int j = 0; j < 3; ++j)
            load8f(hc_fn + (int64_t)(3 * warp + j) * K + (int64_t)st * kProjCols + lane * 8, w[j]);
#pragma unroll
        for (int tt = 0; tt < kProjTok; ++tt) {
            float xv[8];
            unpack8(tile[tt * (kProjCols / 8) + lane], xv);
#pragma unroll
            for (int j = 0; j < 3; ++j)
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[tt][j] = fmaf(xv[e], w[j][e], acc[tt][j]);
            if ((tt >> 1) == warp)
#pragma unroll
                for (int e = 0; e < 8; ++e) ss[tt & 1] = fmaf(xv[e], xv[e], ss[tt & 1]);
        }
    }
    cp_async_wait<0>();
#pragma unroll
    for (int tt = 0; tt < kProjTok; ++tt)
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const float v = warp_sum(acc[tt][j]);
            if (lane == 0 && t0 + tt < n) ws[(t0 + tt) * kWs + kA + 3 * warp + j] = v;
        }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const float v = warp_sum(ss[q]);
        if (lane == 0 && t0 + 2 * warp + q < n) ws[(t0 + 2 * warp + q) * kWs + kSS] = v;
    }
}

// One token per CTA.  Shared memory: h of the token (d bf16), then the
// Sinkhorn iterates and the reciprocals of their sums (2 * iters matrices of
// 16 each).  Reads a and sum x^2 from the record (k_bwd_proj), writes the
// rest of it.
__global__ void __launch_bounds__(kThreads)
k_bwd_token(const uint16_t *__restrict__ x, const float *__restrict__ pre_mix,
            const uint16_t *__restrict__ f, const float *__restrict__ hc_scale,
            const float *__restrict__ hc_base, const float *__restrict__ norm_w, int d, int iters,
            float eps, float norm_eps, const float *__restrict__ g_hn, const float *__restrict__ g_y,
            const float *__restrict__ g_pre, float *__restrict__ g_pm, float *__restrict__ ws) {
    extern __shared__ uint4 smem_u4[];
    uint4 *sh = smem_u4;                                             // d/8 chunks of h
    float *sP = reinterpret_cast<float *>(smem_u4 + (d >> 3));      // 2*iters*16 iterates
    float *sI = sP + 2 * iters * kHC * kHC;                         // their 1 / (sum + eps)
    __shared__ float red[kWarps][32];
    __shared__ float tot[32];
    __shared__ float sGz[kMix];
    const int64_t t = blockIdx.x;
    const int K = kHC * d, d8 = d >> 3;
    const uint16_t *xt = x + t * K;
    float *wt = ws + t * kWs;
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

    const float rs = rsqrtf(tot[0] / (float)d + norm_eps);
    const float k3 = rs * rs * rs / (float)d * tot[1];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0) {
        // (c) warp 0: the comb part of the split and Sinkhorn, one matrix
        // element per lane (lane & 15 = 4j + k; lanes 16-31 repeat 0-15);
        // the row sums reduce over lanes ^1, ^2, the column sums over ^4, ^8.
        const int e = lane & 15;
        const float r = rsqrtf(wt[kSS] / (float)K + norm_eps);
        const float s2 = __ldg(hc_scale + 2);
        const float L = fmaf(wt[kA + 2 * kHC + e] * r, s2, __ldg(hc_base + 2 * kHC + e));
        float mx = fmaxf(L, __shfl_xor_sync(0xffffffffu, L, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float ex = expf(L - mx);
        float sum = ex + __shfl_xor_sync(0xffffffffu, ex, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        const float S = ex / sum;
        float P = S + eps;
        if (lane < 16) sP[e] = P;
        // steps 1 .. 2*iters-1: a column step for odd, a row step for even
        // steps; sI keeps each step's 1 / (sum + eps)
        for (int st = 1; st < 2 * iters; ++st) {
            const int m1 = (st & 1) ? 4 : 1, m2 = (st & 1) ? 8 : 2;
            float q = P + __shfl_xor_sync(0xffffffffu, P, m1);
            q += __shfl_xor_sync(0xffffffffu, q, m2);
            const float inv = 1.0f / (q + eps);
            P *= inv;
            if (lane < 16) {
                sP[st * 16 + e] = P;
                sI[st * 16 + e] = inv;
            }
        }
        if (lane < 16) wt[kComb + e] = P;
        // back through the steps: g, the gradient of the current iterate
        float g = tot[2 + kHC + e];
        __syncwarp();
        for (int st = 2 * iters - 1; st >= 1; --st) {
            const int m1 = (st & 1) ? 4 : 1, m2 = (st & 1) ? 8 : 2;
            const float pb = sP[st * 16 + e], inv = sI[st * 16 + e];
            float dot = g * pb;
            dot += __shfl_xor_sync(0xffffffffu, dot, m1);
            dot += __shfl_xor_sync(0xffffffffu, dot, m2);
            g = (g - dot) * inv;
        }
        // through the row softmax
        float dot = g * S;
        dot += __shfl_xor_sync(0xffffffffu, dot, 1);
        dot += __shfl_xor_sync(0xffffffffu, dot, 2);
        const float gzc = S * (g - dot);
        if (lane < 16) sGz[2 * kHC + e] = gzc;
        __syncwarp();
        if (lane == 0) {
            // pre and post (sigmoids), then the gradient of the projection
            const float s0 = __ldg(hc_scale), s1 = __ldg(hc_scale + 1);
            float a[kMix], m[kMix], gz[kMix], gm[kMix];
#pragma unroll
            for (int i = 0; i < kMix; ++i) {
                a[i] = wt[kA + i];
                m[i] = a[i] * r;
            }
#pragma unroll
            for (int i = 2 * kHC; i < kMix; ++i) gz[i] = sGz[i];
            float gzm0 = 0.0f, gzm1 = 0.0f, gzm2 = 0.0f;
#pragma unroll
            for (int j = 0; j < kHC; ++j) {
                const float sp = sigm(fmaf(m[j], s0, __ldg(hc_base + j)));
                gz[j] = (g_pre ? __ldg(g_pre + t * kHC + j) : 0.0f) * sp * (1.0f - sp);
                const float sq = sigm(fmaf(m[kHC + j], s1, __ldg(hc_base + kHC + j)));
                gz[kHC + j] = tot[2 + j] * 2.0f * sq * (1.0f - sq);
                wt[kPost + j] = 2.0f * sq;
                wt[kPm + j] = pm[j];
                gm[j] = gz[j] * s0;
                gm[kHC + j] = gz[kHC + j] * s1;
                gzm0 = fmaf(gz[j], m[j], gzm0);
                gzm1 = fmaf(gz[kHC + j], m[kHC + j], gzm1);
            }
#pragma unroll
            for (int i = 2 * kHC; i < kMix; ++i) {
                gm[i] = gz[i] * s2;
                gzm2 = fmaf(gz[i], m[i], gzm2);
            }
            float gr = 0.0f;
#pragma unroll
            for (int i = 0; i < kMix; ++i) gr = fmaf(gm[i], a[i], gr);
#pragma unroll
            for (int i = 0; i < kMix; ++i) {
                wt[kGa + i] = gm[i] * r;
                wt[kGz + i] = gz[i];
            }
            wt[kGzm] = gzm0;
            wt[kGzm + 1] = gzm1;
            wt[kGzm + 2] = gzm2;
            wt[kRs] = rs;
            wt[kCr] = -gr * r * r * r / (float)K;  // the statistic's term: cr * x_k
            wt[kK3] = k3;
        }
    }

    // (d) warps 1-7, beside (c): g_pre_mix_s = sum_c x_s g_h, with
    // g_h = rs w g_hn - k3 h
    {
        float gp[kHC] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (warp != 0) {
            for (int c = threadIdx.x - 32; c < d8; c += kThreads - 32) {
                float h[8], w[8], gh[8], gu[8];
                unpack8(sh[c], h);
                load8f(norm_w + 8 * c, w);
                load8f(g_hn + t * d + 8 * c, gh);
#pragma unroll
                for (int e = 0; e < 8; ++e) gu[e] = rs * (w[e] * gh[e]) - k3 * h[e];
#pragma unroll
                for (int s = 0; s < kHC; ++s) {
                    float xv[8];
                    unpack8(__ldg(reinterpret_cast<const uint4 *>(xt + s * d) + c), xv);
#pragma unroll
                    for (int e = 0; e < 8; ++e) gp[s] = fmaf(xv[e], gu[e], gp[s]);
                }
            }
        }
        block_sums<kHC>(gp, red, tot);
        if (threadIdx.x < kHC) g_pm[t * kHC + threadIdx.x] = tot[threadIdx.x];
    }
}

// g_x, g_f and the block's partial sums of the parameter gradients.  Thread
// (s, c): stream s, column c of d; it holds W[i][s*d + c] for the 24 rows and
// sums g_a[t][i] * x[t][s][c] over the block's tokens.  Per token:
//   g_h  = rs_h w_c g_hn - k3 h_c                  (h_c as the forward rounded it)
//   g_x  = pm_s g_h + cr x_s + sum_k comb_sk g_y_k + sum_i g_a_i W_i
//   g_f  = sum_k post_k g_y_k                       (s = 0 only)
//   g_norm_w partial += h_c rs_h g_hn              (s = 0 only)
// The CTAs of column block 0 also sum the block's g_z and gzm (the hc_base
// and hc_scale terms).  Tiles of kGxTile tokens (their x, g_y and g_hn for
// the CTA's columns, and their records) are staged through a kGxStages-deep
// cp.async ring; tokens past the block are zero-filled and skipped.
struct GxStage {
    uint16_t x[kGxTile][kHC][kGxCols];
    float gy[kGxTile][kHC][kGxCols];
    float ghn[kGxTile][kGxCols];
    float rec[kGxTile][kA];
};
constexpr size_t kGxSmem = sizeof(GxStage) * kGxStages;

__global__ void __launch_bounds__(kThreads, 2)
k_bwd_gx(const uint16_t *__restrict__ x, const float *__restrict__ hc_fn,
         const float *__restrict__ norm_w, const float *__restrict__ g_hn,
         const float *__restrict__ g_y, const float *__restrict__ ws, int64_t n, int d,
         float *__restrict__ g_x, float *__restrict__ g_f, float *__restrict__ part_fn,
         float *__restrict__ part_w, float *__restrict__ part_s) {
    extern __shared__ uint4 smem_u4[];
    GxStage *stg = reinterpret_cast<GxStage *>(smem_u4);
    const int s = threadIdx.x / kGxCols;  // warp-uniform
    const int cl = threadIdx.x % kGxCols;
    const int c0 = blockIdx.x * kGxCols;
    const int c = c0 + cl;
    const int64_t K = (int64_t)kHC * d;
    const int64_t col = (int64_t)s * d + c;
    const int64_t t0 = (int64_t)blockIdx.y * kTokBlock;
    const int64_t t1 = (t0 + kTokBlock < n) ? t0 + kTokBlock : n;
    const int ntiles = (int)((t1 - t0 + kGxTile - 1) / kGxTile);
    const bool small = blockIdx.x == 0;
    const int rec4 = (small ? kA : kRec) / 4;  // float4s staged per token record

    auto issue = [&](int it) {
        if (it < ntiles) {
            GxStage &g = stg[it % kGxStages];
            const int64_t tb = t0 + (int64_t)it * kGxTile;
            for (int q = threadIdx.x; q < kGxTile * kHC * (kGxCols / 8); q += kThreads) {
                const int u = q / (kHC * kGxCols / 8), j = (q / (kGxCols / 8)) % kHC, v = q % (kGxCols / 8);
                const bool ok = tb + u < t1;
                cp_async16(&g.x[u][j][8 * v], ok ? x + ((tb + u) * kHC + j) * d + c0 + 8 * v : x, ok ? 16 : 0);
            }
            for (int q = threadIdx.x; q < kGxTile * kHC * (kGxCols / 4); q += kThreads) {
                const int u = q / (kHC * kGxCols / 4), j = (q / (kGxCols / 4)) % kHC, v = q % (kGxCols / 4);
                const bool ok = tb + u < t1;
                cp_async16(&g.gy[u][j][4 * v], ok ? g_y + ((tb + u) * kHC + j) * d + c0 + 4 * v : g_y,
                           ok ? 16 : 0);
            }
            for (int q = threadIdx.x; q < kGxTile * (kGxCols / 4); q += kThreads) {
                const int u = q / (kGxCols / 4), v = q % (kGxCols / 4);
                const bool ok = tb + u < t1;
                cp_async16(&g.ghn[u][4 * v], ok ? g_hn + (tb + u) * d + c0 + 4 * v : g_hn, ok ? 16 : 0);
            }
            for (int q = threadIdx.x; q < kGxTile * rec4; q += kThreads) {
                const int u = q / rec4, v = q % rec4;
                const bool ok = tb + u < t1;
                cp_async16(&g.rec[u][4 * v], ok ? ws + (tb + u) * kWs + 4 * v : ws, ok ? 16 : 0);
            }
        }
        cp_async_commit();
    };

    float W[kMix], gW[kMix];
#pragma unroll
    for (int i = 0; i < kMix; ++i) {
        W[i] = __ldg(hc_fn + i * K + col);
        gW[i] = 0.0f;
    }
    const float wn = __ldg(norm_w + c);
    float gw = 0.0f, sm = 0.0f;
#pragma unroll
    for (int it = 0; it < kGxStages - 1; ++it) issue(it);
    for (int it = 0; it < ntiles; ++it) {
        cp_async_wait<kGxStages - 2>();
        __syncthreads();  // tile it landed for every thread; slot (it - 1) is free
        issue(it + kGxStages - 1);
        const GxStage &g = stg[it % kGxStages];
        const int64_t tb = t0 + (int64_t)it * kGxTile;
        const int cnt = (int)((t1 - tb < kGxTile) ? t1 - tb : kGxTile);
        if (small && threadIdx.x < kMix + 3)
            for (int u = 0; u < cnt; ++u) sm += g.rec[u][kGz + threadIdx.x];
#pragma unroll 4
        for (int u = 0; u < cnt; ++u) {
            const int64_t t = tb + u;
            const float *rec = g.rec[u];
            float xv[kHC], gy[kHC];
#pragma unroll
            for (int j = 0; j < kHC; ++j) {
                xv[j] = bf16lo(g.x[u][j][cl]);
                gy[j] = g.gy[u][j][cl];
            }
            const float ghn = g.ghn[u][cl];
            float h = rec[kPm] * xv[0];
#pragma unroll
            for (int j = 1; j < kHC; ++j) h = fmaf(rec[kPm + j], xv[j], h);
            h = bf16lo(pack_bf16x2(h, 0.0f));  // the forward's bf16 h
            const float rs = rec[kRs];
            const float gh = rs * (wn * ghn) - rec[kK3] * h;
            const float xs = s == 0 ? xv[0] : s == 1 ? xv[1] : s == 2 ? xv[2] : xv[3];
            float gx = fmaf(rec[kPm + s], gh, rec[kCr] * xs);
#pragma unroll
            for (int k = 0; k < kHC; ++k) gx = fmaf(rec[kComb + s * kHC + k], gy[k], gx);
#pragma unroll
            for (int i = 0; i < kMix; ++i) {
                const float ga = rec[kGa + i];
                gx = fmaf(ga, W[i], gx);
                gW[i] = fmaf(ga, xs, gW[i]);
            }
            g_x[(t * kHC + s) * d + c] = gx;
            if (s == 0) {
                gw = fmaf(h * rs, ghn, gw);
                float gf = rec[kPost] * gy[0];
#pragma unroll
                for (int k = 1; k < kHC; ++k) gf = fmaf(rec[kPost + k], gy[k], gf);
                g_f[t * d + c] = gf;
            }
        }
    }
    cp_async_wait<0>();
#pragma unroll
    for (int i = 0; i < kMix; ++i) part_fn[((int64_t)blockIdx.y * kMix + i) * K + col] = gW[i];
    if (s == 0) part_w[(int64_t)blockIdx.y * d + c] = gw;
    if (small && threadIdx.x < kMix + 3) part_s[(int64_t)blockIdx.y * kSmall + threadIdx.x] = sm;
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

// g_hc_base[i] = sum_b part_s[b][i], g_hc_scale[j] = sum_b part_s[b][24 + j],
// blocks in order.
__global__ void k_bwd_small(const float *__restrict__ part_s, int blocks, float *__restrict__ g_base,
                            float *__restrict__ g_scale) {
    const int j = threadIdx.x;
    if (j >= kMix + 3) return;
    float s = 0.0f;
    for (int b = 0; b < blocks; ++b) s += part_s[(int64_t)b * kSmall + j];
    if (j < kMix) g_base[j] = s;
    else g_scale[j - kMix] = s;
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
    return (size_t)(n * bw::kWs + blocks * (kMix * K + d + bw::kSmall)) * sizeof(float);
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
    float *part_s = part_w + (int64_t)blocks * d;
    const size_t smem = (size_t)d * 2 + (size_t)(4 * iters) * kHC * kHC * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(k_bwd_token, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    k_bwd_proj<<<(unsigned)((n + kProjTok - 1) / kProjTok), kThreads, 0, s>>>(x, hc_fn, n, (int)K, ws);
    k_bwd_token<<<(unsigned)n, kThreads, smem, s>>>(x, pre_mix, f, hc_scale, hc_base, norm_w, d, iters,
                                                   eps, norm_eps, g_hn, g_y, g_pre, g_pm, ws);
    if ((e = cudaFuncSetAttribute(k_bwd_gx, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGxSmem)) !=
        cudaSuccess)
        return e;
    k_bwd_gx<<<dim3((unsigned)(d / kGxCols), (unsigned)blocks), kThreads, kGxSmem, s>>>(
        x, hc_fn, norm_w, g_hn, g_y, ws, n, d, g_x, g_f, part_fn, part_w, part_s);
    k_bwd_sum_blocks<<<(unsigned)((kMix * K + 255) / 256), 256, 0, s>>>(part_fn, blocks, kMix * K, g_fn);
    k_bwd_sum_blocks<<<(unsigned)((d + 255) / 256), 256, 0, s>>>(part_w, blocks, d, g_w);
    k_bwd_small<<<1, 32, 0, s>>>(part_s, blocks, g_base, g_scale);
    return cudaGetLastError();
}

}  // namespace hc
