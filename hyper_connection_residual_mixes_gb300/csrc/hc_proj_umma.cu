// hc_proj_umma.cu -- the mix projection a = x hc_fn^T on the fifth-generation
// tensor cores (tcgen05), for GB300.
//
// What it computes: the matrix product inside Block.hc_mixes (DeepSeek-V4.1
// Block page, Code section): for every token t and mix row i,
//   a[t][i] = sum_k x[t][k] hc_fn[i][k],   k over the hc * d flattened streams,
// before the RMS scaling.  x is bf16 (exact as an MMA operand); hc_fn is fp32
// and is carried as three bf16 parts hi + mid + lo (hi = bf16(w), mid =
// bf16(w - hi), lo = bf16(w - hi - mid)), which hold it to about 2^-24
// relative.  Each bf16 x bf16 product is exact in fp32.
//
// How:
//   k_split_w     hc_fn -> the three parts, as one bf16 matrix of N rows
//                 (part p, mix i at row p * MIX + i; rows past 3 * MIX zero).
//   k_proj_umma   each CTA owns a contiguous range of tokens and walks it in
//                 tiles of 128.  A producer thread streams, per 64 columns of
//                 K, the tile's x box (4 TMA loads of 32 rows, 128-byte
//                 swizzle) and the N x 64 box of split weights into a ring of
//                 shared-memory stages.  One thread issues tcgen05.mma
//                 (M = 128 tokens, N split-weight rows, K = 16 per
//                 instruction, both operands K-major from shared memory) into
//                 an fp32 accumulator in tensor memory.  The tensor core's
//                 fp32 accumulation does not round to nearest, so an
//                 accumulator takes only kDrain stages (8 instructions)
//                 before four drain warps read it (tcgen05.ld), add its three
//                 parts and fold it into their running fp32 sums with ordinary
//                 adds; two accumulators alternate so that the MMAs go on
//                 while one is drained.  Lane r of drain warp w holds token
//                 32 w + r of the tile.
//   The forward flavour (a1-a3 for hc_block_step) also has the drain warps
//   read each stage's x rows for the token's sum of squares (one swizzled
//   128-byte row per lane), and at the end of a tile each lane finishes its
//   token: the RMS scale, split + Sinkhorn (Stream combination page,
//   hc_split_sinkhorn), pre / post / comb (and the mixes) out, and post +
//   comb parked at the start of the token's y row for the a4-a6 pass.
// Every wait is bounded; on a timeout the CTA records the error, waits
// (bounded) for its copies and MMAs in flight, frees its tensor memory and
// returns.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "hc_device.cuh"
#include "hc_launch.h"
#include "hc_ptx.cuh"

namespace hc {

namespace pu {

constexpr int kM = 128;        // tokens per tile: the MMA's M, one TMEM lane each
constexpr int kBK = 64;        // columns of K per stage (one 128-byte swizzled row of bf16)
constexpr int kGroup = 32;     // rows per x box
constexpr int kStages = 4;
constexpr int kDrain = 2;      // stages per accumulator (4 MMAs each)
constexpr int kThreads = 192;  // warps 0-3 drain, warp 4 loads, warp 5 issues the MMAs

template <int MIX>
struct Cfg {
    static constexpr int kParts = 3 * MIX;                  // split-weight rows that carry data
    static constexpr int kN = (kParts + 15) / 16 * 16;      // the MMA's N (multiple of 16 for M = 128)
    static constexpr int kTmemCols = 2 * kN <= 64 ? 64 : 2 * kN <= 128 ? 128 : 2 * kN <= 256 ? 256 : 512;
    static constexpr int kABytes = kM * kBK * 2;
    static constexpr int kBBytes = kN * kBK * 2;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kSmem = kStages * kStageBytes + 1024;  // + slack for the 1024-byte alignment
    // CTAs per SM the launch aims at: two where their tensor memory and shared
    // memory fit beside each other
    static constexpr int kCtasPerSm = (kTmemCols <= 256 && 2 * kSmem <= 227 * 1024) ? 2 : 1;
    static_assert(kN <= 256, "the split weights must fit one MMA");
    static_assert(kStageBytes % 1024 == 0, "stages keep the 1024-byte alignment of the 128-byte swizzle");
};

// Shared-memory matrix descriptor of a K-major bf16 operand written by TMA
// with the 128-byte swizzle: rows of 128 bytes, 8-row groups 1024 bytes apart.
// A K step of 16 elements is a start address 32 bytes further on.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor of kind::f16: bf16 A and B, both K-major, fp32 D, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}
// D (tensor memory) (+)= A (shared memory) x B (shared memory), one thread.
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// One arrival on `bar` once every tcgen05.mma this thread issued before it has
// completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
// Eight columns of this lane at each of three column offsets, waited for in the
// same asm statement (no register copy can slip between the load and the wait).
__device__ __forceinline__ void tmem_ld8x3(uint32_t t0, uint32_t t1, uint32_t t2, uint32_t (&v)[24]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%24];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8, %9, %10, %11, %12, %13, %14, %15}, [%25];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16, %17, %18, %19, %20, %21, %22, %23}, [%26];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
          "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
          "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
          "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23])
        : "r"(t0), "r"(t1), "r"(t2)
        : "memory");
}

// hc_fn [MIX][K] fp32 -> wsplit [kN][K] bf16: row p * MIX + i holds part p of
// row i; rows from 3 * MIX on are zero.
template <int MIX>
__global__ void k_split_w(const float *__restrict__ hc_fn, int64_t K, uint16_t *__restrict__ wsplit) {
    using C = Cfg<MIX>;
    const int64_t total = (int64_t)C::kN * K;
    for (int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < (int64_t)MIX * K;
         o += (int64_t)gridDim.x * blockDim.x) {
        const float w = __ldg(hc_fn + o);
        const uint32_t h = pack_bf16x2(w, 0.0f) & 0xffffu;
        const float r1 = w - bf16lo(h);
        const uint32_t m = pack_bf16x2(r1, 0.0f) & 0xffffu;
        const float r2 = r1 - bf16lo(m);
        const uint32_t l = pack_bf16x2(r2, 0.0f) & 0xffffu;
        wsplit[o] = (uint16_t)h;
        wsplit[(int64_t)MIX * K + o] = (uint16_t)m;
        wsplit[(int64_t)2 * MIX * K + o] = (uint16_t)l;
    }
    for (int64_t o = (int64_t)C::kParts * K + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; o < total;
         o += (int64_t)gridDim.x * blockDim.x)
        wsplit[o] = 0;
}

// Bounded wait that ignores the CTA's abort flag: used on the way out, for
// copies and MMAs already issued, which must land before the CTA leaves.
__device__ __forceinline__ void mbar_wait_exit(uint32_t bar, uint32_t parity) {
    for (uint32_t i = 0; i < (1u << 22); ++i) {
        if (mbar_try_wait(bar, parity)) return;
        __nanosleep(128);
    }
    atomicOr(&g_device_error, kErrWaitTimeout);
}

// What the forward flavour needs beyond the projection.
struct FwdArgs {
    const float *hc_scale, *hc_base;
    int iters;
    float eps, norm_eps;
    float *pre_out, *post_out, *comb_out, *mixes_out;  // each may be null
    float *coef_rows;                                 // post, comb at the start of row t (stride K / 2 floats)
    int part_off;                                     // K split: partial sums at this float of row t
    int64_t part_stride;                              // K split, raw output: floats between slices
};

constexpr int hc_of_mix(int mix) { return mix == 8 ? 2 : mix == 24 ? 4 : 8; }

template <int MIX, bool kFwd>
__global__ void __launch_bounds__(kThreads, 1)
k_proj_umma(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w, int64_t n,
            int K, int rows_per_cta, float *__restrict__ out, int out_stride, FwdArgs fa) {
    using C = Cfg<MIX>;
    constexpr int HC = hc_of_mix(MIX);
    static_assert((2 + HC) * HC == MIX, "mix rows of a stream count");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    __shared__ __align__(8) uint64_t full_bar[kStages];
    __shared__ __align__(8) uint64_t empty_bar[kStages];
    __shared__ __align__(8) uint64_t acc_full[2];
    __shared__ __align__(8) uint64_t acc_empty[2];
    __shared__ __align__(8) uint64_t done_bar;
    __shared__ uint32_t s_tmem;
    __shared__ volatile int s_abort;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r0 = (int64_t)blockIdx.x * rows_per_cta;
    const int64_t r1 = (r0 + rows_per_cta < n) ? r0 + rows_per_cta : n;
    const int ntiles = r1 > r0 ? (int)((r1 - r0 + kM - 1) / kM) : 0;
    // this CTA's slice of K: stages [kb_lo, kb_lo + nkb) of the row (all of it
    // unless the launch splits K over gridDim.y CTAs)
    const int nkb_all = (K + kBK - 1) / kBK;
    const int kb_lo = (int)((int64_t)blockIdx.y * nkb_all / gridDim.y);
    const int nkb = (int)((int64_t)(blockIdx.y + 1) * nkb_all / gridDim.y) - kb_lo;
    const int nch = (nkb + kDrain - 1) / kDrain;  // accumulator chunks per tile

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full_bar[s]), 1);
            mbar_init(smem_u32(&empty_bar[s]), kFwd ? 5 : 1);  // the MMAs (+ the four drain warps)
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&acc_full[b]), 1);
            mbar_init(smem_u32(&acc_empty[b]), 4);
        }
        mbar_init(smem_u32(&done_bar), 1);
        s_abort = 0;
        fence_mbar_init_cluster();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&s_tmem), C::kTmemCols);
        tmem_relinquish();
    }
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    const uint32_t tbase = s_tmem;

    if (warp == 4) {
        if (lane == 0) {
            prefetch_tmap(&tm_x);
            prefetch_tmap(&tm_w);
            const uint64_t pol_x = policy_evict_first(), pol_w = policy_evict_last();
            int it = 0;
            for (int tile = 0; tile < ntiles && !s_abort; ++tile) {
                const int64_t tr = r0 + (int64_t)tile * kM;
                const int64_t left = (r1 - tr + kGroup - 1) / kGroup;  // 32-row boxes of this CTA's rows
                const int groups = left < kM / kGroup ? (int)left : kM / kGroup;
                for (int kb = 0; kb < nkb; ++kb, ++it) {
                    const int slot = it % kStages;
                    if (!mbar_wait<false>(smem_u32(&empty_bar[slot]), ((uint32_t)(it / kStages) & 1u) ^ 1u,
                                          &s_abort))
                        break;
                    const uint32_t st = sbase + (uint32_t)slot * C::kStageBytes;
                    const uint32_t bar = smem_u32(&full_bar[slot]);
                    mbar_arrive_expect_tx(bar, (uint32_t)(groups * kGroup * kBK * 2 + C::kBBytes));
                    for (int g = 0; g < groups; ++g)
                        tma_load_2d(st + (uint32_t)(g * kGroup * kBK * 2), &tm_x, bar, (kb_lo + kb) * kBK,
                                    (int)(tr + g * kGroup), pol_x);
                    tma_load_2d(st + C::kABytes, &tm_w, bar, (kb_lo + kb) * kBK, 0, pol_w);
                }
            }
            // the last stages issued must land before the CTA leaves
            for (int k = (it > kStages ? it - kStages : 0); k < it; ++k)
                mbar_wait_exit(smem_u32(&full_bar[k % kStages]), (uint32_t)(k / kStages) & 1u);
        }
    } else if (warp == 5) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(kM, C::kN);
            int it = 0, c = 0;
            bool ok = true;
            for (int tile = 0; tile < ntiles && ok; ++tile)
                for (int ch = 0; ch < nch && ok; ++ch, ++c) {
                    const int b = c & 1;
                    if (!(ok = mbar_wait<false>(smem_u32(&acc_empty[b]), ((uint32_t)(c >> 1) & 1u) ^ 1u,
                                                &s_abort)))
                        break;
                    tmem_fence_after_sync();
                    const uint32_t d = tbase + (uint32_t)(b * C::kN);
                    const int kb1 = (ch + 1) * kDrain < nkb ? (ch + 1) * kDrain : nkb;
                    for (int kb = ch * kDrain; kb < kb1; ++kb, ++it) {
                        const int slot = it % kStages;
                        if (!(ok = mbar_wait<false>(smem_u32(&full_bar[slot]), (uint32_t)(it / kStages) & 1u,
                                                    &s_abort)))
                            break;
                        tmem_fence_after_sync();
                        const uint32_t st = sbase + (uint32_t)slot * C::kStageBytes;
#pragma unroll
                        for (int ks = 0; ks < kBK / 16; ++ks)
                            umma_ss(d, desc_sw128(st + (uint32_t)(ks * 32)),
                                    desc_sw128(st + C::kABytes + (uint32_t)(ks * 32)), idesc,
                                    (kb > ch * kDrain || ks > 0) ? 1u : 0u);
                        umma_commit(smem_u32(&empty_bar[slot]));
                    }
                    if (ok) umma_commit(smem_u32(&acc_full[b]));
                }
            // every MMA issued has completed before the tensor memory is freed
            umma_commit(smem_u32(&done_bar));
            mbar_wait_exit(smem_u32(&done_bar), 0u);
        }
    } else {
        // drain warps: lane r of warp w holds token 32 w + r of the tile
        const uint32_t lane_base = tbase + ((uint32_t)(32 * warp) << 16);
        float run[MIX];
        int c = 0, it = 0;
        for (int tile = 0; tile < ntiles; ++tile) {
#pragma unroll
            for (int i = 0; i < MIX; ++i) run[i] = 0.0f;
            float ssx = 0.0f;
            bool ok = true;
            for (int ch = 0; ch < nch; ++ch, ++c) {
                if constexpr (kFwd) {
                    // this lane's x row of each stage of the chunk: 8 chunks of 16 bytes,
                    // chunk j at position j ^ (row & 7) (the 128-byte swizzle)
                    const int r = 32 * warp + lane;
                    const int kb1 = (ch + 1) * kDrain < nkb ? (ch + 1) * kDrain : nkb;
                    for (int kb = ch * kDrain; kb < kb1 && ok; ++kb, ++it) {
                        const int slot = it % kStages;
                        if (!(ok = mbar_wait_warp<false>(smem_u32(&full_bar[slot]), (uint32_t)(it / kStages) & 1u,
                                                         &s_abort)))
                            break;
                        const uint8_t *row = smem_raw + (sbase - smem_u32(smem_raw)) + slot * C::kStageBytes + r * 128;
                        f32x2 acc2 = f2_dup(0.0f);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const uint4 v = *reinterpret_cast<const uint4 *>(row + ((j ^ (r & 7)) << 4));
                            const f32x2 a = f2_from_bf16x2(v.x), b2 = f2_from_bf16x2(v.y);
                            const f32x2 c2 = f2_from_bf16x2(v.z), d2 = f2_from_bf16x2(v.w);
                            acc2 = f2_fma(a, a, acc2);
                            acc2 = f2_fma(b2, b2, acc2);
                            acc2 = f2_fma(c2, c2, acc2);
                            acc2 = f2_fma(d2, d2, acc2);
                        }
                        ssx += f2_hsum(acc2);
                        // the loaded values are used before the slot is handed back
                        asm volatile("" ::"f"(ssx));
                        __threadfence_block();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&empty_bar[slot]));
                    }
                    if (!ok) break;
                }
                const int b = c & 1;
                if (!(ok = mbar_wait_warp<false>(smem_u32(&acc_full[b]), (uint32_t)(c >> 1) & 1u, &s_abort)))
                    break;
                tmem_fence_after_sync();
                const uint32_t ta = lane_base + (uint32_t)(b * C::kN);
#pragma unroll
                for (int i0 = 0; i0 < MIX; i0 += 8) {
                    uint32_t v[24];
                    tmem_ld8x3(ta + (uint32_t)i0, ta + (uint32_t)(MIX + i0), ta + (uint32_t)(2 * MIX + i0), v);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        run[i0 + e] += (__uint_as_float(v[16 + e]) + __uint_as_float(v[8 + e])) +
                                       __uint_as_float(v[e]);
                }
                tmem_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&acc_empty[b]));
            }
            if (!ok) break;
            const int64_t row = r0 + (int64_t)tile * kM + 32 * warp + lane;
            if (kFwd && gridDim.y > 1) {
                // K split over CTAs: this slice's dots and sum of squares, summed and
                // finished by k_mix_finish; at float fa.part_off of the token's y row
                if (row < r1) {
                    float *o = fa.coef_rows + row * (int64_t)(K / 2) + fa.part_off + blockIdx.y * (MIX + 1);
#pragma unroll
                    for (int i = 0; i < MIX; ++i) o[i] = run[i];
                    o[MIX] = ssx;
                }
            } else if constexpr (!kFwd) {
                if (row < r1) {
                    // with K split over gridDim.y CTAs, slice blockIdx.y's partial sums go
                    // to the slice's own array (fa.part_stride floats apart)
                    float *o = out + (int64_t)blockIdx.y * fa.part_stride + row * (int64_t)out_stride;
#pragma unroll
                    for (int i = 0; i < MIX; ++i) o[i] = run[i];
                }
            } else if (row < r1) {
                const float rsx = rsqrtf(ssx / (float)K + fa.norm_eps);
#pragma unroll
                for (int i = 0; i < MIX; ++i) run[i] *= rsx;
                float pr[HC], po[HC], cm[HC * HC];
                split_sinkhorn_token_hc<HC>(run, __ldg(fa.hc_scale), __ldg(fa.hc_scale + 1), __ldg(fa.hc_scale + 2),
                                            fa.hc_base, fa.iters, fa.eps, pr, po, cm);
#pragma unroll
                for (int k = 0; k < HC; ++k) {
                    if (fa.pre_out) fa.pre_out[row * HC + k] = pr[k];
                    if (fa.post_out) fa.post_out[row * HC + k] = po[k];
                }
                if (fa.comb_out) {
#pragma unroll
                    for (int i = 0; i < HC * HC; ++i) fa.comb_out[row * HC * HC + i] = cm[i];
                }
                if (fa.mixes_out) {
#pragma unroll
                    for (int i = 0; i < MIX; ++i) fa.mixes_out[row * MIX + i] = run[i];
                }
                if (fa.coef_rows) {
                    float *dst = fa.coef_rows + row * (int64_t)(K / 2);
#pragma unroll
                    for (int k = 0; k < HC; ++k) dst[k] = po[k];
#pragma unroll
                    for (int i = 0; i < HC * HC; ++i) dst[HC + i] = cm[i];
                }
            }
        }
    }
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    if (warp == 0) tmem_dealloc(tbase, C::kTmemCols);
}

// The K-split forward's last step, one warp per token: the slices' dots and
// sums of squares added in slice order, the RMS scale, then split + Sinkhorn
// with the same formulas as split_sinkhorn_token_hc (accurate flavour), the
// comb matrix spread over the lanes (element e = lane + 32 q; at HC*HC < 32
// the lanes repeat it): row sums over lanes ^1 .. ^HC/2, column sums over
// ^HC .. ^16 and the lane's elements.  Mix row i = lane + 32 u.
template <int HC>
__device__ __forceinline__ float wrow_sum(float v) {
#pragma unroll
    for (int m = 1; m < HC; m <<= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}
template <int HC>
__device__ __forceinline__ float wrow_max(float v) {
#pragma unroll
    for (int m = 1; m < HC; m <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
    return v;
}
template <int HC>
__device__ __forceinline__ float wcol_sum(float v) {
#pragma unroll
    for (int m = HC; m < 32 && m < HC * HC; m <<= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
    return v;
}

template <int HC>
__global__ void __launch_bounds__(128)
k_mix_finish(int64_t n, int K, int ksplit, FwdArgs fa) {
    constexpr int MIX = (2 + HC) * HC, H2 = HC * HC;
    constexpr int EPL = H2 > 32 ? H2 / 32 : 1, MPL = (MIX + 31) / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t row = (int64_t)blockIdx.x * 4 + warp;
    if (row >= n) return;  // warp-uniform
    float *rowp = fa.coef_rows + row * (int64_t)(K / 2);
    float mv[MPL];
#pragma unroll
    for (int u = 0; u < MPL; ++u) {
        const int i = lane + 32 * u;
        float acc = 0.0f;
        if (i < MIX)
            for (int ks = 0; ks < ksplit; ++ks) acc += rowp[fa.part_off + ks * (MIX + 1) + i];
        mv[u] = acc;
    }
    float ssx = 0.0f;
    for (int ks = 0; ks < ksplit; ++ks) ssx += rowp[fa.part_off + ks * (MIX + 1) + MIX];
    const float rsx = rsqrtf(ssx / (float)K + fa.norm_eps);
    const float s0 = __ldg(fa.hc_scale), s1 = __ldg(fa.hc_scale + 1), s2 = __ldg(fa.hc_scale + 2);
#pragma unroll
    for (int u = 0; u < MPL; ++u) {
        const int i = lane + 32 * u;
        mv[u] *= rsx;
        if (i >= MIX) continue;
        if (fa.mixes_out) fa.mixes_out[row * MIX + i] = mv[u];
        if (i < HC) {
            const float pr = sigmoid<false>(fmaf(mv[u], s0, __ldg(fa.hc_base + i))) + fa.eps;
            if (fa.pre_out) fa.pre_out[row * HC + i] = pr;
        } else if (i < 2 * HC) {
            const float po = 2.0f * sigmoid<false>(fmaf(mv[u], s1, __ldg(fa.hc_base + i)));
            if (fa.post_out) fa.post_out[row * HC + i - HC] = po;
        }
    }
    // comb logits: element e is mix 2HC + e, held by lane (2HC + e) % 32 in slot (2HC + e) / 32
    float c[EPL];
    int el[EPL];
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
        el[q] = (lane + 32 * q) % H2;
        const int src = 2 * HC + el[q];
        float v = 0.0f;
#pragma unroll
        for (int u = 0; u < MPL; ++u) {
            const float t = __shfl_sync(0xffffffffu, mv[u], src & 31);
            if ((src >> 5) == u) v = t;
        }
        c[q] = fmaf(v, s2, __ldg(fa.hc_base + src));
    }
    // first round: row softmax + eps, then columns; then (iters - 1) rounds of rows, columns
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
        const float ex = expo<false>(c[q] - wrow_max<HC>(c[q]));
        c[q] = fmaf(ex, recip<false>(wrow_sum<HC>(ex)), fa.eps);
    }
    for (int it = 0; it < fa.iters; ++it) {
        if (it > 0) {
#pragma unroll
            for (int q = 0; q < EPL; ++q) c[q] *= recip<false>(wrow_sum<HC>(c[q]) + fa.eps);
        }
        float cs = 0.0f;
#pragma unroll
        for (int q = 0; q < EPL; ++q) cs += wcol_sum<HC>(c[q]);
        const float r = recip<false>(cs + fa.eps);
#pragma unroll
        for (int q = 0; q < EPL; ++q) c[q] *= r;
    }
    // post and comb at the start of the token's y row for the a4-a6 pass (the
    // slices' partial sums sit further along the row)
#pragma unroll
    for (int u = 0; u < MPL; ++u) {
        const int i = lane + 32 * u;
        if (i >= HC && i < 2 * HC) rowp[i - HC] = 2.0f * sigmoid<false>(fmaf(mv[u], s1, __ldg(fa.hc_base + i)));
    }
#pragma unroll
    for (int q = 0; q < EPL; ++q)
        if (lane + 32 * q < H2) {
            if (fa.comb_out) fa.comb_out[row * H2 + el[q]] = c[q];
            rowp[HC + el[q]] = c[q];
        }
}

// The raw projection with K split: out[t][i] = sum over the slices, in order.
__global__ void k_proj_sum_slices(const float *__restrict__ part, int64_t n, int mix, int ksplit,
                                  int64_t part_stride, float *__restrict__ out, int out_stride) {
    const int64_t o = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (o >= n * mix) return;
    const int64_t t = o / mix;
    const int i = (int)(o % mix);
    float v = 0.0f;
    for (int ks = 0; ks < ksplit; ++ks) v += part[(int64_t)ks * part_stride + t * mix + i];
    out[t * out_stride + i] = v;
}

static_assert(Cfg<24>::kCtasPerSm == 2 && Cfg<8>::kCtasPerSm == 2 && Cfg<80>::kCtasPerSm == 1,
              "occupancy the launcher assumes");

}  // namespace pu

namespace {

PFN_cuTensorMapEncodeTiled_v12000 proj_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        cudaDriverEntryPointQueryResult q;
        void *f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// rows x cols bf16 (row stride cols), box of box_rows x 64 columns, 128-byte swizzle
bool proj_tmap(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int box_rows) {
    auto enc = proj_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)pu::kBK, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    static int count[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!count[dev] && cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        count[dev] = 148;
    return count[dev];
}

template <int MIX, bool kFwd>
cudaError_t proj_umma_impl(const uint16_t *x, const float *hc_fn, int64_t n, int64_t K, uint16_t *wsplit,
                           float *out, int out_stride, pu::FwdArgs fa, cudaStream_t s, float *scratch = nullptr,
                           int64_t scratch_floats = 0) {
    using C = pu::Cfg<MIX>;
    {
        const int64_t blocks = ((int64_t)MIX * K + 255) / 256;
        pu::k_split_w<MIX><<<(unsigned)(blocks < 1024 ? blocks : 1024), 256, 0, s>>>(hc_fn, K, wsplit);
    }
    CUtensorMap tmx, tmw;
    if (!proj_tmap(&tmx, x, n, K, pu::kGroup) || !proj_tmap(&tmw, wsplit, C::kN, K, C::kN))
        return cudaErrorInvalidValue;
    // Contiguous token ranges of whole 32-row boxes, about one range per CTA
    // slot.  In the forward, when there are fewer 128-token tiles than slots,
    // each tile's K is split over several CTAs instead (full tiles: no MMA rows
    // wasted, the split weights streamed once per tile), with partial sums in
    // the token's y row, as long as they fit there, and k_mix_finish after.
    const int64_t slots = (int64_t)sm_count() * C::kCtasPerSm;
    const int64_t tiles = (n + pu::kM - 1) / pu::kM;
    // (the raw projection of the backward: slices into the caller's scratch,
    // added by k_proj_sum_slices)
    int ksplit = 1;
    if (tiles < slots && (kFwd || scratch)) {
        const int64_t nkb_all = (K + pu::kBK - 1) / pu::kBK;
        int64_t cand = slots / tiles;
        if (cand > nkb_all / 8) cand = nkb_all / 8;  // at least 8 stages per slice
        if (cand > 8) cand = 8;
        if (kFwd)
            while (cand > 1 && fa.part_off + cand * (MIX + 1) > K / 2) --cand;
        else
            while (cand > 1 && cand * n * MIX > scratch_floats) --cand;
        ksplit = cand > 1 ? (int)cand : 1;
    }
    float *const final_out = out;
    const int final_stride = out_stride;
    if (!kFwd && ksplit > 1) {
        out = scratch;
        out_stride = MIX;
        fa.part_stride = n * MIX;
    }
    int64_t per;
    if (ksplit > 1) {
        per = pu::kM;
    } else {
        per = (n + slots - 1) / slots;
        per = (per + pu::kGroup - 1) / pu::kGroup * pu::kGroup;
    }
    const int64_t grid = (n + per - 1) / per;
    cudaError_t e = cudaFuncSetAttribute(pu::k_proj_umma<MIX, kFwd>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kSmem);
    if (e != cudaSuccess) return e;
    pu::k_proj_umma<MIX, kFwd><<<dim3((unsigned)grid, (unsigned)ksplit), pu::kThreads, C::kSmem, s>>>(
        tmx, tmw, n, (int)K, (int)per, out, out_stride, fa);
    if (ksplit > 1) {
        if (kFwd)
            pu::k_mix_finish<pu::hc_of_mix(MIX)><<<(unsigned)((n + 3) / 4), 128, 0, s>>>(n, (int)K, ksplit, fa);
        else
            pu::k_proj_sum_slices<<<(unsigned)((n * MIX + 255) / 256), 256, 0, s>>>(
                scratch, n, MIX, ksplit, fa.part_stride, final_out, final_stride);
    }
    return cudaGetLastError();
}

}  // namespace

size_t proj_umma_wsplit_bytes(int hc, int64_t K) {
    const int mix = (2 + hc) * hc;
    const int nrows = (3 * mix + 15) / 16 * 16;
    return (size_t)nrows * (size_t)K * 2;
}

cudaError_t launch_proj_umma(const uint16_t *x, const float *hc_fn, int64_t n, int hc, int d, uint16_t *wsplit,
                             float *out, int out_stride, cudaStream_t s, float *scratch, int64_t scratch_floats) {
    const int64_t K = (int64_t)hc * d;
    const pu::FwdArgs none{};
    switch (hc) {
        case 2: return proj_umma_impl<8, false>(x, hc_fn, n, K, wsplit, out, out_stride, none, s, scratch, scratch_floats);
        case 4: return proj_umma_impl<24, false>(x, hc_fn, n, K, wsplit, out, out_stride, none, s, scratch, scratch_floats);
        case 8: return proj_umma_impl<80, false>(x, hc_fn, n, K, wsplit, out, out_stride, none, s, scratch, scratch_floats);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_mixes_umma(const uint16_t *x, const float *hc_fn, const float *hc_scale, const float *hc_base,
                              int64_t n, int hc, int d, int iters, float eps, float norm_eps, uint16_t *wsplit,
                              float *pre_out, float *post_out, float *comb_out, float *mixes_out,
                              uint16_t *coef_rows, cudaStream_t s) {
    const int64_t K = (int64_t)hc * d;
    const pu::FwdArgs fa{hc_scale, hc_base, iters, eps, norm_eps, pre_out, post_out, comb_out, mixes_out,
                         reinterpret_cast<float *>(coef_rows), 128, 0};
    switch (hc) {
        case 2: return proj_umma_impl<8, true>(x, hc_fn, n, K, wsplit, nullptr, 0, fa, s);
        case 4: return proj_umma_impl<24, true>(x, hc_fn, n, K, wsplit, nullptr, 0, fa, s);
        case 8: return proj_umma_impl<80, true>(x, hc_fn, n, K, wsplit, nullptr, 0, fa, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t consume_proj_device_error(cudaStream_t s, unsigned int *flag) {
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    unsigned int v = 0;
    e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof v);
    if (e != cudaSuccess) return e;
    *flag = v;
    if (v) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
    }
    return e;
}

}  // namespace hc
