// hc_chain.cu -- the hyper-connection side steps of a chain of sides, fused
// across sides, for GB300.
//
// What it computes: per side, the same path as hc_block_step (DeepSeek-V4.1
// Block page, Code section: Block.hc_mixes, Block.hc_pre, Block.hc_post;
// "Stream combination" page: hc_split_sinkhorn), for the chain the page's
// Block.forward builds: the streams a side reads are the y the previous side
// wrote, and each side reads its sublayer input with the previous side's pre.
//
// How: one launch per side.  It runs phase 3 of side i (y and h_norm, from the
// state of side i that the previous launch computed) and, on the y it has just
// written into shared memory, phase 1 of side i+1 (the projection with side
// i+1's weights on the tensor cores, the sum of squares of y, and the sum of
// squares of side i+1's bf16 h), then the cross-CTA reduction and the split +
// Sinkhorn of side i+1, whose results form the state of side i+1.  Each side's
// streams are read from HBM once; y and h_norm leave through TMA stores from
// the place where the CUDA-core warps wrote them.  Cluster layout, tensor-
// memory weights and the owner reduction are those of hc_block_cluster.cu,
// with the same per-thread columns and summation order, so every output equals
// bit for bit what hc_block_step computes side by side.
//
// Modes: kBegin (phase 1 of the first side, from its x), kSide (phase 3 of side
// i + phase 1 of side i+1), kLast (phase 3 of the last side only).
//
// State row per token (kStateF = 32 fp32): post[4], comb[16], rs_h, 3 pad,
// pre[4] (the side's pre = the next side's pre_mix), pre_mix[4] (the pre_mix
// the side reads its sublayer input with).
//
// Warp roles (512 threads): warps 0-3 tensor-core MMA (warp w: stream w, TMEM
// quadrant w); warp 4 TMA producer; warp 5 owner-side reduction + Sinkhorn;
// warps 6-13 CUDA-core math; warp 14 sends each tile's partial sums to the
// owners; warp 15 TMA stores of y and h_norm.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "hc_device.cuh"
#include "hc_launch.h"
#include "hc_ptx.cuh"

namespace hc {

namespace ch {

constexpr int kC = 16;           // CTAs per cluster = column slices of d
constexpr int kT = 64;           // tokens per tile
constexpr int kCB = 64;          // columns per slot per stream (128-byte box rows)
constexpr int kItems = 2;        // 8-column items per CUDA-core thread per slot
constexpr int kStepsPerSlot = kCB / 16;
constexpr int kSlots = 4;        // TMA ring depth (40 KB per slot)
// Tiles in flight between the CUDA-core warps and the owners: the partial-sum
// buffers at the owners and the sum-of-squares buffers rotate over kBufs, and
// the CUDA-core warps start tile j once the owners are done with tile j - kBufs.
// The owners' reduction + Sinkhorn latency sits in that loop; with two tiles the
// loop had no slack (measured: the launch time tracked the Sinkhorn rounds).
constexpr int kBufs = 3;
constexpr uint32_t kTmemCols = 512;
constexpr int kThreads = 512;
constexpr int kBoxBytes = kT * kCB * 2;                // 8 KB
constexpr int kStageXBytes = kHC * kBoxBytes;          // 32 KB
constexpr int kSlotBytes = kStageXBytes + kBoxBytes;   // + f box = 40 KB
constexpr int kTokPerOwner = kT / kC;                  // 4
constexpr int kPartF = 28;       // 24 partial dots, sum x^2, sum h^2, 2 pad
constexpr int kStateF = 32;      // floats per token in a state row
constexpr int kWarpMma = 0;
constexpr int kMmaWarps = 4;
constexpr int kWarpProducer = 4;
constexpr int kWarpReducer = 5;
constexpr int kWarpCuda = 6;     // warps 6..13
constexpr int kCudaWarps = 8;
constexpr int kWarpSender = 14;
constexpr int kWarpStore = 15;
constexpr int kWCols = 18;       // TMEM columns per k16 step: 3 n-tiles x (hi, mid, lo) x (b0, b1)
constexpr int kBegin = 0, kSide = 1, kLast = 2;
constexpr int kNumBars = 3 * kSlots + 3 * kBufs + 2 + 2;  // full, empty, staged, part, coef, ss, mma, state

struct Params {
    const float *state_in;   // [n, 32]: state of side i (kSide, kLast)
    const float *pre_mix;    // [n, 4]: the first side's pre_mix (kBegin)
    const float *hc_fn;      // weights of the side whose phase 1 runs here
    const float *hc_scale;
    const float *hc_base;
    const float *norm_w;     // [d]: side i's RMSNorm weight (kSide, kLast)
    float *state_out;        // [n, 32]: state of the side whose phase 1 runs here
    float *pre_out;          // [n, 4], optional: that side's pre
    int64_t n;
    int d;
    int iters;
    float eps;
    float norm_eps;
    int num_tiles;
};

// Shared-memory layout (byte offsets from a 1024-aligned base).
struct Layout {
    int dc, ncb, wcols;
    int off_state, off_mma, off_part, off_ss, off_normw, off_bar, off_tmem, total;
};

__host__ __device__ inline Layout make_layout(int d) {
    Layout L;
    L.dc = d / kC;
    L.ncb = L.dc / kCB;
    L.wcols = kWCols * (L.dc / 16);
    int o = kSlots * kSlotBytes;
    L.off_state = o;  // two tiles of state rows (kBegin: of pre_mix rows)
    o += 2 * kT * kStateF * 4;
    L.off_mma = o;
    o += kMmaWarps * kT * kMix * 4;
    L.off_part = o;
    o += kBufs * kC * kTokPerOwner * kPartF * 4;
    L.off_ss = o;
    o += kBufs * kT * 2 * 4;
    L.off_normw = o;
    o += L.dc * 4;
    o = (o + 15) & ~15;
    L.off_bar = o;
    o += kNumBars * 8;
    o = (o + 15) & ~15;
    L.off_tmem = o;
    o += 16;
    L.total = o + 1024;
    return L;
}

__device__ __forceinline__ void split3(float w0, float w1, uint32_t &hi, uint32_t &mid, uint32_t &lo) {
    hi = pack_bf16x2(w0, w1);
    const float r0 = w0 - bf16lo(hi), r1 = w1 - bf16hi(hi);
    mid = pack_bf16x2(r0, r1);
    const float s0 = r0 - bf16lo(mid), s1 = r1 - bf16hi(mid);
    lo = pack_bf16x2(s0, s1);
}

// Byte offset of (row r, 16-byte unit u) in a 64-column box with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(int r, int u) { return (uint32_t)(r * 128 + ((u ^ (r & 7)) << 4)); }

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
k_chain(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_f,
        const __grid_constant__ CUtensorMap tm_y, const __grid_constant__ CUtensorMap tm_h,
        const __grid_constant__ CUtensorMap tm_s, const Params p) {
    constexpr bool kP1 = kMode != kLast;   // phase 1 of a side runs here
    constexpr bool kP3 = kMode != kBegin;  // phase 3 of side i runs here
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    // the ring again, in the shared address space (ld.shared / st.shared)
    uint8_t *smem_ring = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ volatile int s_abort;
    const Layout L = make_layout(p.d);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int cid = (int)cluster_id_x(), ncl = (int)cluster_count_x();
    const int J = (p.num_tiles > cid) ? (p.num_tiles - cid + ncl - 1) / ncl : 0;
    const int ncb = L.ncb, dc = L.dc, d = p.d;
    const int64_t K = (int64_t)kHC * d;
    const int U = J * ncb;  // ring uses, in order: tile by tile, column block by column block

    float *sState = reinterpret_cast<float *>(smem + L.off_state);
    float *sMma = reinterpret_cast<float *>(smem + L.off_mma);
    float *sPart = reinterpret_cast<float *>(smem + L.off_part);
    float *sSS = reinterpret_cast<float *>(smem + L.off_ss);
    float *sNormW = reinterpret_cast<float *>(smem + L.off_normw);
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + L.off_tmem);
    const uint32_t bar0 = smem_u32(smem + L.off_bar);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kSlots + s); };
    // the CUDA-core warps have written y and h_norm over the slot's x and f
    auto staged_bar = [&](int s) { return bar0 + 8u * (2 * kSlots + s); };
    auto part_bar = [&](int b) { return bar0 + 8u * (3 * kSlots + b); };
    // one arrival pair per owner and tile: paces the CUDA-core warps (see there)
    auto coef_bar = [&](int b) { return bar0 + 8u * (3 * kSlots + kBufs + b); };
    const uint32_t mma_full = bar0 + 8u * (3 * kSlots + 2 * kBufs);
    const uint32_t mma_free = bar0 + 8u * (3 * kSlots + 2 * kBufs + 1);
    auto ss_bar = [&](int b) { return bar0 + 8u * (3 * kSlots + 2 * kBufs + 2 + b); };
    // the CUDA-core warps are done with a tile's state rows (buffer b)
    auto state_free = [&](int b) { return bar0 + 8u * (3 * kSlots + 3 * kBufs + 2 + b); };
    const uint32_t slot0 = smem_u32(smem);

    if (threadIdx.x == kWarpProducer * 32) {
        s_abort = 0;
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(full_bar(s), 1);
            // kBegin: MMA + CUDA-core warps; kSide: MMA warps + the store warp; kLast: the store warp
            mbar_init(empty_bar(s), kMode == kBegin ? kMmaWarps + kCudaWarps : kMode == kSide ? kMmaWarps + 1 : 1);
            mbar_init(staged_bar(s), kCudaWarps);
        }
        for (int b = 0; b < kBufs; ++b) {
            mbar_init(part_bar(b), kC * 4);
            mbar_init(coef_bar(b), kC * 2);
            mbar_init(ss_bar(b), kT);
        }
        for (int b = 0; b < 2; ++b) mbar_init(state_free(b), kCudaWarps);
        mbar_init(mma_full, kMmaWarps * 32);
        mbar_init(mma_free, 32);
        fence_mbar_init_cluster();
        prefetch_tmap(&tm_x);
        if (kP3) {
            prefetch_tmap(&tm_f);
            prefetch_tmap(&tm_y);
            prefetch_tmap(&tm_h);
            prefetch_tmap(&tm_s);
        }
    }
    if (kP1 && warp == kWarpMma) {
        tmem_alloc(smem_u32(sTmem), kTmemCols);
        tmem_relinquish();
    }
    if (kP3)
        for (int c = threadIdx.x; c < dc; c += kThreads) sNormW[c] = __ldg(p.norm_w + rank * dc + c);
    tmem_fence_before_sync();
    cluster_sync_all();
    tmem_fence_after_sync();
    const uint32_t tmem_base = kP1 ? *sTmem : 0u;

    if (warp < kWarpMma + kMmaWarps) {
        // ------------------------------------------------------------ tensor-core projection
        if (kP1) {
            const int s = warp - kWarpMma;
            const int g = lane >> 2, t = lane & 3;
            // weight fragments in TMEM, as in hc_block_cluster.cu
            const uint32_t tw = tmem_base + ((uint32_t)(32 * (warp & 3)) << 16);
            for (int q = 0; q < dc / 16; ++q) {
                const int64_t col = (int64_t)s * d + (int64_t)rank * dc + 16 * q + 2 * t;
#pragma unroll
                for (int nt = 0; nt < 3; ++nt) {
                    const float *wr = p.hc_fn + (int64_t)(nt * 8 + g) * K + col;
                    const float2 p0 = __ldg(reinterpret_cast<const float2 *>(wr));
                    const float2 p1 = __ldg(reinterpret_cast<const float2 *>(wr + 8));
                    uint32_t h0, m0, l0, h1, m1, l1;
                    split3(p0.x, p0.y, h0, m0, l0);
                    split3(p1.x, p1.y, h1, m1, l1);
                    const uint32_t c0 = tw + kWCols * q + 6 * nt;
                    tmem_st2(c0 + 0, h0, h1);
                    tmem_st2(c0 + 2, m0, m1);
                    tmem_st2(c0 + 4, l0, l1);
                }
            }
            tmem_wait_st();
            float acc[4][3][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 3; ++b)
#pragma unroll
                    for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.0f;
            int tiles_done = 0, cb = 0;
            for (int u = 0; u < U; ++u) {
                const int slot = u % kSlots;
                const uint32_t ph = (uint32_t)(u / kSlots) & 1u;
                // kBegin: the slot holds x; kSide: wait until y has replaced it
                if (!mbar_wait_warp<false>(kMode == kBegin ? full_bar(slot) : staged_bar(slot), ph, &s_abort)) break;
                const uint32_t box = slot0 + slot * kSlotBytes + s * kBoxBytes;
#pragma unroll
                for (int hp = 0; hp < kStepsPerSlot / 2; ++hp) {
                    uint32_t bw[36];
                    tmem_ld36(tw + kWCols * (cb * kStepsPerSlot + 2 * hp), bw);
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int h = 2 * hp + h2;
#pragma unroll
                        for (int mt = 0; mt < 4; ++mt) {
                            const int r = mt * 16 + (lane & 15);
                            uint32_t a0, a1, a2, a3;
                            ldmatrix_x4(box + swz(r, 2 * h + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
                            for (int nt = 0; nt < 3; ++nt) {
                                const uint32_t *b = bw + kWCols * h2 + 6 * nt;
                                mma_bf16_16816(acc[mt][nt], a0, a1, a2, a3, b[4], b[5]);  // lo
                                mma_bf16_16816(acc[mt][nt], a0, a1, a2, a3, b[2], b[3]);  // mid
                                mma_bf16_16816(acc[mt][nt], a0, a1, a2, a3, b[0], b[1]);  // hi
                            }
                        }
                    }
                }
                // the slot's last ldmatrix loads complete before it goes (as in hc_block_cluster.cu)
                __threadfence_block();
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(slot));
                if (++cb == ncb) {
                    cb = 0;
                    if (!mbar_wait_warp<false>(mma_free, ((uint32_t)tiles_done & 1u) ^ 1u, &s_abort)) break;
                    float *mine = sMma + s * kT * kMix;
#pragma unroll
                    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                        for (int nt = 0; nt < 3; ++nt) {
                            const int r = mt * 16 + g, c = nt * 8 + 2 * t;
                            *reinterpret_cast<float2 *>(mine + r * kMix + c) = make_float2(acc[mt][nt][0], acc[mt][nt][1]);
                            *reinterpret_cast<float2 *>(mine + (r + 8) * kMix + c) = make_float2(acc[mt][nt][2], acc[mt][nt][3]);
                            acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.0f;
                        }
                    mbar_arrive(mma_full);
                    ++tiles_done;
                }
            }
        }
    } else if (warp == kWarpProducer) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();  // every byte is read once
            const uint64_t pol_state = policy_evict_normal();  // the 16 CTAs of a cluster read each state row
            int armed = 0, j = 0, cb = 0;
            for (int u = 0; u < U; ++u) {
                const int slot = u % kSlots;
                const uint32_t ph = (uint32_t)(u / kSlots) & 1u;
                if (!mbar_wait<false>(empty_bar(slot), ph ^ 1u, &s_abort)) break;
                const int row = (cid + j * ncl) * kT;
                const int col = (int)rank * dc + cb * kCB;
                const uint32_t dst = slot0 + slot * kSlotBytes;
                // the tile's state rows (kBegin: its pre_mix rows) travel with its first slot,
                // into the buffer the CUDA-core warps released two tiles ago
                uint32_t side_bytes = 0;
                if (cb == 0) {
                    if (j >= 2 &&
                        !mbar_wait<false>(state_free(j & 1), (uint32_t)((j - 2) >> 1) & 1u, &s_abort))
                        break;
                    const int64_t rows_left = p.n - (int64_t)row;
                    const uint32_t rows = (uint32_t)(rows_left < kT ? rows_left : kT);
                    // a TMA box always delivers all its bytes (rows past n read as zero)
                    side_bytes = kMode == kBegin ? 16u * rows : 4u * kStateF * kT;
                }
                mbar_arrive_expect_tx(full_bar(slot), (kP3 ? kSlotBytes : kStageXBytes) + side_bytes);
                if (cb == 0) {
                    const uint32_t sdst = smem_u32(sState) + (j & 1) * kT * kStateF * 4;
                    if (kMode == kBegin)
                        bulk_load(sdst, p.pre_mix + (int64_t)row * kHC, side_bytes, full_bar(slot));
                    else
                        tma_load_2d(sdst, &tm_s, full_bar(slot), 0, row, pol_state);
                }
                for (int s = 0; s < kHC; ++s) tma_load_2d(dst + s * kBoxBytes, &tm_x, full_bar(slot), s * d + col, row, pol);
                if (kP3) tma_load_2d(dst + kStageXBytes, &tm_f, full_bar(slot), col, row, pol);
                armed = u + 1;
                if (++cb == ncb) {
                    cb = 0;
                    ++j;
                }
            }
            for (int u = (armed > kSlots ? armed - kSlots : 0); u < armed; ++u)
                mbar_wait<false>(full_bar(u % kSlots), (uint32_t)(u / kSlots) & 1u, &s_abort);
        }
    } else if (warp == kWarpReducer) {
        // ------------------------------------------------------------ owner: statistics + Sinkhorn
        // As in hc_block_cluster.cu; the results form this side's state rows.
        if (kP1) {
            const float s0 = __ldg(p.hc_scale), s1 = __ldg(p.hc_scale + 1), s2 = __ldg(p.hc_scale + 2);
            const int tl = lane >> 3, sub = lane & 7;
            const int tk = (int)rank * kTokPerOwner + tl;
            // The pre_mix the side reads with (the first side's input, or the previous
            // side's pre, kept in the previous side's state) goes into the state row.  It
            // is read from global memory one tile ahead, so that its latency does not hold
            // up the next tile's reduction.
            auto load_pmx = [&](int jj) {
                const int64_t t = (int64_t)(cid + jj * ncl) * kT + tk;
                if (jj >= J || t >= p.n) return make_float4(0.f, 0.f, 0.f, 0.f);
                return kMode == kBegin ? __ldg(reinterpret_cast<const float4 *>(p.pre_mix) + t)
                                       : __ldg(reinterpret_cast<const float4 *>(p.state_in + t * kStateF + 24));
            };
            float4 pmx_next = load_pmx(0);
            for (int j = 0; j < J; ++j) {
                const float4 pmx = pmx_next;
                pmx_next = load_pmx(j + 1);
                const int buf = j % kBufs;
                if (!mbar_wait_warp<true>(part_bar(buf), (uint32_t)(j / kBufs) & 1u, &s_abort)) break;
                const int tile = cid + j * ncl;
                const int64_t tok = (int64_t)tile * kT + tk;
                float m[kMix + 2];
                {
                    const float *e0 = sPart + ((buf * kC + sub) * kTokPerOwner + tl) * kPartF;
                    const float *e1 = sPart + ((buf * kC + sub + 8) * kTokPerOwner + tl) * kPartF;
#pragma unroll
                    for (int i = 0; i < kMix + 2; ++i) m[i] = e0[i] + e1[i];
                }
#pragma unroll
                for (int i = 0; i < kMix + 2; ++i) {
                    m[i] += __shfl_xor_sync(0xffffffffu, m[i], 1);
                    m[i] += __shfl_xor_sync(0xffffffffu, m[i], 2);
                    m[i] += __shfl_xor_sync(0xffffffffu, m[i], 4);
                }
                const float ssx = m[kMix], ssh = m[kMix + 1];
                const float r = rsqrtf(ssx / (float)K + p.norm_eps);
                float mm[kMix];
#pragma unroll
                for (int i = 0; i < kMix; ++i) mm[i] = m[i] * r;
                float pr[kHC], po[kHC], c[kHC * kHC];
                split_sinkhorn_token<true>(mm, s0, s1, s2, p.hc_base, p.iters, p.eps, pr, po, c);
                const float rs_h = rsqrtf(ssh / (float)d + p.norm_eps);
                // pace the CUDA-core warps of every CTA: they wait for this arrival of
                // tile j before starting tile j + kBufs (lane l -> destination CTA l % 16)
                // the partials read above complete before the senders may overwrite them
                __threadfence_block();
                mbar_arrive_remote(mapa(coef_bar(buf), lane & 15));
                if (sub == 0 && tok < p.n) {
                    float4 *st = reinterpret_cast<float4 *>(p.state_out + tok * kStateF);
                    st[0] = make_float4(po[0], po[1], po[2], po[3]);
#pragma unroll
                    for (int q = 0; q < 4; ++q) st[1 + q] = make_float4(c[4 * q], c[4 * q + 1], c[4 * q + 2], c[4 * q + 3]);
                    st[5] = make_float4(rs_h, 0.f, 0.f, 0.f);
                    st[6] = make_float4(pr[0], pr[1], pr[2], pr[3]);
                    st[7] = pmx;
                    if (p.pre_out) reinterpret_cast<float4 *>(p.pre_out)[tok] = make_float4(pr[0], pr[1], pr[2], pr[3]);
                }
            }
        }
    } else if (warp == kWarpSender) {
        // ------------------------------------------------------------ partial sums -> owners
        if (kP1) {
            for (int j = 0; j < J; ++j) {
                if (!mbar_wait_warp<false>(mma_full, (uint32_t)j & 1u, &s_abort)) break;
                if (!mbar_wait_warp<false>(ss_bar(j % kBufs), (uint32_t)(j / kBufs) & 1u, &s_abort)) break;
                const int buf = j % kBufs;
#pragma unroll
                for (int i2 = 0; i2 < 2; ++i2) {
                    // tokens lane and lane + 32: neighbouring lanes read neighbouring rows
                    const int tk = lane + 32 * i2;
                    const int owner = tk / kTokPerOwner, tl = tk % kTokPerOwner;
                    float v[kPartF];
#pragma unroll
                    for (int i = 0; i < kMix; ++i) v[i] = 0.0f;
#pragma unroll
                    for (int w = 0; w < kMmaWarps; ++w) {
                        const float *e = sMma + (w * kT + tk) * kMix;
#pragma unroll
                        for (int i = 0; i < kMix; ++i) v[i] += e[i];
                    }
                    const float2 ss = *reinterpret_cast<const float2 *>(sSS + ((j % kBufs) * kT + tk) * 2);
                    v[kMix] = ss.x;
                    v[kMix + 1] = ss.y;
                    v[kMix + 2] = v[kMix + 3] = 0.0f;
                    const uint32_t dst = mapa(smem_u32(sPart + ((buf * kC + rank) * kTokPerOwner + tl) * kPartF), owner);
#pragma unroll
                    for (int q = 0; q < kPartF / 4; ++q)
                        st_cluster_v4(dst + 16 * q, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                    mbar_arrive_remote(mapa(part_bar(buf), owner));
                }
                mbar_arrive(mma_free);
            }
        }
    } else if (warp == kWarpStore) {
        // ------------------------------------------------------------ TMA stores of y and h_norm
        if (kP3 && lane == 0) {
            const uint64_t pol = policy_evict_first();
            int j = 0, cb = 0;
            for (int u = 0; u < U; ++u) {
                const int slot = u % kSlots;
                if (!mbar_wait<false>(staged_bar(slot), (uint32_t)(u / kSlots) & 1u, &s_abort)) break;
                const int row = (cid + j * ncl) * kT;
                const int col = (int)rank * dc + cb * kCB;
                const uint32_t src = slot0 + slot * kSlotBytes;
                for (int k = 0; k < kHC; ++k) tma_store_2d(&tm_y, src + k * kBoxBytes, k * d + col, row, pol);
                tma_store_2d(&tm_h, src + kStageXBytes, col, row, pol);
                bulk_commit_group();
                bulk_wait_group_read<0>();  // the slot's bytes are out: it may be refilled
                mbar_arrive(empty_bar(slot));
                if (++cb == ncb) {
                    cb = 0;
                    ++j;
                }
            }
            bulk_wait_group<0>();  // every store has landed before the CTA leaves
        }
    } else {
        // ------------------------------------------------------------ CUDA-core streaming math
        // 256 threads; per slot, thread tc handles token row r and the 8-column
        // units uu + 4i (i < 2), rows and units as in hc_block_cluster.cu.
        const int tc = threadIdx.x - kWarpCuda * 32;
        const int uu = lane & 3;
        const int r = 8 * (tc >> 5) + (lane >> 3) + 4 * ((lane >> 2) & 1);
        int u = 0;
        bool ok = true;
        for (int j = 0; j < J && ok; ++j) {
            if (kP1 && j >= kBufs) {
                // Wait for the owners' signal for tile j - kBufs: every hand-off buffer
                // of that tile (sums of squares here, partials at the owners) has been read.
                const int jw = j - kBufs;
                if (!mbar_wait_warp<true>(coef_bar(jw % kBufs), (uint32_t)(jw / kBufs) & 1u, &s_abort)) break;
            }
            const int64_t tok = (int64_t)(cid + j * ncl) * kT + r;
            const bool live = tok < p.n;
            // this tile's state rows (kSide, kLast: 128-byte rows with the 128-byte swizzle,
            // so the eight rows of a warp read distinct banks; kBegin: pre_mix rows)
            const uint8_t *srow = reinterpret_cast<const uint8_t *>(sState) + (j & 1) * kT * kStateF * 4;
            f32x2 ssx2[kHC], ssh2[kItems];
#pragma unroll
            for (int s = 0; s < kHC; ++s) ssx2[s] = f2_dup(0.0f);
#pragma unroll
            for (int it = 0; it < kItems; ++it) ssh2[it] = f2_dup(0.0f);
            for (int cb = 0; cb < ncb; ++cb, ++u) {
                const int slot = u % kSlots;
                if (!mbar_wait_warp<false>(full_bar(slot), (uint32_t)(u / kSlots) & 1u, &s_abort)) {
                    ok = false;
                    break;
                }
                uint8_t *sb = smem_ring + slot * kSlotBytes;
                uint4 xr[kItems][kHC];
#pragma unroll
                for (int it = 0; it < kItems; ++it)
#pragma unroll
                    for (int s = 0; s < kHC; ++s)
                        xr[it][s] = *reinterpret_cast<const uint4 *>(sb + s * kBoxBytes + swz(r, uu + 4 * it));
                if (kMode == kBegin) {
                    // ---------------- phase 1 of the first side, on x
                    __threadfence_block();  // the loads above complete before the slot goes
                    __syncwarp();
                    if (lane == 0) mbar_arrive(empty_bar(slot));
                    const float4 v = live ? *reinterpret_cast<const float4 *>(sState + (j & 1) * kT * kStateF + r * kHC)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                    const f32x2 pm[kHC] = {f2_dup(v.x), f2_dup(v.y), f2_dup(v.z), f2_dup(v.w)};
#pragma unroll
                    for (int it = 0; it < kItems; ++it) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            f32x2 xs[kHC];
#pragma unroll
                            for (int s = 0; s < kHC; ++s) {
                                const uint4 &w = xr[it][s];
                                xs[s] = f2_from_bf16x2(q == 0 ? w.x : q == 1 ? w.y : q == 2 ? w.z : w.w);
                                ssx2[s] = f2_fma(xs[s], xs[s], ssx2[s]);
                            }
                            f32x2 h = f2_mul(pm[0], xs[0]);
                            h = f2_fma(pm[1], xs[1], h);
                            h = f2_fma(pm[2], xs[2], h);
                            h = f2_fma(pm[3], xs[3], h);
                            const f32x2 hr = f2_from_bf16x2(f2_to_bf16x2(h));
                            ssh2[it] = f2_fma(hr, hr, ssh2[it]);
                        }
                    }
                } else {
                    // ---------------- phase 3 of side i, then phase 1 of side i+1 on its y
                    const uint4 fr0 = *reinterpret_cast<const uint4 *>(sb + kStageXBytes + swz(r, uu));
                    const uint4 fr1 = *reinterpret_cast<const uint4 *>(sb + kStageXBytes + swz(r, uu + 4));
                    if (live) {
                        float cf[kHC + kHC * kHC];  // post, comb: 16-byte chunks 0-4 of the row
#pragma unroll
                        for (int c = 0; c < 5; ++c) {
                            const float4 v = *reinterpret_cast<const float4 *>(srow + swz(r, c));
                            cf[4 * c] = v.x;
                            cf[4 * c + 1] = v.y;
                            cf[4 * c + 2] = v.z;
                            cf[4 * c + 3] = v.w;
                        }
                        const float rs = *reinterpret_cast<const float *>(srow + swz(r, 5));
                        const float4 pmv = *reinterpret_cast<const float4 *>(srow + swz(r, 7));
#pragma unroll
                        for (int it = 0; it < kItems; ++it) {
                            const uint4 &fw = it == 0 ? fr0 : fr1;
                            const int un = uu + 4 * it;
                            const float4 *nw = reinterpret_cast<const float4 *>(sNormW + cb * kCB + un * 8);
                            const float4 w0 = nw[0], w1 = nw[1];
                            const f32x2 wv[4] = {f2_make(w0.x, w0.y), f2_make(w0.z, w0.w), f2_make(w1.x, w1.y),
                                                 f2_make(w1.z, w1.w)};
                            uint32_t yo[kHC][4], ho[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                f32x2 xs[kHC];
#pragma unroll
                                for (int s = 0; s < kHC; ++s) {
                                    const uint4 &w = xr[it][s];
                                    xs[s] = f2_from_bf16x2(q == 0 ? w.x : q == 1 ? w.y : q == 2 ? w.z : w.w);
                                }
                                const f32x2 fv = f2_from_bf16x2(q == 0 ? fw.x : q == 1 ? fw.y : q == 2 ? fw.z : fw.w);
#pragma unroll
                                for (int k = 0; k < kHC; ++k) {
                                    f32x2 a = f2_mul(f2_dup(cf[k]), fv);
#pragma unroll
                                    for (int jj = 0; jj < kHC; ++jj) a = f2_fma(f2_dup(cf[kHC + jj * kHC + k]), xs[jj], a);
                                    yo[k][q] = f2_to_bf16x2(a);
                                }
                                f32x2 h = f2_mul(f2_dup(pmv.x), xs[0]);
                                h = f2_fma(f2_dup(pmv.y), xs[1], h);
                                h = f2_fma(f2_dup(pmv.z), xs[2], h);
                                h = f2_fma(f2_dup(pmv.w), xs[3], h);
                                const f32x2 hr = f2_from_bf16x2(f2_to_bf16x2(h));
                                ho[q] = f2_to_bf16x2(f2_mul(f2_mul(hr, f2_dup(rs)), wv[q]));
                            }
                            // y and h_norm replace, in place, the x and f words this thread alone read
                            uint8_t *wb = sb + swz(r, un);
#pragma unroll
                            for (int k = 0; k < kHC; ++k)
                                *reinterpret_cast<uint4 *>(wb + k * kBoxBytes) = make_uint4(yo[k][0], yo[k][1], yo[k][2], yo[k][3]);
                            *reinterpret_cast<uint4 *>(wb + kStageXBytes) = make_uint4(ho[0], ho[1], ho[2], ho[3]);
                            if (kMode == kSide) {
                                // phase 1 of side i+1 on this y: its x is y, its pre_mix side i's pre
                                const float4 pn = *reinterpret_cast<const float4 *>(srow + swz(r, 6));
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    f32x2 ys[kHC];
#pragma unroll
                                    for (int s = 0; s < kHC; ++s) {
                                        ys[s] = f2_from_bf16x2(yo[s][q]);
                                        ssx2[s] = f2_fma(ys[s], ys[s], ssx2[s]);
                                    }
                                    f32x2 h = f2_mul(f2_dup(pn.x), ys[0]);
                                    h = f2_fma(f2_dup(pn.y), ys[1], h);
                                    h = f2_fma(f2_dup(pn.z), ys[2], h);
                                    h = f2_fma(f2_dup(pn.w), ys[3], h);
                                    const f32x2 hr = f2_from_bf16x2(f2_to_bf16x2(h));
                                    ssh2[it] = f2_fma(hr, hr, ssh2[it]);
                                }
                            }
                        }
                    }
                    // the MMA warps (ldmatrix) and the store warp's TMA stores read these writes
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(staged_bar(slot));
                }
            }
            if (!ok) break;
            // this tile's state rows are no longer needed: the buffer may be refilled
            // (once every read of them has completed)
            __threadfence_block();
            __syncwarp();
            if (lane == 0) mbar_arrive(state_free(j & 1));
            if (kP1) {
                // tile finished: this CTA's sums of squares of the token go to the sender
                float ssx = f2_hsum(f2_add(f2_add(ssx2[0], ssx2[1]), f2_add(ssx2[2], ssx2[3])));
                float ssh = f2_hsum(f2_add(ssh2[0], ssh2[1]));
                ssx += __shfl_xor_sync(0xffffffffu, ssx, 1);
                ssx += __shfl_xor_sync(0xffffffffu, ssx, 2);
                ssh += __shfl_xor_sync(0xffffffffu, ssh, 1);
                ssh += __shfl_xor_sync(0xffffffffu, ssh, 2);
                if (uu == 0) {
                    *reinterpret_cast<float2 *>(sSS + ((j % kBufs) * kT + r) * 2) = make_float2(ssx, ssh);
                    mbar_arrive(ss_bar(j % kBufs));
                }
            }
        }
    }
    __syncwarp();
    tmem_fence_before_sync();
    cluster_sync_all();  // no CTA leaves while a peer may still touch its shared memory
    tmem_fence_after_sync();
    if (kP1 && warp == kWarpMma) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace ch

// ---------------------------------------------------------------- host side
namespace {

PFN_cuTensorMapEncodeTiled_v12000 chain_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        cudaDriverEntryPointQueryResult q;
        void *f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }
    return fn;
}

// rows x cols bf16 matrix, box of 64 rows x 64 columns, 128-byte swizzle
bool chain_tmap(CUtensorMap *m, const void *base, int64_t rows, int64_t cols) {
    auto enc = chain_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)ch::kCB, (cuuint32_t)ch::kT};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// n x 32 fp32 state rows, box of 64 rows x 32 floats (128 bytes), 128-byte swizzle
bool chain_state_tmap(CUtensorMap *m, const float *base, int64_t rows) {
    auto enc = chain_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)ch::kStateF, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)ch::kStateF * 4};
    cuuint32_t box[2] = {(cuuint32_t)ch::kStateF, (cuuint32_t)ch::kT};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int g_chain_clusters[64] = {};

template <int kMode>
cudaError_t launch_chain_impl(const ch::Params &prm, const uint16_t *x, const uint16_t *f,
                              uint16_t *y, uint16_t *h_norm, cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const ch::Layout L = ch::make_layout(prm.d);
    auto kern = ch::k_chain<kMode>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = ch::kC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(ch::kThreads);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = s;
    int &mc = g_chain_clusters[(dev & 63)];
    if (mc <= 0) {
        cfg.gridDim = dim3(ch::kC * 64);
        e = cudaOccupancyMaxActiveClusters(&mc, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (mc <= 0) return cudaErrorInvalidConfiguration;
    }
    const int64_t tiles = (prm.n + ch::kT - 1) / ch::kT;
    const int ncl = (int)(tiles < mc ? tiles : mc);
    cfg.gridDim = dim3(ch::kC * ncl);
    const int d = prm.d;
    CUtensorMap tmx, tmf, tmy, tmh, tms;
    if (!chain_tmap(&tmx, x, prm.n, (int64_t)kHC * d)) return cudaErrorInvalidValue;
    if (kMode != ch::kBegin) {
        if (!chain_tmap(&tmf, f, prm.n, d) || !chain_tmap(&tmy, y, prm.n, (int64_t)kHC * d) ||
            !chain_tmap(&tmh, h_norm, prm.n, d) || !chain_state_tmap(&tms, prm.state_in, prm.n))
            return cudaErrorInvalidValue;
    } else {
        tmf = tmy = tmh = tms = tmx;
    }
    ch::Params p = prm;
    p.num_tiles = (int)tiles;
    e = cudaLaunchKernelEx(&cfg, kern, tmx, tmf, tmy, tmh, tms, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

bool chain_supported(int d) {
    if (d <= 0 || d % (ch::kC * ch::kCB) != 0) return false;
    const ch::Layout L = ch::make_layout(d);
    return L.wcols <= (int)ch::kTmemCols && L.total <= 232448 && 2 * L.total > 233472;
}

cudaError_t launch_chain_begin(const uint16_t *x, const float *pre_mix, const float *hc_fn,
                               const float *hc_scale, const float *hc_base, int64_t n, int d,
                               int iters, float eps, float norm_eps, float *state_out,
                               float *pre_out, cudaStream_t s) {
    ch::Params p = {};
    p.pre_mix = pre_mix;
    p.hc_fn = hc_fn;
    p.hc_scale = hc_scale;
    p.hc_base = hc_base;
    p.state_out = state_out;
    p.pre_out = pre_out;
    p.n = n;
    p.d = d;
    p.iters = iters;
    p.eps = eps;
    p.norm_eps = norm_eps;
    return launch_chain_impl<ch::kBegin>(p, x, nullptr, nullptr, nullptr, s);
}

cudaError_t launch_chain_side(const uint16_t *x, const uint16_t *f, const float *state_in,
                              const float *norm_w, const float *hc_fn_next,
                              const float *hc_scale_next, const float *hc_base_next, int64_t n,
                              int d, int iters, float eps, float norm_eps, uint16_t *h_norm,
                              uint16_t *y, float *state_out, float *pre_out, cudaStream_t s) {
    ch::Params p = {};
    p.state_in = state_in;
    p.hc_fn = hc_fn_next;
    p.hc_scale = hc_scale_next;
    p.hc_base = hc_base_next;
    p.norm_w = norm_w;
    p.state_out = state_out;
    p.pre_out = pre_out;
    p.n = n;
    p.d = d;
    p.iters = iters;
    p.eps = eps;
    p.norm_eps = norm_eps;
    if (hc_fn_next) return launch_chain_impl<ch::kSide>(p, x, f, y, h_norm, s);
    return launch_chain_impl<ch::kLast>(p, x, f, y, h_norm, s);
}

cudaError_t consume_chain_device_error(cudaStream_t s, unsigned int *flag) {
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
