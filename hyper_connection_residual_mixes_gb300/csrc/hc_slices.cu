// hc_slices.cu -- the fused hyper-connection side steps on every SM of GB300.
//
// What it computes: per side, a1-a6 of the DeepSeek-V4.1 Block page, Code
// section (Block.hc_mixes, Block.hc_pre, Block.hc_post) with the split +
// Sinkhorn of the "Stream combination" page (hc_split_sinkhorn), for the chain
// Block.forward builds: the streams a side reads are the y the previous side
// wrote, and each side reads its sublayer input with the previous side's pre.
//
// How:
//  * The model dimension is cut into 16 column slices.  CTA b owns slice
//    c = b % 16 (columns [c d/16, (c+1) d/16) of every stream) and keeps the
//    matching 24 x 4d/16 slice of hc_fn in tensor memory for the whole launch,
//    split into bf16 hi + mid + lo laid out as mma.sync B fragments.  The CTAs
//    form groups of 16, one CTA per slice (nine groups on 152 SMs); group g takes
//    the 64-token tiles g, g + 9, ..., so all slices of a tile stream together.
//  * Phase 1 of a tile (the 24 projections on the tensor cores, the sum of
//    squares of the streams and of the bf16 sublayer input) gives, per token
//    and slice, 28 partial sums.  They go to global scratch, followed by an
//    arrival flag of the tile and slice.  The CTA of slice c that ran phase 1
//    of tile j then owns tokens 4c .. 4c+3 of the tile: it waits for the 16
//    arrival flags, adds the 16 partials in a fixed order, runs the split +
//    Sinkhorn and writes the coefficient rows of its tokens.
//  * Those rows are the state of the side: the next launch's phase 3 (y and
//    the sublayer input h_norm) reads them, so no CTA waits for another within
//    a launch except an owner for the 16 partial sums of its tokens.
//  * Flags hold the launch's epoch (a 64-bit value that differs from launch to
//    launch), so scratch never needs clearing.  A one-thread kernel enqueued
//    just before each launch writes the epoch into the state buffer's header
//    from a device counter, so a launch recorded into a CUDA graph draws a new
//    epoch at every replay.  Launches with flags are cooperative: every CTA
//    is resident, so a wait on another CTA's flag always ends; every wait is
//    bounded anyway and reports a timeout through the device error flag.  The
//    last side's launch (phase 3 alone) has no flags and is an ordinary one.
//
// Modes: kBegin (phase 1 of a chain's first side, on its x), kSide (phase 3 of
// side i, then phase 1 of side i + 1 on the y it has just produced), kLast
// (phase 3 of the last side).
//
// Scratch: the caller's state buffer holds the coefficient rows ([n, 32]
// fp32), then the partial sums ([n][16][28] fp32) and the arrival flags
// ([tiles][16] u64).
//
// Coefficient row (32 fp32 per token): post[4], comb[16] (row-major j*4+k),
// rs_h, 3 zeros, pre[4] (the side's pre: the next side's pre_mix), pre_mix[4]
// (the one the side reads its sublayer input with).
//
// Warp roles (512 threads): warps 0-3 tensor-core MMA (warp w: stream w, TMEM
// quadrant w); warp 4 TMA producer; warp 5 owner reduction + Sinkhorn; warps
// 6-13 CUDA-core streaming math; warp 14 sends each tile's partial sums; warp
// 15 TMA stores of y and h_norm.
#include <chrono>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "hc_device.cuh"
#include "hc_launch.h"
#include "hc_ptx.cuh"

namespace hc {

namespace sl {

constexpr int kS = 16;           // column slices of d
constexpr int kT = 64;           // tokens per tile
constexpr int kCB = 64;          // columns per slot per stream (128-byte box rows)
constexpr int kItems = 2;        // 8-column items per CUDA-core thread per slot
constexpr int kStepsPerSlot = kCB / 16;
constexpr int kSlots = 4;        // TMA ring depth (40 KB per slot)
constexpr int kBufs = 3;         // sums-of-squares hand-off buffers (CUDA-core warps -> sender)
constexpr uint32_t kTmemCols = 512;
constexpr int kThreads = 512;
constexpr int kBoxBytes = kT * kCB * 2;                // 8 KB
constexpr int kStageXBytes = kHC * kBoxBytes;          // 32 KB
constexpr int kSlotBytes = kStageXBytes + kBoxBytes;   // + f / h box = 40 KB
constexpr int kTokPerOwner = kT / kS;                  // 4
constexpr int kPartF = 28;       // 24 partial dots, sum x^2, sum h^2, 2 zeros
constexpr int kStateF = 32;      // floats per coefficient row
constexpr int kWarpMma = 0;
constexpr int kMmaWarps = 4;
constexpr int kWarpProducer = 4;
constexpr int kWarpOwner = 5;
constexpr int kWarpCuda = 6;     // warps 6..13
constexpr int kCudaWarps = 8;
constexpr int kWarpSender = 14;
constexpr int kWarpStore = 15;
constexpr int kWCols = 18;       // TMEM columns per k16 step: 3 n-tiles x (hi, mid, lo) x (b0, b1)
// Every slot use is released by the MMA warps, the CUDA-core warps and the store
// warp, and every use completes one phase of each of the slot's three barriers
// (full, staged, empty), whatever the use does: so phase parities follow the use
// count.  A role with nothing to do in a use still waits for the slot before it
// arrives, so that its arrival cannot count toward the previous use of the slot.
// And every role waits on the same barrier in every use (MMA warps: full, or
// staged in kSide; CUDA-core warps: full; store warp: staged): a parity wait
// only tells a phase from the one before it, so a role that skipped a barrier in
// some uses could run two phases ahead of it and pass a wait it should not
// (seen in a version that mixed use kinds in one ring).
constexpr int kEmptyArrivals = kMmaWarps + kCudaWarps + 1;
constexpr int kBegin = 0, kSide = 1, kLast = 2;
// what a block of slot uses does: phase 1 on x, phase 3, or phase 3 then phase 1 on its y
constexpr int kUseP1 = 0, kUseP3 = 1, kUseSide = 2;
// the bf16 box written over the f box: none, h_norm of the phase-3 side, or the
// unnormalised bf16 h of the side whose phase 1 runs here
constexpr int kHNone = 0, kHNorm = 1, kHPre = 2;
constexpr int kNumBars = 3 * kSlots + 2 * kBufs + 2 + 2 + 2 + 2;

struct Params {
    const float *state_in;   // kSide, kLast: coefficient rows of side i [n, 32]
    const float *pre_mix;    // kBegin: [n, 4]
    const float *hc_fn;      // weights of the side whose phase 1 runs here
    const float *hc_scale;
    const float *hc_base;
    const float *norm_w;     // [d]: the phase-3 side's RMSNorm weight
    float *state_out;        // kBegin, kSide: coefficient rows of the phase-1 side [n, 32]
    float *pre_out;          // [n, 4], optional: the phase-1 side's pre
    // scratch (see the file comment)
    float *part;             // partial sums of (token t, slice c): part + t*part_tok + c*part_slice
    int64_t part_tok, part_slice;
    unsigned long long *arrive;  // arrival flag of (tile j, slice c): arrive + j*arr_tile + c*arr_slice
    int64_t arr_tile, arr_slice;
    const unsigned long long *epoch;  // this launch's epoch (header of state_out)
    int64_t n;
    int d;
    int iters;
    float eps;
    float norm_eps;
    int num_tiles;
};

// The next epoch into a state buffer's header, just before the launch that
// writes the buffer (same stream): each launch, and each replay of a captured
// one, takes a value no earlier launch of the process has taken.
__device__ unsigned long long g_chain_launches = 0;
__global__ void k_chain_epoch(unsigned long long *hdr, unsigned long long base) {
    *hdr = base + atomicAdd(&g_chain_launches, 1ull) + 1ull;
}
constexpr bool kAnyP1Of(int mode) { return mode != kLast; }

// Shared-memory layout (byte offsets from a 1024-aligned base).
struct Layout {
    int dc, ncb, wcols;
    int off_state, off_pm, off_mma, off_ss, off_normw, off_bar, off_tmem, total;
};

__host__ __device__ inline Layout make_layout(int d) {
    Layout L;
    L.dc = d / kS;
    L.ncb = L.dc / kCB;
    L.wcols = kWCols * (L.dc / 16);
    int o = kSlots * kSlotBytes;
    L.off_state = o;  // two tiles of coefficient rows (phase 3)
    o += 2 * kT * kStateF * 4;
    L.off_pm = o;     // two tiles of pre_mix rows (phase 1 on x)
    o += 2 * kT * kHC * 4;
    L.off_mma = o;
    o += kMmaWarps * kT * kMix * 4;
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

// Block b of a CTA's slot uses (one tile phase, ncb uses) -> what it does and
// the index k of the tile in the CTA's list (tile g + k * groups).
template <int kMode>
__device__ __forceinline__ void block_of(int b, int J, int &type, int &k) {
    (void)J;
    type = kMode == kBegin ? kUseP1 : kMode == kSide ? kUseSide : kUseP3;
    k = b;
}
// What a use does, with what the mode rules out known at compile time.
template <int kMode>
__device__ __forceinline__ bool has_p1(int type) {
    (void)type;
    return kMode == kBegin || kMode == kSide;
}
template <int kMode>
__device__ __forceinline__ bool has_p3(int type) {
    (void)type;
    return kMode == kSide || kMode == kLast;
}

template <int kMode, int kH>
__global__ void __launch_bounds__(kThreads, 1)
k_slices(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_f,
         const __grid_constant__ CUtensorMap tm_y, const __grid_constant__ CUtensorMap tm_h,
         const __grid_constant__ CUtensorMap tm_s, const Params p) {
    constexpr bool kAnyP1 = kMode != kLast;
    constexpr bool kAnyP3 = kMode != kBegin;
    // written by k_chain_epoch, which ran to completion before this launch began
    const unsigned long long epoch = kAnyP1 ? *reinterpret_cast<const volatile unsigned long long *>(p.epoch) : 0ull;
    constexpr bool kPmRows = kMode == kBegin;  // phase 1 reads pre_mix rows
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    // the ring again, in the shared address space (ld.shared / st.shared)
    uint8_t *smem_ring = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ volatile int s_abort;
    const Layout L = make_layout(p.d);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = (int)gridDim.x;
    const int c = (int)blockIdx.x % kS;           // this CTA's column slice
    const int g = (int)blockIdx.x / kS;           // its index among the slice's CTAs
    const int m = (G - c + kS - 1) / kS;          // CTAs serving slice c
    const int J = (p.num_tiles > g) ? (p.num_tiles - g + m - 1) / m : 0;  // tiles g, g + m, ...
    const int NB = J;                             // blocks of slot uses (one per tile)
    const int ncb = L.ncb, dc = L.dc, d = p.d;
    const int64_t K = (int64_t)kHC * d;
    constexpr int hmode = kH;

    float *sState = reinterpret_cast<float *>(smem + L.off_state);
    float *sPm = reinterpret_cast<float *>(smem + L.off_pm);
    float *sMma = reinterpret_cast<float *>(smem + L.off_mma);
    float *sSS = reinterpret_cast<float *>(smem + L.off_ss);
    float *sNormW = reinterpret_cast<float *>(smem + L.off_normw);
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + L.off_tmem);
    const uint32_t bar0 = smem_u32(smem + L.off_bar);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kSlots + s); };
    // the CUDA-core warps have written y / h over the slot's x and f
    auto staged_bar = [&](int s) { return bar0 + 8u * (2 * kSlots + s); };
    auto ss_bar = [&](int b) { return bar0 + 8u * (3 * kSlots + b); };
    auto ss_free = [&](int b) { return bar0 + 8u * (3 * kSlots + kBufs + b); };
    const uint32_t mma_full = bar0 + 8u * (3 * kSlots + 2 * kBufs);
    const uint32_t mma_free = bar0 + 8u * (3 * kSlots + 2 * kBufs + 1);
    // the CUDA-core warps are done with a tile's coefficient rows / pre_mix rows (buffer b)
    auto state_free = [&](int b) { return bar0 + 8u * (3 * kSlots + 2 * kBufs + 2 + b); };
    auto pm_free = [&](int b) { return bar0 + 8u * (3 * kSlots + 2 * kBufs + 4 + b); };
    // this CTA's slice of hc_fn, bulk-copied into the (still empty) ring at launch
    // (wload), and the MMA warps done reading it from there (wfree)
    const uint32_t wload_bar = bar0 + 8u * (3 * kSlots + 2 * kBufs + 6);
    const uint32_t wfree_bar = bar0 + 8u * (3 * kSlots + 2 * kBufs + 7);
    const uint32_t slot0 = smem_u32(smem);

    if (threadIdx.x == kWarpProducer * 32) {
        s_abort = 0;
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kEmptyArrivals);
            mbar_init(staged_bar(s), kCudaWarps);
        }
        for (int b = 0; b < kBufs; ++b) {
            mbar_init(ss_bar(b), kT);
            mbar_init(ss_free(b), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(state_free(b), kCudaWarps);
            mbar_init(pm_free(b), kCudaWarps);
        }
        mbar_init(mma_full, kMmaWarps * 32);
        mbar_init(mma_free, 1);
        mbar_init(wload_bar, 1);
        mbar_init(wfree_bar, kMmaWarps);
        fence_mbar_init_cluster();
        prefetch_tmap(&tm_x);
        if (kAnyP3) {
            prefetch_tmap(&tm_f);
            prefetch_tmap(&tm_y);
            prefetch_tmap(&tm_s);
        }
        if (kH != kHNone) prefetch_tmap(&tm_h);
    }
    if (kAnyP1 && warp == kWarpMma) {
        tmem_alloc(smem_u32(sTmem), kTmemCols);
        tmem_relinquish();
    }
    if (kAnyP3)
        for (int i = threadIdx.x; i < dc; i += kThreads) sNormW[i] = __ldg(p.norm_w + c * dc + i);
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    const uint32_t tmem_base = kAnyP1 ? *sTmem : 0u;

    if (warp < kWarpMma + kMmaWarps) {
        // ------------------------------------------------------------ tensor-core projection
        const int s = warp - kWarpMma;
        const int gq = lane >> 2, t = lane & 3;
        const uint32_t tw = tmem_base + ((uint32_t)(32 * (warp & 3)) << 16);
        bool wok = true;
        if (kAnyP1) {
            // B fragments of this slice's weights: k16 step q occupies TMEM columns
            // 18q .. 18q + 17 as, per n-tile nt, hi(b0), hi(b1), mid(b0), mid(b1),
            // lo(b0), lo(b1) of W[nt*8+gq][k0+2t, +1] (b0) and W[nt*8+gq][k0+8+2t, +1] (b1).
            // The slice was bulk-copied into the ring at launch: row i of stream s at
            // floats (s * kMix + i) * dc.
            wok = mbar_wait_warp<false>(wload_bar, 0u, &s_abort);
            if (wok) {
                const float *wsm = reinterpret_cast<const float *>(smem) + (int64_t)s * kMix * dc;
                for (int q = 0; q < dc / 16; ++q) {
                    const int col = 16 * q + 2 * t;
#pragma unroll
                    for (int nt = 0; nt < 3; ++nt) {
                        const float *wr = wsm + (nt * 8 + gq) * dc + col;
                        const float2 p0 = *reinterpret_cast<const float2 *>(wr);
                        const float2 p1 = *reinterpret_cast<const float2 *>(wr + 8);
                        uint32_t h0, m0, l0, h1, m1, l1;
                        split3(p0.x, p0.y, h0, m0, l0);
                        split3(p1.x, p1.y, h1, m1, l1);
                        const uint32_t c0 = tw + kWCols * q + 6 * nt;
                        tmem_st2(c0 + 0, h0, h1);
                        tmem_st2(c0 + 2, m0, m1);
                        tmem_st2(c0 + 4, l0, l1);
                    }
                }
            }
            tmem_wait_st();
            // every value read from the ring has gone into tensor memory: the ring is the producer's
            __threadfence_block();
            __syncwarp();
            if (lane == 0) mbar_arrive(wfree_bar);
        }
        float acc[4][3][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 3; ++b)
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[a][b][e] = 0.0f;
        int u = 0, tiles_done = 0;
        bool ok = wok;
        for (int b = 0; b < NB && ok; ++b) {
            int type, k;
            block_of<kMode>(b, J, type, k);
            for (int cb = 0; cb < ncb; ++cb, ++u) {
                const int slot = u % kSlots;
                const uint32_t ph = (uint32_t)(u / kSlots) & 1u;
                // phase 1 on x: the slot's x; phase 1 on y: once y has replaced it; phase 3
                // alone: the slot only has to be filled before this warp may release it
                if (!mbar_wait_warp<false>(kMode == kSide ? staged_bar(slot) : full_bar(slot), ph, &s_abort)) {
                    ok = false;
                    break;
                }
                if (has_p1<kMode>(type)) {
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
                                    const uint32_t *bq = bw + kWCols * h2 + 6 * nt;
                                    mma_bf16_16816(acc[mt][nt], a0, a1, a2, a3, bq[4], bq[5]);  // lo
                                    mma_bf16_16816(acc[mt][nt], a0, a1, a2, a3, bq[2], bq[3]);  // mid
                                    mma_bf16_16816(acc[mt][nt], a0, a1, a2, a3, bq[0], bq[1]);  // hi
                                }
                            }
                        }
                    }
                }
                // the slot's last ldmatrix loads complete before it goes
                __threadfence_block();
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar(slot));
                if (has_p1<kMode>(type) && cb + 1 == ncb) {
                    if (!mbar_wait_warp<false>(mma_free, ((uint32_t)tiles_done & 1u) ^ 1u, &s_abort)) {
                        ok = false;
                        break;
                    }
                    float *mine = sMma + s * kT * kMix;
#pragma unroll
                    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
                        for (int nt = 0; nt < 3; ++nt) {
                            const int r = mt * 16 + gq, cc = nt * 8 + 2 * t;
                            *reinterpret_cast<float2 *>(mine + r * kMix + cc) = make_float2(acc[mt][nt][0], acc[mt][nt][1]);
                            *reinterpret_cast<float2 *>(mine + (r + 8) * kMix + cc) = make_float2(acc[mt][nt][2], acc[mt][nt][3]);
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
            const uint64_t pol_state = policy_evict_normal();  // 16 CTAs read each coefficient row
            int armed = 0, u = 0;
            int n_p1 = 0, n_p3 = 0;  // tiles whose phase 1 / phase 3 has started here
            bool ok = true;
            if (kAnyP1) {
                // the slice of hc_fn into the ring: 4 streams x 24 rows of dc floats
                mbar_arrive_expect_tx(wload_bar, (uint32_t)(kHC * kMix * dc * 4));
                for (int s = 0; s < kHC; ++s)
                    for (int i = 0; i < kMix; ++i)
                        bulk_load(slot0 + (uint32_t)((s * kMix + i) * dc * 4),
                                  p.hc_fn + (int64_t)i * K + (int64_t)s * d + (int64_t)c * dc,
                                  (uint32_t)(dc * 4), wload_bar);
                ok = mbar_wait<false>(wfree_bar, 0u, &s_abort);
            }
            for (int b = 0; b < NB && ok; ++b) {
                int type, k;
                block_of<kMode>(b, J, type, k);
                const int tile = g + k * m;
                const int row = tile * kT;
                for (int cb = 0; cb < ncb; ++cb, ++u) {
                    const int slot = u % kSlots;
                    const uint32_t ph = (uint32_t)(u / kSlots) & 1u;
                    if (!mbar_wait<false>(empty_bar(slot), ph ^ 1u, &s_abort)) {
                        ok = false;
                        break;
                    }
                    const int col = c * dc + cb * kCB;
                    const uint32_t dst = slot0 + slot * kSlotBytes;
                    uint32_t side_bytes = 0;
                    int pm_rows = 0;
                    if (cb == 0) {
                        if (kPmRows && has_p1<kMode>(type)) {
                            const int j = n_p1;
                            if (j >= 2 && !mbar_wait<false>(pm_free(j & 1), (uint32_t)((j - 2) >> 1) & 1u, &s_abort)) {
                                ok = false;
                                break;
                            }
                            const int64_t left = p.n - (int64_t)row;
                            pm_rows = (int)(left < kT ? left : kT);
                            side_bytes = 16u * (uint32_t)pm_rows;
                        }
                        if (has_p3<kMode>(type)) {
                            const int j = n_p3;
                            if (j >= 2 && !mbar_wait<false>(state_free(j & 1), (uint32_t)((j - 2) >> 1) & 1u, &s_abort)) {
                                ok = false;
                                break;
                            }
                            side_bytes = 4u * kStateF * kT;  // a TMA box always delivers all its bytes
                        }
                    }
                    mbar_arrive_expect_tx(full_bar(slot), (has_p3<kMode>(type) ? kSlotBytes : kStageXBytes) + side_bytes);
                    if (cb == 0) {
                        if (pm_rows > 0)
                            bulk_load(smem_u32(sPm) + (n_p1 & 1) * kT * kHC * 4, p.pre_mix + (int64_t)row * kHC,
                                      side_bytes, full_bar(slot));
                        if (has_p3<kMode>(type)) {
                            const uint32_t sdst = smem_u32(sState) + (n_p3 & 1) * kT * kStateF * 4;
                            tma_load_2d(sdst, &tm_s, full_bar(slot), 0, row, pol_state);
                        }
                    }
                    for (int s = 0; s < kHC; ++s) tma_load_2d(dst + s * kBoxBytes, &tm_x, full_bar(slot), s * d + col, row, pol);
                    if (has_p3<kMode>(type)) tma_load_2d(dst + kStageXBytes, &tm_f, full_bar(slot), col, row, pol);
                    armed = u + 1;
                }
                if (kPmRows && has_p1<kMode>(type)) ++n_p1;
                if (has_p3<kMode>(type)) ++n_p3;
            }
            for (int v = (armed > kSlots ? armed - kSlots : 0); v < armed; ++v)
                mbar_wait<false>(full_bar(v % kSlots), (uint32_t)(v / kSlots) & 1u, &s_abort);
        }
    } else if (warp == kWarpOwner) {
        // ------------------------------------------------------------ owner: statistics + Sinkhorn
        // Tokens 4c .. 4c+3 of every tile whose phase 1 ran here; 8 lanes per token,
        // lane `sub` adding the partials of slices sub and sub + 8, then a butterfly
        // over the 8 lanes: the token's 16 partials summed as
        // ((v0+v1)+(v2+v3)) + ((v4+v5)+(v6+v7)), v_s = e_s + e_{s+8}.
        if (kAnyP1) {
            const float s0 = __ldg(p.hc_scale), s1 = __ldg(p.hc_scale + 1), s2 = __ldg(p.hc_scale + 2);
            const int tl = lane >> 3, sub = lane & 7;
            const int tk = c * kTokPerOwner + tl;
            // the pre_mix the side reads with (the input, or the previous side's pre
            // kept in its coefficient rows), read one tile ahead
            auto load_pmx = [&](int kk) {
                const int64_t t = (int64_t)(g + kk * m) * kT + tk;
                if (kk >= J || t >= p.n) return make_float4(0.f, 0.f, 0.f, 0.f);
                return kMode == kSide ? __ldg(reinterpret_cast<const float4 *>(p.state_in + t * kStateF + 24))
                                      : __ldg(reinterpret_cast<const float4 *>(p.pre_mix) + t);
            };
            float4 pmx_next = load_pmx(0);
            for (int b = 0; b < NB; ++b) {
                int type, k;
                block_of<kMode>(b, J, type, k);
                if (!has_p1<kMode>(type)) continue;
                const float4 pmx = pmx_next;
                pmx_next = load_pmx(k + 1);
                const int tile = g + k * m;
                const int64_t tok = (int64_t)tile * kT + tk;
                bool ok = true;
                if (lane < kS) ok = flag_wait(p.arrive + (int64_t)tile * p.arr_tile + (int64_t)lane * p.arr_slice, epoch, &s_abort);
                if (!__all_sync(0xffffffffu, ok)) break;
                __threadfence();
                float mv[kMix + 2];
                if (tok < p.n) {
                    const float4 *e0 = reinterpret_cast<const float4 *>(p.part + tok * p.part_tok + (int64_t)sub * p.part_slice);
                    const float4 *e1 = reinterpret_cast<const float4 *>(p.part + tok * p.part_tok + (int64_t)(sub + 8) * p.part_slice);
                    float4 a[7], bb[7];
#pragma unroll
                    for (int q = 0; q < 7; ++q) {
                        a[q] = __ldcg(e0 + q);
                        bb[q] = __ldcg(e1 + q);
                    }
#pragma unroll
                    for (int q = 0; q < 7; ++q) {
                        if (4 * q < kMix + 2) mv[4 * q] = a[q].x + bb[q].x;
                        if (4 * q + 1 < kMix + 2) mv[4 * q + 1] = a[q].y + bb[q].y;
                        if (4 * q + 2 < kMix + 2) mv[4 * q + 2] = a[q].z + bb[q].z;
                        if (4 * q + 3 < kMix + 2) mv[4 * q + 3] = a[q].w + bb[q].w;
                    }
                } else {
#pragma unroll
                    for (int i = 0; i < kMix + 2; ++i) mv[i] = 0.0f;
                }
#pragma unroll
                for (int i = 0; i < kMix + 2; ++i) {
                    mv[i] += __shfl_xor_sync(0xffffffffu, mv[i], 1);
                    mv[i] += __shfl_xor_sync(0xffffffffu, mv[i], 2);
                    mv[i] += __shfl_xor_sync(0xffffffffu, mv[i], 4);
                }
                const float ssx = mv[kMix], ssh = mv[kMix + 1];
                const float r = rsqrtf(ssx / (float)K + p.norm_eps);
                float mm[kMix];
#pragma unroll
                for (int i = 0; i < kMix; ++i) mm[i] = mv[i] * r;
                float pr[kHC], po[kHC], cmb[kHC * kHC];
                split_sinkhorn_token<true>(mm, s0, s1, s2, p.hc_base, p.iters, p.eps, pr, po, cmb);
                const float rs_h = rsqrtf(ssh / (float)d + p.norm_eps);
                if (tok < p.n) {
                    const float4 row[8] = {make_float4(po[0], po[1], po[2], po[3]),
                                           make_float4(cmb[0], cmb[1], cmb[2], cmb[3]),
                                           make_float4(cmb[4], cmb[5], cmb[6], cmb[7]),
                                           make_float4(cmb[8], cmb[9], cmb[10], cmb[11]),
                                           make_float4(cmb[12], cmb[13], cmb[14], cmb[15]),
                                           make_float4(rs_h, 0.f, 0.f, 0.f),
                                           make_float4(pr[0], pr[1], pr[2], pr[3]), pmx};
                    if (sub == 0) {
                        float4 *st = reinterpret_cast<float4 *>(p.state_out + tok * kStateF);
#pragma unroll
                        for (int q = 0; q < 8; ++q) st[q] = row[q];
                    }
                    if (sub == 0 && p.pre_out) reinterpret_cast<float4 *>(p.pre_out)[tok] = row[6];
                }
            }
        }
    } else if (warp == kWarpSender) {
        // ------------------------------------------------------------ partial sums -> global scratch
        if (kAnyP1) {
            int tiles_done = 0;
            for (int b = 0; b < NB; ++b) {
                int type, k;
                block_of<kMode>(b, J, type, k);
                if (!has_p1<kMode>(type)) continue;
                const int tile = g + k * m;
                const int buf = tiles_done % kBufs;
                if (!mbar_wait_warp<false>(mma_full, (uint32_t)tiles_done & 1u, &s_abort)) break;
                if (!mbar_wait_warp<false>(ss_bar(buf), (uint32_t)(tiles_done / kBufs) & 1u, &s_abort)) break;
                float v[2][kPartF];
#pragma unroll
                for (int i2 = 0; i2 < 2; ++i2) {
                    // tokens lane and lane + 32: neighbouring lanes read neighbouring rows
                    const int tk = lane + 32 * i2;
#pragma unroll
                    for (int i = 0; i < kMix; ++i) v[i2][i] = 0.0f;
#pragma unroll
                    for (int w = 0; w < kMmaWarps; ++w) {
                        const float *e = sMma + (w * kT + tk) * kMix;
#pragma unroll
                        for (int i = 0; i < kMix; ++i) v[i2][i] += e[i];
                    }
                    const float2 ss = *reinterpret_cast<const float2 *>(sSS + (buf * kT + tk) * 2);
                    v[i2][kMix] = ss.x;
                    v[i2][kMix + 1] = ss.y;
                    v[i2][kMix + 2] = v[i2][kMix + 3] = 0.0f;
                }
                // the hand-off buffers are read: give them back
                __threadfence_block();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(mma_free);
                    mbar_arrive(ss_free(buf));
                }
#pragma unroll
                for (int i2 = 0; i2 < 2; ++i2) {
                    const int64_t tok = (int64_t)tile * kT + lane + 32 * i2;
                    if (tok < p.n) {
                        float4 *dst = reinterpret_cast<float4 *>(p.part + tok * p.part_tok + (int64_t)c * p.part_slice);
#pragma unroll
                        for (int q = 0; q < kPartF / 4; ++q)
                            __stcg(dst + q, make_float4(v[i2][4 * q], v[i2][4 * q + 1], v[i2][4 * q + 2], v[i2][4 * q + 3]));
                    }
                }
                __threadfence();
                __syncwarp();
                if (lane == 0) st_release_u64(p.arrive + (int64_t)tile * p.arr_tile + (int64_t)c * p.arr_slice, epoch);
                ++tiles_done;
            }
        }
    } else if (warp == kWarpStore) {
        // ------------------------------------------------------------ TMA stores of y and h
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int u = 0;
            bool ok = true;
            for (int b = 0; b < NB && ok; ++b) {
                int type, k;
                block_of<kMode>(b, J, type, k);
                const int row = (g + k * m) * kT;
                const bool store_h = hmode == kHPre ? has_p1<kMode>(type) : (hmode == kHNorm && has_p3<kMode>(type));
                const bool stores = has_p3<kMode>(type) || store_h;
                for (int cb = 0; cb < ncb; ++cb, ++u) {
                    const int slot = u % kSlots;
                    const uint32_t ph = (uint32_t)(u / kSlots) & 1u;
                    // `staged` in every use, stores or not: a parity wait tells a phase only from
                    // the one before it, so a waiter must never run two phases ahead of a barrier
                    if (!mbar_wait<false>(staged_bar(slot), ph, &s_abort)) {
                        ok = false;
                        break;
                    }
                    if (stores) {
                        const int col = c * dc + cb * kCB;
                        const uint32_t src = slot0 + slot * kSlotBytes;
                        if (has_p3<kMode>(type))
                            for (int s = 0; s < kHC; ++s) tma_store_2d(&tm_y, src + s * kBoxBytes, s * d + col, row, pol);
                        if (store_h) tma_store_2d(&tm_h, src + kStageXBytes, col, row, pol);
                        bulk_commit_group();
                        bulk_wait_group_read<0>();  // the slot's bytes are out: it may be refilled
                    }
                    mbar_arrive(empty_bar(slot));
                }
            }
            bulk_wait_group<0>();  // every store has landed before the CTA leaves
        }
    } else {
        // ------------------------------------------------------------ CUDA-core streaming math
        // 256 threads; per slot, thread tc handles token row r and the 8-column
        // units uu + 4i (i < 2).  Each quarter-warp reads rows r and r + 4, which
        // the 128-byte swizzle maps to complementary bank halves.
        const int tc = threadIdx.x - kWarpCuda * 32;
        const int uu = lane & 3;
        const int r = 8 * (tc >> 5) + (lane >> 3) + 4 * ((lane >> 2) & 1);
        int u = 0, n_p1 = 0, n_p3 = 0, tiles_done = 0;
        bool ok = true;
        for (int b = 0; b < NB && ok; ++b) {
            int type, k;
            block_of<kMode>(b, J, type, k);
            const int64_t tok = (int64_t)(g + k * m) * kT + r;
            const bool live = tok < p.n;
            // this tile's coefficient rows (128-byte rows with the 128-byte swizzle, so the
            // eight rows a warp reads fall on distinct banks) or pre_mix rows
            const uint8_t *srow = reinterpret_cast<const uint8_t *>(sState) + (n_p3 & 1) * kT * kStateF * 4;
            const float *pmrow = sPm + (n_p1 & 1) * kT * kHC;
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
                if (has_p1<kMode>(type) && kMode != kSide) {
                    // ---------------- phase 1 on x
                    constexpr bool write_h = hmode == kHPre;
                    const float4 v = live ? *reinterpret_cast<const float4 *>(pmrow + r * kHC) : make_float4(0.f, 0.f, 0.f, 0.f);
                    const f32x2 pm[kHC] = {f2_dup(v.x), f2_dup(v.y), f2_dup(v.z), f2_dup(v.w)};
#pragma unroll
                    for (int it = 0; it < kItems; ++it) {
                        uint32_t ho[4];
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
                            ho[q] = f2_to_bf16x2(h);
                            const f32x2 hr = f2_from_bf16x2(ho[q]);
                            ssh2[it] = f2_fma(hr, hr, ssh2[it]);
                        }
                        if (write_h)  // the side's bf16 h, over the f box (not loaded in phase 1)
                            *reinterpret_cast<uint4 *>(sb + kStageXBytes + swz(r, uu + 4 * it)) = make_uint4(ho[0], ho[1], ho[2], ho[3]);
                    }
                    // The slot goes only once every value loaded from it has been used: a
                    // release right after the loads (with a CTA-scope fence) still let the
                    // next use's TMA load overwrite the slot under this warp's loads in
                    // runs with phase 3 blocks in between (measured: a few sums of squares
                    // differing from run to run).  Every use arrives on `staged` too, so
                    // that each slot's barriers complete exactly one phase per use.
                    if (write_h) fence_proxy_async_smem();
                    __threadfence_block();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(staged_bar(slot));
                        mbar_arrive(empty_bar(slot));
                    }
                } else {
                    // ---------------- phase 3 of side i (then phase 1 of side i + 1 on its y)
                    const uint4 fr0 = *reinterpret_cast<const uint4 *>(sb + kStageXBytes + swz(r, uu));
                    const uint4 fr1 = *reinterpret_cast<const uint4 *>(sb + kStageXBytes + swz(r, uu + 4));
                    if (live) {
                        float cf[kHC + kHC * kHC];  // post, comb: 16-byte chunks 0-4 of the row
#pragma unroll
                        for (int q = 0; q < 5; ++q) {
                            const float4 v = *reinterpret_cast<const float4 *>(srow + swz(r, q));
                            cf[4 * q] = v.x;
                            cf[4 * q + 1] = v.y;
                            cf[4 * q + 2] = v.z;
                            cf[4 * q + 3] = v.w;
                        }
                        const float rs = *reinterpret_cast<const float *>(srow + swz(r, 5));
                        const float4 pmv = *reinterpret_cast<const float4 *>(srow + swz(r, 7));
                        const float4 pn = *reinterpret_cast<const float4 *>(srow + swz(r, 6));
#pragma unroll
                        for (int it = 0; it < kItems; ++it) {
                            const uint4 &fw = it == 0 ? fr0 : fr1;
                            const int un = uu + 4 * it;
                            uint32_t yo[kHC][4], ho[4];
                            if constexpr (hmode == kHNorm) {
                                const float4 *nw = reinterpret_cast<const float4 *>(sNormW + cb * kCB + un * 8);
                                const float4 w0 = nw[0], w1 = nw[1];
                                const f32x2 wv[4] = {f2_make(w0.x, w0.y), f2_make(w0.z, w0.w), f2_make(w1.x, w1.y),
                                                     f2_make(w1.z, w1.w)};
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    f32x2 xs[kHC];
#pragma unroll
                                    for (int s = 0; s < kHC; ++s) {
                                        const uint4 &w = xr[it][s];
                                        xs[s] = f2_from_bf16x2(q == 0 ? w.x : q == 1 ? w.y : q == 2 ? w.z : w.w);
                                    }
                                    f32x2 h = f2_mul(f2_dup(pmv.x), xs[0]);
                                    h = f2_fma(f2_dup(pmv.y), xs[1], h);
                                    h = f2_fma(f2_dup(pmv.z), xs[2], h);
                                    h = f2_fma(f2_dup(pmv.w), xs[3], h);
                                    const f32x2 hr = f2_from_bf16x2(f2_to_bf16x2(h));
                                    ho[q] = f2_to_bf16x2(f2_mul(f2_mul(hr, f2_dup(rs)), wv[q]));
                                }
                            }
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
                                for (int kk = 0; kk < kHC; ++kk) {
                                    f32x2 a = f2_mul(f2_dup(cf[kk]), fv);
#pragma unroll
                                    for (int jj = 0; jj < kHC; ++jj) a = f2_fma(f2_dup(cf[kHC + jj * kHC + kk]), xs[jj], a);
                                    yo[kk][q] = f2_to_bf16x2(a);
                                }
                            }
                            // y replaces, in place, the x words this thread alone read
                            uint8_t *wb = sb + swz(r, un);
#pragma unroll
                            for (int kk = 0; kk < kHC; ++kk)
                                *reinterpret_cast<uint4 *>(wb + kk * kBoxBytes) = make_uint4(yo[kk][0], yo[kk][1], yo[kk][2], yo[kk][3]);
                            if (kMode == kSide) {
                                // phase 1 of side i + 1 on this y: its x is y, its pre_mix side i's pre
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
                                    const uint32_t hb = f2_to_bf16x2(h);
                                    if constexpr (hmode == kHPre) ho[q] = hb;
                                    const f32x2 hr = f2_from_bf16x2(hb);
                                    ssh2[it] = f2_fma(hr, hr, ssh2[it]);
                                }
                            }
                            if constexpr (hmode != kHNone)  // h_norm of side i, or side i + 1's bf16 h, over the f words
                                *reinterpret_cast<uint4 *>(wb + kStageXBytes) = make_uint4(ho[0], ho[1], ho[2], ho[3]);
                        }
                    }
                    // the MMA warps (ldmatrix) and the store warp's TMA stores read these writes
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(staged_bar(slot));
                        mbar_arrive(empty_bar(slot));
                    }
                }
            }
            if (!ok) break;
            // this tile's coefficient / pre_mix rows are no longer needed (once every read completed)
            __threadfence_block();
            __syncwarp();
            if (has_p3<kMode>(type)) {
                if (lane == 0) mbar_arrive(state_free(n_p3 & 1));
                ++n_p3;
            }
            if (kPmRows && has_p1<kMode>(type)) {
                if (lane == 0) mbar_arrive(pm_free(n_p1 & 1));
                ++n_p1;
            }
            if (has_p1<kMode>(type)) {
                // tile finished: this CTA's sums of squares of the token go to the sender
                float ssx = f2_hsum(f2_add(f2_add(ssx2[0], ssx2[1]), f2_add(ssx2[2], ssx2[3])));
                float ssh = f2_hsum(f2_add(ssh2[0], ssh2[1]));
                ssx += __shfl_xor_sync(0xffffffffu, ssx, 1);
                ssx += __shfl_xor_sync(0xffffffffu, ssx, 2);
                ssh += __shfl_xor_sync(0xffffffffu, ssh, 1);
                ssh += __shfl_xor_sync(0xffffffffu, ssh, 2);
                const int buf = tiles_done % kBufs;
                if (tiles_done >= kBufs &&
                    !mbar_wait_warp<false>(ss_free(buf), (uint32_t)((tiles_done / kBufs) - 1) & 1u, &s_abort))
                    break;
                if (uu == 0) {
                    *reinterpret_cast<float2 *>(sSS + (buf * kT + r) * 2) = make_float2(ssx, ssh);
                    mbar_arrive(ss_bar(buf));
                }
                ++tiles_done;
            }
        }
    }
    __syncwarp();
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    if (kAnyP1 && warp == kWarpMma) tmem_dealloc(tmem_base, kTmemCols);
}

}  // namespace sl

// ---------------------------------------------------------------- host side
namespace {

PFN_cuTensorMapEncodeTiled_v12000 slices_encode() {
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
bool slices_tmap(CUtensorMap *map, const void *base, int64_t rows, int64_t cols) {
    auto enc = slices_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)sl::kCB, (cuuint32_t)sl::kT};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// n x 32 fp32 coefficient rows, box of 64 rows x 32 floats (128 bytes), 128-byte swizzle
bool slices_state_tmap(CUtensorMap *map, const float *base, int64_t rows) {
    auto enc = slices_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)sl::kStateF, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)sl::kStateF * 4};
    cuuint32_t box[2] = {(cuuint32_t)sl::kStateF, (cuuint32_t)sl::kT};
    cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The epochs: a per-process base (below 2^63, drawn from the clock) plus the
// count of chain launches so far on the device, so that flags written by an
// earlier launch (or left in a reused buffer) never match the current one's.
unsigned long long epoch_base() {
    static const unsigned long long base =
        ((unsigned long long)std::chrono::steady_clock::now().time_since_epoch().count() * 0x9E3779B97F4A7C15ull) >>
        1;
    return base;
}

int g_slices_ctas[64] = {};  // co-resident CTAs per device (one per SM)

template <int kMode, int kH>
cudaError_t launch_slices_impl(sl::Params p, const uint16_t *x, const uint16_t *f, uint16_t *y,
                               uint16_t *h, cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const sl::Layout L = sl::make_layout(p.d);
    auto kern = sl::k_slices<kMode, kH>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
    if (e != cudaSuccess) return e;
    int &cap = g_slices_ctas[dev & 63];
    if (cap <= 0) {
        int sms = 0, per_sm = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, sl::kThreads, L.total);
        if (e != cudaSuccess) return e;
        if (per_sm < 1 || sms < sl::kS) return cudaErrorInvalidConfiguration;
        // One CTA per SM (each takes the whole tensor memory), in whole groups of 16:
        // group g takes tiles g, g + G/16, ..., so the 16 slices of a tile are read at
        // the same time (each x row is read in 16 adjacent pieces, one per slice).
        cap = (sms / sl::kS) * sl::kS;
    }
    const int64_t tiles = (p.n + sl::kT - 1) / sl::kT;
    const int64_t want = tiles * sl::kS;
    const int grid = (int)(want < cap ? want : cap);
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    // only launches with a cross-slice reduction wait on other CTAs' flags and need
    // every CTA resident; the last side's (phase 3 alone) is an ordinary launch
    cfg.numAttrs = sl::kAnyP1Of(kMode) ? 1 : 0;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(sl::kThreads);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = s;
    const int d = p.d;
    CUtensorMap tmx, tmf, tmy, tmh, tms;
    if (!slices_tmap(&tmx, x, p.n, (int64_t)kHC * d)) return cudaErrorInvalidValue;
    tmf = tmy = tmh = tms = tmx;
    if (kMode != sl::kBegin) {
        if (!slices_tmap(&tmf, f, p.n, d) || !slices_tmap(&tmy, y, p.n, (int64_t)kHC * d))
            return cudaErrorInvalidValue;
        if (!slices_state_tmap(&tms, p.state_in, p.n)) return cudaErrorInvalidValue;
    }
    if (kH != sl::kHNone && !slices_tmap(&tmh, h, p.n, d)) return cudaErrorInvalidValue;
    p.num_tiles = (int)tiles;
    if (sl::kAnyP1Of(kMode)) {
        sl::k_chain_epoch<<<1, 1, 0, s>>>(const_cast<unsigned long long *>(p.epoch), epoch_base());
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    e = cudaLaunchKernelEx(&cfg, kern, tmx, tmf, tmy, tmh, tms, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Scratch of the chain inside a state buffer: after the n coefficient rows
// (rounded up to 256 bytes), the partial sums [n][16][28] fp32, the arrival
// flags [tiles][16] u64, then a 16-byte header holding the epoch of the launch
// that writes this buffer.
struct ChainScratch {
    size_t part_off, flag_off, hdr_off, total;
};
ChainScratch chain_scratch(int64_t n) {
    ChainScratch cs;
    const size_t rows = ((size_t)n * sl::kStateF * 4 + 255) & ~size_t(255);
    cs.part_off = rows;
    cs.flag_off = cs.part_off + (size_t)n * sl::kS * sl::kPartF * 4;
    const size_t tiles = (size_t)((n + sl::kT - 1) / sl::kT);
    cs.hdr_off = cs.flag_off + tiles * sl::kS * 8;
    cs.total = cs.hdr_off + 16;
    return cs;
}

void set_chain_scratch(sl::Params &p, float *state_out) {
    const ChainScratch cs = chain_scratch(p.n);
    uint8_t *base = reinterpret_cast<uint8_t *>(state_out);
    p.part = reinterpret_cast<float *>(base + cs.part_off);
    p.part_tok = (int64_t)sl::kS * sl::kPartF;
    p.part_slice = sl::kPartF;
    p.arrive = reinterpret_cast<unsigned long long *>(base + cs.flag_off);
    p.arr_tile = sl::kS;
    p.arr_slice = 1;
    p.epoch = reinterpret_cast<const unsigned long long *>(base + cs.hdr_off);
}

}  // namespace

bool slices_supported(int d) {
    if (d <= 0 || d % (sl::kS * sl::kCB) != 0) return false;
    const sl::Layout L = sl::make_layout(d);
    // the weight slice is staged at launch over the ring and the row buffers
    // after it, which nothing uses before the MMA warps have read it
    const bool staged_fits = kHC * kMix * L.dc * 4 <= L.off_mma;
    return L.wcols <= (int)sl::kTmemCols && staged_fits && L.total <= 232448 && 2 * L.total > 233472;
}

size_t chain_state_bytes(int64_t n) { return chain_scratch(n).total; }

cudaError_t launch_slices_begin(const uint16_t *x, const float *pre_mix, const float *hc_fn,
                                const float *hc_scale, const float *hc_base, int64_t n, int d,
                                int iters, float eps, float norm_eps, float *state_out,
                                float *pre_out, uint16_t *h_pre_out, cudaStream_t s) {
    sl::Params p = {};
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
    set_chain_scratch(p, state_out);
    if (h_pre_out) return launch_slices_impl<sl::kBegin, sl::kHPre>(p, x, nullptr, nullptr, h_pre_out, s);
    return launch_slices_impl<sl::kBegin, sl::kHNone>(p, x, nullptr, nullptr, nullptr, s);
}

cudaError_t launch_slices_side(const uint16_t *x, const uint16_t *f, const float *state_in,
                               const float *norm_w, const float *hc_fn_next,
                               const float *hc_scale_next, const float *hc_base_next, int64_t n,
                               int d, int iters, float eps, float norm_eps, uint16_t *h_norm,
                               uint16_t *y, float *state_out, float *pre_out, uint16_t *h_pre_out,
                               cudaStream_t s) {
    sl::Params p = {};
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
    if (hc_fn_next) {
        // h_norm of side i and side i + 1's bf16 h share the box over f: one or the other
        set_chain_scratch(p, state_out);
        if (h_pre_out) return launch_slices_impl<sl::kSide, sl::kHPre>(p, x, f, y, h_pre_out, s);
        return launch_slices_impl<sl::kSide, sl::kHNorm>(p, x, f, y, h_norm, s);
    }
    if (h_norm) return launch_slices_impl<sl::kLast, sl::kHNorm>(p, x, f, y, h_norm, s);
    return launch_slices_impl<sl::kLast, sl::kHNone>(p, x, f, y, nullptr, s);
}

cudaError_t consume_slices_device_error(cudaStream_t s, unsigned int *flag) {
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
