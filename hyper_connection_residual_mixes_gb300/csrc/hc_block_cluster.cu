// hc_block_cluster.cu -- the fused hyper-connection side step for GB300.
//
// What it computes (DeepSeek-V4.1 Block page, Code section: Block.hc_mixes,
// Block.hc_pre, Block.hc_post; "Stream combination" page: hc_split_sinkhorn):
// per token, the 24 mix numbers from the flattened streams and one
// rsqrt(mean(x^2) + norm_eps) statistic, split + Sinkhorn into pre/post/comb,
// h = bf16(sum_s pre_mix[s] x[s]), h_norm = bf16(RMSNorm(h) * w) and
// y[k] = bf16(post[k] f + sum_j comb[j][k] x[j]).
//
// How (one launch per side step, persistent thread-block clusters):
//  * A cluster of kC = 16 CTAs (one per SM) splits the model dimension d into
//    16 column slices; CTA `rank` owns columns [rank*d/16, (rank+1)*d/16) of
//    each of the 4 streams.
//  * The CTA's slice of hc_fn (24 rows x 4*d/16 columns) is split once, at
//    launch, into three bf16 parts per fp32 weight (hi + mid + lo, exact to
//    ~2^-24 relative) laid out as mma.sync B fragments, and kept in tensor
//    memory for the whole launch: one 32-lane TMEM quadrant per MMA warp, one
//    stream per MMA warp.  Weights are never re-read per token and take no
//    shared memory.
//  * A cluster walks 64-token tiles.  Each tile's streams pass through a
//    4-slot TMA ring (64 columns x 64 tokens x 4 streams per slot, 128-byte
//    swizzle, plus the f box in phase 3) twice: phase 1 (the projection, sum
//    of squares, and the sum of squares of the bf16-rounded h) and phase 3
//    (y and h_norm).  The second read comes from L2 (the first read is tagged
//    evict_last, the second evict_first); phase 1 of the next tile runs
//    between them so the cross-CTA reduction of a tile is hidden behind
//    useful streaming.
//  * The projection runs on the tensor cores (mma.sync m16n8k16, bf16 in,
//    fp32 accumulate); x is bf16 and enters exactly; the three weight parts
//    accumulate into the same fp32 sums.
//  * Partial sums (24 dots, sum x^2, sum h^2) of each token go to the token's
//    owner CTA through distributed shared memory with cluster-scope mbarrier
//    arrivals; the owner finishes the statistics, runs the split + 20-round
//    Sinkhorn in registers, writes pre/post/comb, and broadcasts post, comb
//    and the RMSNorm scale back to all 16 CTAs.
//
// Warp roles (480 threads): warps 0-3 tensor-core MMA (warp w: stream w, TMEM
// quadrant w); warp 4 TMA producer; warp 5 owner-side reduction + Sinkhorn +
// broadcast; warps 6-13 CUDA-core streaming math (two 8-column units of one
// token per thread per slot, packed f32x2 arithmetic, one block of slots per
// tile phase); warp 14 sends each tile's partial sums to the owners.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "hc_device.cuh"
#include "hc_launch.h"
#include "hc_ptx.cuh"

namespace hc {

namespace cl {

constexpr int kC = 16;          // CTAs per cluster = column slices of d
constexpr int kT = 64;          // tokens per tile
#ifndef HC_CB
#define HC_CB 64
#endif
constexpr int kCB = HC_CB;      // columns per slot (per stream): 32 (64-byte rows) or 64 (128-byte rows)
constexpr int kUnits = kCB / 8;  // 16-byte units per box row
constexpr int kItems = kUnits / 4;  // 8-column items per CUDA-core thread per slot
constexpr int kStepsPerSlot = kCB / 16;  // k16 MMA steps per stream per slot
static_assert(kCB == 32 || kCB == 64, "column block must be 32 or 64");
// Tuning knobs (compile-time): ring depth and the phase-3 lag.
#ifndef HC_SLOTS
#define HC_SLOTS 4
#endif
#ifndef HC_LAG
#define HC_LAG 1
#endif
#ifndef HC_STORE_EVICT_FIRST
#define HC_STORE_EVICT_FIRST 1
#endif
constexpr int kSlots = HC_SLOTS;  // TMA ring depth (40 KB per slot)
constexpr int kLag = HC_LAG;      // phase 3 of tile j runs after phase 1 of tile j + kLag
constexpr int kBufs = kLag + 1; // partial / coefficient buffers in rotation
constexpr uint32_t kTmemCols = 512;  // the whole tensor memory of the SM (1 CTA per SM)
constexpr int kThreads = 480;
constexpr int kBoxBytes = kT * kCB * 2;             // 64 tokens x kCB bf16 = 8 KB
constexpr int kStageXBytes = kHC * kBoxBytes;       // 4 streams = 32 KB
constexpr int kSlotBytes = kStageXBytes + kBoxBytes;  // + f box = 40 KB
constexpr int kTokPerOwner = kT / kC;               // 4
constexpr int kPartF = 28;      // 24 partial dots, sum x^2, sum h^2, 2 pad
constexpr int kCoefF = 24;      // post[4], comb[16], rs_h, 3 pad
constexpr int kWarpMma = 0;     // warps 0..3: MMA warp w owns stream w and TMEM quadrant w
constexpr int kMmaWarps = 4;
constexpr int kWarpProducer = 4;
constexpr int kWarpReducer = 5;
constexpr int kWarpCuda = 6;    // warps 6..13
constexpr int kCudaWarps = 8;
constexpr int kWarpSender = 14; // adds up each tile's partial sums and sends them to the owners
constexpr int kWCols = 18;      // TMEM columns per k16 step: 3 n-tiles x (hi, mid, lo) x (b0, b1)
// pre_mix tile buffers: tile j's rows must survive until phase 3 of tile j has
// read them.  With one column block per tile phase (d = 1024) the ring can load
// phase 1 of tile j + 3 as soon as phase 1 of tile j + 1 is released, which may
// precede phase 3 of tile j; a fourth buffer keeps tile j + 4 further out.
constexpr int kPmBufs = 4;

struct Params {
    const float *pre_mix;
    const float *hc_fn;
    const float *hc_scale;
    const float *hc_base;
    const float *norm_w;
    uint16_t *h_norm;
    uint16_t *y;
    float *pre_out;
    float *post_out;
    float *comb_out;
    float *mixes_out;
    int64_t n;
    int d;
    int iters;
    float eps;
    float norm_eps;
    int num_tiles;
};

// Shared-memory layout (byte offsets from a 1024-aligned base).
struct Layout {
    int dc;        // columns per CTA per stream = d / 16
    int ncb;       // slots per tile phase = dc / kCB
    int wcols;     // tensor-memory columns per MMA warp: 18 per k16 step, 2*ncb steps
    int off_coef, off_part, off_mma, off_ss, off_pm, off_normw, off_bar, off_tmem, total;
};

__host__ __device__ inline Layout make_layout(int d) {
    Layout L;
    L.dc = d / kC;
    L.ncb = L.dc / kCB;
    L.wcols = kWCols * (L.dc / 16);
    int o = kSlots * kSlotBytes;
    L.off_coef = o;
    o += kBufs * kT * kCoefF * 4;
    L.off_part = o;
    o += kBufs * kC * kTokPerOwner * kPartF * 4;
    L.off_mma = o;
    o += kMmaWarps * kT * kMix * 4;
    L.off_ss = o;  // CTA-local sums of squares, handed from the CUDA-core to the MMA warps
    o += 2 * kT * 2 * 4;
    L.off_pm = o;  // pre_mix rows of a tile, copied in with its first slot; 3 tiles in rotation
    o += kPmBufs * kT * 16;
    L.off_normw = o;
    o += L.dc * 4;
    o = (o + 15) & ~15;
    L.off_bar = o;
    o += (2 * kSlots + 2 * kBufs + 6) * 8;  // full[], empty[], part[], coef[], 2 MMA meetings, ss[2], weights
    o = (o + 15) & ~15;
    L.off_tmem = o;
    o += 16;
    L.total = o + 1024;  // slack for aligning the base
    return L;
}

// Split an fp32 pair into three bf16x2 parts with hi + mid + lo == w to ~2^-24.
__device__ __forceinline__ void split3(float w0, float w1, uint32_t &hi, uint32_t &mid, uint32_t &lo) {
    hi = pack_bf16x2(w0, w1);
    const float r0 = w0 - bf16lo(hi), r1 = w1 - bf16hi(hi);
    mid = pack_bf16x2(r0, r1);
    const float s0 = r0 - bf16lo(mid), s1 = r1 - bf16hi(mid);
    lo = pack_bf16x2(s0, s1);
}

// Byte offset of (row r, 16-byte unit u) inside a TMA box of kCB-column rows,
// written with the 64-byte (kCB = 32) or 128-byte (kCB = 64) swizzle: the
// unit index is XORed with address bits 7-8 (resp. 7-9).
__device__ __forceinline__ uint32_t swz(int r, int u) {
    if constexpr (kCB == 32) return (uint32_t)(r * 64 + ((u ^ ((r >> 1) & 3)) << 4));
    else return (uint32_t)(r * 128 + ((u ^ (r & 7)) << 4));
}

// The ring walks, per cluster, blocks of `ncb` slot uses:
//   P1(0) .. P1(kLag-1), then pairs P1(j + kLag), P3(j), then the last P3s.
// Phase 3 of a tile thus starts kLag tiles of streaming after its phase 1,
// which hides the cross-CTA reduction, Sinkhorn and broadcast of that tile.
// Use u -> (phase 3?, local tile j, column block cb).
struct Use {
    bool p3;
    int j;
    int cb;
};
// Block b (ncb consecutive uses) -> (phase 3?, local tile j); no division.
__device__ __forceinline__ Use block_use(int b, int J, bool full) {
    Use r;
    r.cb = 0;
    if (!full) {
        r.p3 = false;
        r.j = b;
        return r;
    }
    const int l0 = J < kLag ? J : kLag;
    if (b < l0) {
        r.p3 = false;
        r.j = b;
        return r;
    }
    const int c = b - l0;
    const int pairs = J - l0;
    if (c < 2 * pairs) {
        r.p3 = (c & 1) != 0;
        r.j = r.p3 ? (c >> 1) : l0 + (c >> 1);
        return r;
    }
    r.p3 = true;
    r.j = pairs + (c - 2 * pairs);
    return r;
}
__device__ __forceinline__ Use decode_use(int u, int ncb, int J, bool full) {
    Use r = block_use(u / ncb, J, full);
    r.cb = u % ncb;
    return r;
}
__device__ __forceinline__ int total_uses(int ncb, int J, bool full) {
    return full ? 2 * ncb * J : ncb * J;
}

template <bool kFull>
__global__ void __launch_bounds__(kThreads, 1)
k_block_cluster(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_f,
                const Params p) {
    extern __shared__ uint8_t smem_raw[];
    // The same 1024-byte aligned base twice: a generic pointer (measured faster for
    // the handoff buffers) and one derived from the shared array itself, which the
    // compiler keeps in the shared address space (ld.shared for the slot reads of
    // the CUDA-core warps, measured faster there).
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~uintptr_t(1023));
    const uint8_t *smem_ring = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    __shared__ volatile int s_abort;
    const Layout L = make_layout(p.d);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int cid = (int)cluster_id_x(), ncl = (int)cluster_count_x();
    const int J = (p.num_tiles > cid) ? (p.num_tiles - cid + ncl - 1) / ncl : 0;
    const int ncb = L.ncb, dc = L.dc, d = p.d;
    const int64_t K = (int64_t)kHC * d;
    const int U = total_uses(ncb, J, kFull);

    float *sCoef = reinterpret_cast<float *>(smem + L.off_coef);
    float *sPart = reinterpret_cast<float *>(smem + L.off_part);
    float *sMma = reinterpret_cast<float *>(smem + L.off_mma);
    float *sNormW = reinterpret_cast<float *>(smem + L.off_normw);
    uint32_t *sTmem = reinterpret_cast<uint32_t *>(smem + L.off_tmem);
    const uint32_t bar0 = smem_u32(smem + L.off_bar);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kSlots + s); };
    auto part_bar = [&](int b) { return bar0 + 8u * (2 * kSlots + b); };
    auto coef_bar = [&](int b) { return bar0 + 8u * (2 * kSlots + kBufs + b); };
    // the MMA warps hand each tile's partial dots to the sender warp (full), which
    // hands the buffer back once it has sent them (free)
    const uint32_t mma_full = bar0 + 8u * (2 * kSlots + 2 * kBufs);
    const uint32_t mma_free = bar0 + 8u * (2 * kSlots + 2 * kBufs + 1);
    // the CUDA-core warps hand each tile's sums of squares to the sender warp
    auto ss_bar = [&](int b) { return bar0 + 8u * (2 * kSlots + 2 * kBufs + 2 + b); };
    // this CTA's slice of hc_fn, bulk-copied into the (still empty) ring at launch
    // (wload), and the MMA warps done reading it from there (wfree)
    const uint32_t wload_bar = bar0 + 8u * (2 * kSlots + 2 * kBufs + 4);
    const uint32_t wfree_bar = bar0 + 8u * (2 * kSlots + 2 * kBufs + 5);
    float *sSS = reinterpret_cast<float *>(smem + L.off_ss);
    const uint32_t slot0 = smem_u32(smem);

    if (threadIdx.x == kWarpProducer * 32) {
        s_abort = 0;
        for (int s = 0; s < kSlots; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), kMmaWarps + kCudaWarps);
        }
        for (int b = 0; b < kBufs; ++b) {
            // per tile, from each of the 16 CTAs: the 2 sender lanes serving this owner
            mbar_init(part_bar(b), kC * 2);
            // per tile, from each of the 16 owners: 2 reducer lanes
            mbar_init(coef_bar(b), kC * 2);
        }
        for (int b = 0; b < 2; ++b) mbar_init(ss_bar(b), kT);  // one lane per token
        mbar_init(mma_full, kMmaWarps * 32);
        mbar_init(mma_free, 32);
        mbar_init(wload_bar, 1);
        mbar_init(wfree_bar, kMmaWarps);
        fence_mbar_init_cluster();
        prefetch_tmap(&tm_x);
        if (kFull) prefetch_tmap(&tm_f);
    }
    if (warp == kWarpMma) {  // one warp owns the tensor-memory allocation
        tmem_alloc(smem_u32(sTmem), kTmemCols);
        tmem_relinquish();
    }
    if (kFull)
        for (int c = threadIdx.x; c < dc; c += kThreads) sNormW[c] = __ldg(p.norm_w + rank * dc + c);
    tmem_fence_before_sync();
    cluster_sync_all();  // barriers initialised and visible cluster-wide; TMEM allocated
    tmem_fence_after_sync();
    const uint32_t tmem_base = *sTmem;

    if (warp < kWarpMma + kMmaWarps) {
        // ------------------------------------------------------------ tensor-core projection
        const int s = warp - kWarpMma;  // this warp's stream
        const int g = lane >> 2, t = lane & 3;
        // B fragments of the resident weights in TMEM lane 32*s + lane: k16 step
        // q (columns 16q .. 16q + 15 of this CTA's slice of stream s) occupies
        // TMEM columns 18q .. 18q + 17 as, per n-tile nt, the bf16x2 pairs
        // hi(b0), hi(b1), mid(b0), mid(b1), lo(b0), lo(b1) of
        // W[nt*8+g][k0+2t, k0+2t+1] (b0) and W[nt*8+g][k0+8+2t, k0+9+2t] (b1).
        const uint32_t tw = tmem_base + ((uint32_t)(32 * (warp & 3)) << 16);
        // the slice was bulk-copied into the ring at launch: row i of stream s at floats (s*24 + i) * dc
        const bool wok = mbar_wait_warp<false>(wload_bar, 0u, &s_abort);
        const float *wsm = reinterpret_cast<const float *>(smem) + (int64_t)s * kMix * dc;
        for (int q = 0; wok && q < dc / 16; ++q) {  // k16 step q = columns 16q .. 16q + 15 of the slice
            const int col = 16 * q + 2 * t;
#pragma unroll
            for (int nt = 0; nt < 3; ++nt) {
                const float *wr = wsm + (nt * 8 + g) * dc + col;
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
        tmem_wait_st();
        // every value read from the ring has gone into tensor memory: the ring is the producer's
        __threadfence_block();
        __syncwarp();
        if (lane == 0) mbar_arrive(wfree_bar);
        float acc[4][3][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 3; ++b)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[a][b][c] = 0.0f;
        int tiles_done = 0;
        for (int u = 0; wok && u < U; ++u) {
            const int slot = u % kSlots;
            const uint32_t ph = (uint32_t)(u / kSlots) & 1u;
            if (!mbar_wait_warp<false>(full_bar(slot), ph, &s_abort)) break;
            const Use us = decode_use(u, ncb, J, kFull);
            if (!us.p3) {
                const uint32_t box = slot0 + slot * kSlotBytes + s * kBoxBytes;
#pragma unroll
                for (int hp = 0; hp < kStepsPerSlot / 2; ++hp) {  // pairs of k16 steps
                    uint32_t bw[36];
                    tmem_ld36(tw + kWCols * (us.cb * kStepsPerSlot + 2 * hp), bw);
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
            }
            // The slot's last ldmatrix loads may still be in flight here: nothing
            // forces the mma.sync that consumes them ahead of the arrive, and an
            // mbarrier arrive does not wait for loads.  A CTA-scope fence completes
            // them before the producer may refill the slot.
            __threadfence_block();
            __syncwarp();
            if (lane == 0) mbar_arrive(empty_bar(slot));
            if (!us.p3 && us.cb == ncb - 1) {
                // tile finished: hand this warp's partial dots of the tile's 64 tokens
                // to the sender warp, once it has drained the previous tile's
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
    } else if (warp == kWarpProducer) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_keep = policy_evict_last(), pol_stream = policy_evict_first();
            int armed = 0;
            // the slice of hc_fn into the ring (4 streams x 24 rows of dc floats); the ring
            // is used for streaming once the MMA warps have moved it into tensor memory
            mbar_arrive_expect_tx(wload_bar, (uint32_t)(kHC * kMix * dc * 4));
            for (int s = 0; s < kHC; ++s)
                for (int i = 0; i < kMix; ++i)
                    bulk_load(slot0 + (uint32_t)((s * kMix + i) * dc * 4),
                              p.hc_fn + (int64_t)i * K + (int64_t)s * d + (int64_t)rank * dc,
                              (uint32_t)(dc * 4), wload_bar);
            const bool wok = mbar_wait<false>(wfree_bar, 0u, &s_abort);
            for (int u = 0; wok && u < U; ++u) {
                const int slot = u % kSlots;
                const uint32_t ph = (uint32_t)(u / kSlots) & 1u;
                if (!mbar_wait<false>(empty_bar(slot), ph ^ 1u, &s_abort)) break;
                const Use us = decode_use(u, ncb, J, kFull);
                const int tile = cid + us.j * ncl;
                const int row = tile * kT;
                const int col = (int)rank * dc + us.cb * kCB;
                const uint32_t dst = slot0 + slot * kSlotBytes;
                // the tile's pre_mix rows travel with its first phase-1 slot
                const bool with_pm = kFull && !us.p3 && us.cb == 0;
                const int64_t rows_left = p.n - (int64_t)row;
                const uint32_t pm_bytes = with_pm ? 16u * (uint32_t)(rows_left < kT ? rows_left : kT) : 0u;
                mbar_arrive_expect_tx(full_bar(slot), (us.p3 ? kSlotBytes : kStageXBytes) + pm_bytes);
                if (with_pm)
                    bulk_load(smem_u32(smem + L.off_pm) + (us.j % kPmBufs) * kT * 16,
                              p.pre_mix + (int64_t)row * kHC, pm_bytes, full_bar(slot));
                for (int s = 0; s < kHC; ++s)
                    tma_load_2d(dst + s * kBoxBytes, &tm_x, full_bar(slot), s * d + col, row,
                                us.p3 ? pol_stream : pol_keep);
                if (us.p3) tma_load_2d(dst + kStageXBytes, &tm_f, full_bar(slot), col, row, pol_stream);
                armed = u + 1;
            }
            // no copy may still be landing when the CTA leaves: wait (bounded) for the
            // last armed uses of every slot
            for (int u = (armed > kSlots ? armed - kSlots : 0); u < armed; ++u)
                mbar_wait<false>(full_bar(u % kSlots), (uint32_t)(u / kSlots) & 1u, &s_abort);
        }
    } else if (warp == kWarpReducer) {
        // ------------------------------------------------------------ owner: statistics + Sinkhorn
        // Lanes 8*tl .. 8*tl + 7 serve owned token tl: each sums two of the 16
        // sources, a 3-step shuffle finishes the sums, and all 8 lanes then run
        // the same split + Sinkhorn (fast flavour) so any of them can broadcast.
        const float s0 = __ldg(p.hc_scale), s1 = __ldg(p.hc_scale + 1), s2 = __ldg(p.hc_scale + 2);
        const int tl = lane >> 3, sub = lane & 7;
        for (int j = 0; j < J; ++j) {
            const int buf = j % kBufs;
            if (!mbar_wait_warp<true>(part_bar(buf), (uint32_t)(j / kBufs) & 1u, &s_abort)) break;
            const int tile = cid + j * ncl;
            const int tk = (int)rank * kTokPerOwner + tl;
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
            {
                // broadcast first: lane l -> destination CTA l % 16, tokens 2*(l/16) + {0, 1}.
                // Without phase 3 (hc_mixes) the data goes unused, but the arrivals still
                // pace the CUDA-core warps, which keeps every hand-off buffer in order.
                const int dest = lane & 15;
                const int ta = 2 * (lane >> 4);
#pragma unroll
                for (int k2 = 0; k2 < 2; ++k2) {
                    const int tsel = ta + k2;  // owned token whose coefficients to send
                    const int srcl = 8 * tsel;  // a lane that computed them
                    float v[kCoefF];
#pragma unroll
                    for (int i = 0; i < kCoefF; ++i) v[i] = 0.0f;
#pragma unroll
                    for (int k = 0; k < kHC; ++k) v[k] = __shfl_sync(0xffffffffu, po[k], srcl);
#pragma unroll
                    for (int i = 0; i < kHC * kHC; ++i) v[kHC + i] = __shfl_sync(0xffffffffu, c[i], srcl);
                    v[kHC + kHC * kHC] = __shfl_sync(0xffffffffu, rs_h, srcl);
                    const int trow = (int)rank * kTokPerOwner + tsel;
                    const uint32_t dst = mapa(smem_u32(sCoef + (buf * kT + trow) * kCoefF), dest);
#pragma unroll
                    for (int q = 0; q < kCoefF / 4; ++q)
                        st_cluster_v4(dst + 16 * q, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                }
                mbar_arrive_remote(mapa(coef_bar(buf), dest));
            }
            // then this tile's global outputs (after the release above, not before it)
            if (sub == 0 && tok < p.n) {
                if (p.pre_out) reinterpret_cast<float4 *>(p.pre_out)[tok] = make_float4(pr[0], pr[1], pr[2], pr[3]);
                if (p.post_out) reinterpret_cast<float4 *>(p.post_out)[tok] = make_float4(po[0], po[1], po[2], po[3]);
                if (p.comb_out) {
                    float4 *cd = reinterpret_cast<float4 *>(p.comb_out + tok * kHC * kHC);
#pragma unroll
                    for (int q = 0; q < 4; ++q) cd[q] = make_float4(c[4 * q], c[4 * q + 1], c[4 * q + 2], c[4 * q + 3]);
                }
                if (p.mixes_out) {
                    float4 *md = reinterpret_cast<float4 *>(p.mixes_out + tok * kMix);
#pragma unroll
                    for (int q = 0; q < kMix / 4; ++q) md[q] = make_float4(mm[4 * q], mm[4 * q + 1], mm[4 * q + 2], mm[4 * q + 3]);
                }
            }
        }
    } else if (warp == kWarpSender) {
        // ------------------------------------------------------------ partial sums -> owners
        // Per tile: wait for the four MMA warps' partial dots and the CUDA-core
        // warps' sums of squares, add them up and send each token's numbers to its
        // owner CTA, then hand the partial buffer back to the MMA warps.  Lane l
        // serves tokens 2l and 2l + 1, which have the same owner.  This warp makes no
        // global stores, so its cluster-scope releases do not wait on any.
        for (int j = 0; j < J; ++j) {
            if (!mbar_wait_warp<false>(mma_full, (uint32_t)j & 1u, &s_abort)) break;
            if (!mbar_wait_warp<false>(ss_bar(j & 1), (uint32_t)(j >> 1) & 1u, &s_abort)) break;
            const int buf = j % kBufs;
            const int owner = lane >> 1;
#pragma unroll
            for (int i2 = 0; i2 < 2; ++i2) {
                const int tk = 2 * lane + i2;  // token within the tile
                const int tl = tk % kTokPerOwner;
                float v[kPartF];
#pragma unroll
                for (int i = 0; i < kMix; ++i) v[i] = 0.0f;
#pragma unroll
                for (int w = 0; w < kMmaWarps; ++w) {
                    const float *e = sMma + (w * kT + tk) * kMix;
#pragma unroll
                    for (int i = 0; i < kMix; ++i) v[i] += e[i];
                }
                const float2 ss = *reinterpret_cast<const float2 *>(sSS + ((j & 1) * kT + tk) * 2);
                v[kMix] = ss.x;
                v[kMix + 1] = ss.y;
                v[kMix + 2] = v[kMix + 3] = 0.0f;
                const uint32_t dst = mapa(smem_u32(sPart + ((buf * kC + rank) * kTokPerOwner + tl) * kPartF), owner);
#pragma unroll
                for (int q = 0; q < kPartF / 4; ++q)
                    st_cluster_v4(dst + 16 * q, v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
            }
            mbar_arrive_remote(mapa(part_bar(buf), owner));
            mbar_arrive(mma_free);  // this lane's reads of the partial buffer are done
        }
    } else {
        // ------------------------------------------------------------ CUDA-core streaming math
        // 256 threads; per slot, each thread handles one token row r and the
        // 8-column units uu + 4i (i < kItems), as four packed fp32 pairs per stream.
        // Warp w covers rows 8w .. 8w + 7; each quarter-warp takes rows r and r + 4,
        // whose 16-byte units the 128-byte swizzle puts on complementary halves of
        // the banks, so its 16-byte loads are free of bank conflicts.
        // The slot's data is copied to registers and the slot released at once, so
        // the ring reloads while this warp computes; outputs go out with 16-byte
        // global stores.
        const int tc = threadIdx.x - kWarpCuda * 32;  // 0..255
        const int uu = lane & 3;
        const int r = 8 * (tc >> 5) + (lane >> 3) + 4 * ((lane >> 2) & 1);
        const uint64_t pol_out = HC_STORE_EVICT_FIRST ? policy_evict_first() : policy_evict_normal();
        const float4 *sPm = reinterpret_cast<const float4 *>(smem + L.off_pm);
        // One block = the ncb slots of one phase of one tile.  Registers are scoped
        // per block: the coefficients live only through a phase-3 block, and
        // phase 1 keeps one sum-of-squares accumulator per stream (short chains).
        const int nblk = kFull ? 2 * J : J;
        int u = 0;  // ring use index
        bool ok = true;
        for (int b = 0; b < nblk && ok; ++b) {
            const Use bu = block_use(b, J, kFull);
            const int tile = cid + bu.j * ncl;
            const int64_t tok = (int64_t)tile * kT + r;
            const bool live = tok < p.n;
            if (!kFull && b > kLag) {
                // Phase 1 alone: wait, as phase 3 would, for the coefficients of tile
                // b - kLag - 1 before starting tile b, so that no hand-off buffer (the
                // sums of squares here, the partials at the owners) is refilled before
                // it has been read.
                const int jw = b - kLag - 1;
                if (!mbar_wait_warp<true>(coef_bar(jw % kBufs), (uint32_t)(jw / kBufs) & 1u, &s_abort)) break;
            }
            if (!bu.p3) {
                f32x2 pm[kHC];
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
                    const uint8_t *sb = smem_ring + slot * kSlotBytes;
                    uint4 xr[kItems][kHC];
#pragma unroll
                    for (int it = 0; it < kItems; ++it)
#pragma unroll
                        for (int s = 0; s < kHC; ++s)
                            xr[it][s] = *reinterpret_cast<const uint4 *>(sb + s * kBoxBytes + swz(r, uu + 4 * it));
                    if (kFull && cb == 0) {
                        // pre_mix of this thread's token (copied in with this slot)
                        const float4 v = live ? sPm[(bu.j % kPmBufs) * kT + r] : make_float4(0.f, 0.f, 0.f, 0.f);
                        pm[0] = f2_dup(v.x); pm[1] = f2_dup(v.y); pm[2] = f2_dup(v.z); pm[3] = f2_dup(v.w);
                    }
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
                            if (kFull) {
                                f32x2 h = f2_mul(pm[0], xs[0]);
                                h = f2_fma(pm[1], xs[1], h);
                                h = f2_fma(pm[2], xs[2], h);
                                h = f2_fma(pm[3], xs[3], h);
                                const f32x2 hr = f2_from_bf16x2(f2_to_bf16x2(h));
                                ssh2[it] = f2_fma(hr, hr, ssh2[it]);
                            }
                        }
                    }
                    // The slot goes once every value loaded from it has been used.  A
                    // release right after the loads, behind a CTA-scope fence, still let
                    // the ring refill the slot under a warp's loads (measured on the
                    // kernel of hc_slices.cu, whose phase 1 is this code).
                    __threadfence_block();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(empty_bar(slot));
                }
                if (!ok) break;
                // tile finished: this CTA's sums of squares of the token go to the sender
                float ssx = f2_hsum(f2_add(f2_add(ssx2[0], ssx2[1]), f2_add(ssx2[2], ssx2[3])));
                float ssh = f2_hsum(f2_add(ssh2[0], ssh2[1]));
                ssx += __shfl_xor_sync(0xffffffffu, ssx, 1);
                ssx += __shfl_xor_sync(0xffffffffu, ssx, 2);
                ssh += __shfl_xor_sync(0xffffffffu, ssh, 1);
                ssh += __shfl_xor_sync(0xffffffffu, ssh, 2);
                if (uu == 0) {
                    *reinterpret_cast<float2 *>(sSS + ((bu.j & 1) * kT + r) * 2) = make_float2(ssx, ssh);
                    mbar_arrive(ss_bar(bu.j & 1));
                }
            } else {
                f32x2 pm[kHC];
                float cf[kHC + kHC * kHC];  // post, comb of the token
                f32x2 rs2;                   // RMSNorm scale of the token
                for (int cb = 0; cb < ncb; ++cb, ++u) {
                    const int slot = u % kSlots;
                    if (!mbar_wait_warp<false>(full_bar(slot), (uint32_t)(u / kSlots) & 1u, &s_abort)) {
                        ok = false;
                        break;
                    }
                    const uint8_t *sb = smem_ring + slot * kSlotBytes;
                    uint4 xr[kItems][kHC], fr[kItems];
#pragma unroll
                    for (int it = 0; it < kItems; ++it) {
#pragma unroll
                        for (int s = 0; s < kHC; ++s)
                            xr[it][s] = *reinterpret_cast<const uint4 *>(sb + s * kBoxBytes + swz(r, uu + 4 * it));
                        fr[it] = *reinterpret_cast<const uint4 *>(sb + kStageXBytes + swz(r, uu + 4 * it));
                    }
                    if (cb == 0) {
                        const float4 v = live ? sPm[(bu.j % kPmBufs) * kT + r] : make_float4(0.f, 0.f, 0.f, 0.f);
                        pm[0] = f2_dup(v.x); pm[1] = f2_dup(v.y); pm[2] = f2_dup(v.z); pm[3] = f2_dup(v.w);
                        const int buf = bu.j % kBufs;
                        if (!mbar_wait_warp<true>(coef_bar(buf), (uint32_t)(bu.j / kBufs) & 1u, &s_abort)) {
                            ok = false;
                            break;
                        }
                        const float *c = sCoef + (buf * kT + r) * kCoefF;
#pragma unroll
                        for (int q = 0; q < kHC + kHC * kHC; ++q) cf[q] = c[q];
                        rs2 = f2_dup(c[kHC + kHC * kHC]);
                    }
                    if (live) {
#pragma unroll
                        for (int it = 0; it < kItems; ++it) {
                            const int un = uu + 4 * it;
                            const float4 *nw = reinterpret_cast<const float4 *>(sNormW + cb * kCB + un * 8);
                            const float4 w0 = nw[0], w1 = nw[1];
                            const f32x2 wv[4] = {f2_make(w0.x, w0.y), f2_make(w0.z, w0.w), f2_make(w1.x, w1.y),
                                                 f2_make(w1.z, w1.w)};
                            const int64_t cbase = (int64_t)rank * dc + cb * kCB + un * 8;
                            uint32_t yo[kHC][4], ho[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                f32x2 xs[kHC];
#pragma unroll
                                for (int s = 0; s < kHC; ++s) {
                                    const uint4 &w = xr[it][s];
                                    xs[s] = f2_from_bf16x2(q == 0 ? w.x : q == 1 ? w.y : q == 2 ? w.z : w.w);
                                }
                                const uint4 &fw = fr[it];
                                const f32x2 fv = f2_from_bf16x2(q == 0 ? fw.x : q == 1 ? fw.y : q == 2 ? fw.z : fw.w);
#pragma unroll
                                for (int k = 0; k < kHC; ++k) {
                                    f32x2 a = f2_mul(f2_dup(cf[k]), fv);
#pragma unroll
                                    for (int jj = 0; jj < kHC; ++jj) a = f2_fma(f2_dup(cf[kHC + jj * kHC + k]), xs[jj], a);
                                    yo[k][q] = f2_to_bf16x2(a);
                                }
                                f32x2 h = f2_mul(pm[0], xs[0]);
                                h = f2_fma(pm[1], xs[1], h);
                                h = f2_fma(pm[2], xs[2], h);
                                h = f2_fma(pm[3], xs[3], h);
                                const f32x2 hr = f2_from_bf16x2(f2_to_bf16x2(h));
                                ho[q] = f2_to_bf16x2(f2_mul(f2_mul(hr, rs2), wv[q]));
                            }
                            // outputs are written once and not read here again: keep them from
                            // displacing the tiles of x that phase 3 still has to re-read from L2
#pragma unroll
                            for (int k = 0; k < kHC; ++k)
                                st_global_v4_hint(p.y + (tok * kHC + k) * d + cbase, yo[k][0], yo[k][1], yo[k][2],
                                                  yo[k][3], pol_out);
                            st_global_v4_hint(p.h_norm + tok * d + cbase, ho[0], ho[1], ho[2], ho[3], pol_out);
                        }
                    }
                    // the slot goes once the values loaded from it have been used (see phase 1)
                    __threadfence_block();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(empty_bar(slot));
                }
            }
        }
    }
    __syncwarp();
    tmem_fence_before_sync();
    cluster_sync_all();  // no CTA leaves while a peer may still touch its shared memory
    tmem_fence_after_sync();
    if (warp == kWarpMma) tmem_dealloc(tmem_base, kTmemCols);  // every path ends here
}

}  // namespace cl

// ---------------------------------------------------------------- host side
namespace {

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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

// rows x cols bf16 matrix (row stride `cols` elements), box of kT rows x kCB columns (128-byte swizzle for kCB = 64)
bool make_tmap(CUtensorMap *m, const void *base, int64_t rows, int64_t cols) {
    auto enc = get_encode();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    cuuint32_t box[2] = {(cuuint32_t)cl::kCB, (cuuint32_t)cl::kT};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     cl::kCB == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

struct DevInfo {
    int max_clusters = -1;
};
DevInfo g_dev[64];

}  // namespace

bool cluster_path_supported(int d) {
    if (d % (cl::kC * cl::kCB) != 0 || d <= 0) return false;
    const cl::Layout L = cl::make_layout(d);
    // the weight fragments of one MMA warp must fit its 512 tensor-memory columns,
    // and the CTA must be alone on its SM (it takes the whole tensor memory).  The
    // weight slice is staged at launch over the ring and the coefficient buffers
    // (written only after every CTA of the cluster is past its staging), never over
    // the partial-sum buffers that peers write from the start.
    const bool staged_fits = kHC * kMix * L.dc * 4 <= L.off_part;
    return L.wcols <= (int)cl::kTmemCols && staged_fits && L.total <= 232448 && 2 * L.total > 233472;
}

template <bool kFull>
static cudaError_t launch_cluster_impl(const uint16_t *x, const float *pre_mix, const uint16_t *f,
                                       const float *hc_fn, const float *hc_scale,
                                       const float *hc_base, const float *norm_w, int64_t n, int d,
                                       int iters, float eps, float norm_eps, uint16_t *h_norm,
                                       uint16_t *y, float *pre_out, float *post_out,
                                       float *comb_out, float *mixes_out, cudaStream_t s) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const cl::Layout L = cl::make_layout(d);
    auto kern = cl::k_block_cluster<kFull>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L.total);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl::kC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cfg.blockDim = dim3(cl::kThreads);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = s;
    DevInfo &di = g_dev[dev & 63];
    if (di.max_clusters < 0) {
        cfg.gridDim = dim3(cl::kC * 64);
        int mc = 0;
        e = cudaOccupancyMaxActiveClusters(&mc, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (mc <= 0) return cudaErrorInvalidConfiguration;
        di.max_clusters = mc;
    }
    const int64_t tiles = (n + cl::kT - 1) / cl::kT;
    const int ncl = (int)(tiles < di.max_clusters ? tiles : di.max_clusters);
    cfg.gridDim = dim3(cl::kC * ncl);

    CUtensorMap tmx, tmf;
    if (!make_tmap(&tmx, x, n, (int64_t)kHC * d)) return cudaErrorInvalidValue;
    if (kFull) {
        if (!make_tmap(&tmf, f, n, d)) return cudaErrorInvalidValue;
    } else {
        tmf = tmx;
    }
    cl::Params prm;
    prm.pre_mix = pre_mix;
    prm.hc_fn = hc_fn;
    prm.hc_scale = hc_scale;
    prm.hc_base = hc_base;
    prm.norm_w = norm_w;
    prm.h_norm = h_norm;
    prm.y = y;
    prm.pre_out = pre_out;
    prm.post_out = post_out;
    prm.comb_out = comb_out;
    prm.mixes_out = mixes_out;
    prm.n = n;
    prm.d = d;
    prm.iters = iters;
    prm.eps = eps;
    prm.norm_eps = norm_eps;
    prm.num_tiles = (int)tiles;
    e = cudaLaunchKernelEx(&cfg, kern, tmx, tmf, prm);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

cudaError_t launch_block_cluster(const uint16_t *x, const float *pre_mix, const uint16_t *f,
                                 const float *hc_fn, const float *hc_scale, const float *hc_base,
                                 const float *norm_w, int64_t n, int d, int iters, float eps,
                                 float norm_eps, uint16_t *h_norm, uint16_t *y, float *pre_out,
                                 float *post_out, float *comb_out, float *mixes_out,
                                 cudaStream_t s) {
    if (f)
        return launch_cluster_impl<true>(x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, n, d,
                                         iters, eps, norm_eps, h_norm, y, pre_out, post_out,
                                         comb_out, mixes_out, s);
    return launch_cluster_impl<false>(x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, n, d, iters,
                                      eps, norm_eps, h_norm, y, pre_out, post_out, comb_out,
                                      mixes_out, s);
}

cudaError_t consume_device_error(cudaStream_t s, unsigned int *flag) {
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
