// hc_device.cuh -- device helpers shared by the libhc kernels (sm_103a).
//
// bf16 packing, the per-token split + Sinkhorn of the 24 mix numbers in
// registers, and block reductions.  The split follows the DeepSeek-V4.1
// "Stream combination" page (hc_split_sinkhorn kernel); the sigmoid / 2 sigma /
// + eps_hc placement follows the DeepSeek V4.1 Flash diagram blocks of the
// same names.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace hc {

constexpr int kHC = 4;                      // streams (hc_mult)
constexpr int kMix = (2 + kHC) * kHC;       // 24 mix numbers per token

// ---------------------------------------------------------------- bf16 helpers
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// Two fp32 -> packed bf16x2 (round to nearest, ties to even); `a` lands in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Unpack 8 bf16 held in a uint4 into 8 floats.
__device__ __forceinline__ void unpack8(const uint4 &v, float (&o)[8]) {
    o[0] = bf16lo(v.x); o[1] = bf16hi(v.x);
    o[2] = bf16lo(v.y); o[3] = bf16hi(v.y);
    o[4] = bf16lo(v.z); o[5] = bf16hi(v.z);
    o[6] = bf16lo(v.w); o[7] = bf16hi(v.w);
}

__device__ __forceinline__ uint4 pack8(const float (&o)[8]) {
    return make_uint4(pack_bf16x2(o[0], o[1]), pack_bf16x2(o[2], o[3]),
                      pack_bf16x2(o[4], o[5]), pack_bf16x2(o[6], o[7]));
}

// ---------------------------------------------------------------- packed fp32 pairs
// Two fp32 lanes in one 64-bit register pair, for the sm_100+ packed
// instructions (add/mul/fma .rn.f32x2).  Each lane rounds exactly like the
// scalar instruction, so results are bitwise those of the scalar code.
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 f2_make(float lo, float hi) {
    f32x2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_split(f32x2 v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ f32x2 f2_dup(float a) { return f2_make(a, a); }
__device__ __forceinline__ f32x2 f2_fma(f32x2 a, f32x2 b, f32x2 c) {
    f32x2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ f32x2 f2_mul(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ f32x2 f2_add(f32x2 a, f32x2 b) {
    f32x2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// packed bf16 pair (element 0 in the low half) -> fp32 pair (exact)
__device__ __forceinline__ f32x2 f2_from_bf16x2(uint32_t v) {
    return f2_make(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}
// fp32 pair -> packed bf16 pair, round to nearest even
__device__ __forceinline__ uint32_t f2_to_bf16x2(f32x2 v) {
    float a, b;
    f2_split(v, a, b);
    return pack_bf16x2(a, b);
}
__device__ __forceinline__ float f2_hsum(f32x2 v) {
    float a, b;
    f2_split(v, a, b);
    return a + b;
}

// ---------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ---------------------------------------------------------------- split + Sinkhorn
// Reciprocal: correctly rounded (__frcp_rn) in the accurate flavour, the
// hardware approximation (rcp.approx.ftz, within 1 ulp) in the fast one.
template <bool kFast>
__device__ __forceinline__ float recip(float x) {
    if constexpr (kFast) {
        float r;
        asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
        return r;
    } else {
        return __frcp_rn(x);
    }
}
template <bool kFast>
__device__ __forceinline__ float expo(float x) {
    if constexpr (kFast) return __expf(x);
    else return expf(x);
}
template <bool kFast>
__device__ __forceinline__ float sigmoid(float z) {
    // 1 / (1 + e^-z); e^-z -> inf gives exactly 0.
    return recip<kFast>(1.0f + expo<kFast>(-z));
}

// One token: 24 mix numbers -> pre[4], post[4], comb[16] (row j = input
// stream, column k = output stream).  First round: row softmax (row maximum
// subtracted) + eps, then each column divided by (its sum + eps).  Then
// (iters - 1) rounds of: each row divided by (its sum + eps), each column
// divided by (its sum + eps).  Division is a reciprocal followed by a
// multiply.  Both flavours stay within 1e-6 of the exact values on the
// workloads here; the fast one has a much shorter dependency chain.
template <bool kFast = false>
__device__ __forceinline__ void split_sinkhorn_token(const float (&m)[kMix], float s0, float s1,
                                                     float s2, const float *__restrict__ base,
                                                     int iters, float eps, float (&pre)[kHC],
                                                     float (&post)[kHC], float (&c)[kHC * kHC]) {
#pragma unroll
    for (int j = 0; j < kHC; ++j) pre[j] = sigmoid<kFast>(fmaf(m[j], s0, base[j])) + eps;
#pragma unroll
    for (int j = 0; j < kHC; ++j) post[j] = 2.0f * sigmoid<kFast>(fmaf(m[kHC + j], s1, base[kHC + j]));
#pragma unroll
    for (int i = 0; i < kHC * kHC; ++i) c[i] = fmaf(m[2 * kHC + i], s2, base[2 * kHC + i]);

    // Pairs of adjacent entries of a row, P[j][h] = (c[j][2h], c[j][2h+1]), for the
    // packed multiplies and column sums.  Every element sees exactly the scalar
    // operations in the scalar order (rows summed left to right, columns top to
    // bottom, then + eps, a reciprocal and a multiply), so the results are those of
    // the plain per-element loops, with fewer instructions.
    static_assert(kHC == 4, "a row is two packed pairs");
    const f32x2 eps2 = f2_dup(eps);
    f32x2 P[kHC][2];
    // first round: row softmax + eps
#pragma unroll
    for (int j = 0; j < kHC; ++j) {
        float mx = c[j * kHC];
#pragma unroll
        for (int k = 1; k < kHC; ++k) mx = fmaxf(mx, c[j * kHC + k]);
        float s = 0.0f;
#pragma unroll
        for (int k = 0; k < kHC; ++k) {
            c[j * kHC + k] = expo<kFast>(c[j * kHC + k] - mx);
            s += c[j * kHC + k];
        }
        const f32x2 r = f2_dup(recip<kFast>(s));
        P[j][0] = f2_fma(f2_make(c[j * kHC], c[j * kHC + 1]), r, eps2);
        P[j][1] = f2_fma(f2_make(c[j * kHC + 2], c[j * kHC + 3]), r, eps2);
    }
    auto columns = [&]() {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const f32x2 sum = f2_add(f2_add(f2_add(f2_add(P[0][h], P[1][h]), P[2][h]), P[3][h]), eps2);
            float s0c, s1c;
            f2_split(sum, s0c, s1c);
            const f32x2 r = f2_make(recip<kFast>(s0c), recip<kFast>(s1c));
#pragma unroll
            for (int j = 0; j < kHC; ++j) P[j][h] = f2_mul(P[j][h], r);
        }
    };
    columns();  // first round: columns
    for (int it = 1; it < iters; ++it) {
#pragma unroll
        for (int j = 0; j < kHC; ++j) {
            float a0, a1, a2, a3;
            f2_split(P[j][0], a0, a1);
            f2_split(P[j][1], a2, a3);
            const f32x2 r = f2_dup(recip<kFast>(((a0 + a1) + a2) + a3 + eps));
            P[j][0] = f2_mul(P[j][0], r);
            P[j][1] = f2_mul(P[j][1], r);
        }
        columns();
    }
#pragma unroll
    for (int j = 0; j < kHC; ++j) {
        f2_split(P[j][0], c[j * kHC], c[j * kHC + 1]);
        f2_split(P[j][1], c[j * kHC + 2], c[j * kHC + 3]);
    }
}

// The same split + Sinkhorn for HC streams (mix = (2 + HC) * HC numbers), in
// plain per-element loops; for HC = 4 the packed version above, which gives
// exactly the same results.
template <int HC, bool kFast = false>
__device__ __forceinline__ void split_sinkhorn_token_hc(const float *m, float s0, float s1, float s2,
                                                        const float *__restrict__ base, int iters,
                                                        float eps, float (&pre)[HC],
                                                        float (&post)[HC], float (&c)[HC * HC]) {
    if constexpr (HC == kHC) {
        float mm[kMix];
#pragma unroll
        for (int i = 0; i < kMix; ++i) mm[i] = m[i];
        split_sinkhorn_token<kFast>(mm, s0, s1, s2, base, iters, eps, pre, post, c);
    } else {
#pragma unroll
        for (int j = 0; j < HC; ++j) pre[j] = sigmoid<kFast>(fmaf(m[j], s0, base[j])) + eps;
#pragma unroll
        for (int j = 0; j < HC; ++j) post[j] = 2.0f * sigmoid<kFast>(fmaf(m[HC + j], s1, base[HC + j]));
#pragma unroll
        for (int i = 0; i < HC * HC; ++i) c[i] = fmaf(m[2 * HC + i], s2, base[2 * HC + i]);
        // first round: row softmax + eps, then columns
#pragma unroll
        for (int j = 0; j < HC; ++j) {
            float mx = c[j * HC];
#pragma unroll
            for (int k = 1; k < HC; ++k) mx = fmaxf(mx, c[j * HC + k]);
            float s = 0.0f;
#pragma unroll
            for (int k = 0; k < HC; ++k) {
                c[j * HC + k] = expo<kFast>(c[j * HC + k] - mx);
                s += c[j * HC + k];
            }
            const float r = recip<kFast>(s);
#pragma unroll
            for (int k = 0; k < HC; ++k) c[j * HC + k] = fmaf(c[j * HC + k], r, eps);
        }
        for (int it = 0; it < iters; ++it) {
            if (it > 0) {
#pragma unroll
                for (int j = 0; j < HC; ++j) {
                    float s = 0.0f;
#pragma unroll
                    for (int k = 0; k < HC; ++k) s += c[j * HC + k];
                    const float r = recip<kFast>(s + eps);
#pragma unroll
                    for (int k = 0; k < HC; ++k) c[j * HC + k] *= r;
                }
            }
#pragma unroll
            for (int k = 0; k < HC; ++k) {
                float s = 0.0f;
#pragma unroll
                for (int j = 0; j < HC; ++j) s += c[j * HC + k];
                const float r = recip<kFast>(s + eps);
#pragma unroll
                for (int j = 0; j < HC; ++j) c[j * HC + k] *= r;
            }
        }
    }
}

}  // namespace hc
