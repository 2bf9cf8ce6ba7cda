/*
 * hc_oracle.c -- plain, slow, single-threaded CPU oracle for the
 * hyper-connection residual path (test infrastructure only).
 *
 * This file is TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and
 * the cpu_baseline / reference legs of bench.py may load it. It shares no
 * code, header, table or helper with the CUDA library, and the CUDA library
 * never links or calls it.
 *
 * Arithmetic: every floating-point step is done in IEEE double precision in
 * plain index order. Inputs are taken as their exact bf16 / fp32 values.
 * Results are rounded to bf16 (round to nearest, ties to even) at exactly the
 * three points where the pages store a bf16 tensor: the hc_pre output, the
 * RMSNorm output and the hc_post output. Nothing is blocked, fused or
 * reordered beyond what the definitions state.
 *
 * Sources (the pages this follows):
 *  [BLOCK]  DeepSeek-V4.1 "Block(layer_id, args)" page, Code section:
 *           Block.hc_mixes, Block.hc_pre, Block.hc_post, Block.forward.
 *  [COMB]   DeepSeek-V4.1 "Stream combination" page, Code section:
 *           hc_split_sinkhorn_kernel and its host wrapper, and the
 *           description of the first and the nineteen later rounds.
 *  [DIAG]   DeepSeek V4.1 Flash diagram: blocks "Cast" (BF16->FP32 exact,
 *           FP32->BF16 to the nearest), "sigma", "2 sigma",
 *           "x + eps_hc", "First Sinkhorn Round", "Sinkhorn Round",
 *           "Mixing Coefficients", "Single-Pass mHC".
 *  [MX]     DeepSeek V4.1 Flash diagram, block "Cast to MXFP8": groups of
 *           32 channels of a row, the UE8M0 scale (the group's largest
 *           magnitude, kept at or above 1e-4, over 448, rounded up to a power
 *           of two), each channel over the scale, kept within [-448, 448],
 *           written as the nearest E4M3 number.
 *  [RMS]    DeepSeek-R1 dossier, RMSNorm records (mean square over the last
 *           axis, multiply by 1/sqrt(mean + eps), then by the learned gain,
 *           then restore the input dtype). The V4.1 RMSNorm body itself is
 *           not on the pages; this is the reading taken.
 *
 * Parity pins: every function here is pinned in tests/test_oracle_pins.py
 * against closed forms, invariants, library routines and brute force.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define HCO_OK 0
#define HCO_EINVAL 1
#define HCO_ENOMEM 2

/* ------------------------------------------------------------------------ */
/* bf16 <-> double.  [DIAG] "Cast": BF16 -> FP32 keeps the value; a wider
 * value written as BF16 becomes the nearest BF16 number (ties: to even, the
 * IEEE default, since the pages do not say). */

double hco_bf16_to_double(uint16_t b)
{
    uint32_t bits = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Round half to even on a non-negative double that is an exact multiple of
 * 1/2 at most in its fractional part's relevant bits (any double works). */
static double round_half_even(double q)
{
    double r = floor(q);
    double frac = q - r; /* exact: q and r are close doubles */
    if (frac > 0.5)
        return r + 1.0;
    if (frac < 0.5)
        return r;
    /* exact tie: pick the even neighbour */
    return (fmod(r, 2.0) == 0.0) ? r : r + 1.0;
}

uint16_t hco_bf16_from_double(double v)
{
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    if (isnan(v))
        return (uint16_t)(sign | 0x7fc0u);
    double a = fabs(v);
    if (isinf(a))
        return (uint16_t)(sign | 0x7f80u);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);  /* a = f * 2^e with f in [0.5, 1) */
    int ex = e - 1; /* a in [2^ex, 2^(ex+1)) */
    if (ex < -126)
        ex = -126; /* bf16 subnormals share the spacing of the smallest normal binade */
    double ulp = ldexp(1.0, ex - 7); /* bf16 keeps 8 significant bits */
    double q = a / ulp;              /* exact: division by a power of two */
    double r = round_half_even(q) * ulp;
    if (r >= ldexp(1.0, 128))
        return (uint16_t)(sign | 0x7f80u); /* beyond the largest finite bf16 */
    float fr = (float)r; /* exact: r has at most 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &fr, sizeof bits);
    return (uint16_t)(sign | (uint16_t)(bits >> 16));
}

/* ------------------------------------------------------------------------ */
/* a1: [BLOCK] Block.hc_mixes.  The four streams of a token are flattened to
 * hc*d values and cast to fp32 (exact).  One statistic per token:
 * r = 1/sqrt(mean(x^2) + norm_eps) over all hc*d values.  The projection
 * onto the (2+hc)*hc rows of hc_fn comes first; the result is then scaled
 * by r:  mixes[t, i] = (sum_k x[t, k] * hc_fn[i, k]) * r.
 * x: [n, hc, d] bf16 bits; hc_fn: [(2+hc)*hc, hc*d] fp32 row-major;
 * mixes: [n, (2+hc)*hc] out. */
int hco_mixes(const uint16_t *x, const float *hc_fn, int64_t n, int hc, int d,
              double norm_eps, double *mixes)
{
    if (n < 0 || hc <= 0 || d <= 0 || (n > 0 && (!x || !hc_fn || !mixes)))
        return HCO_EINVAL;
    const int64_t K = (int64_t)hc * d;
    const int mix = (2 + hc) * hc;
    for (int64_t t = 0; t < n; ++t) {
        const uint16_t *xt = x + t * K;
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double v = hco_bf16_to_double(xt[k]);
            ss += v * v;
        }
        double r = 1.0 / sqrt(ss / (double)K + norm_eps);
        for (int i = 0; i < mix; ++i) {
            const float *w = hc_fn + (int64_t)i * K;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += hco_bf16_to_double(xt[k]) * (double)w[k];
            mixes[t * mix + i] = acc * r;
        }
    }
    return HCO_OK;
}

/* ------------------------------------------------------------------------ */
/* a2 + a3: [COMB] hc_split_sinkhorn.  Per token, with m = mixes[t, :]:
 *   pre[j]  = sigmoid(m[j] * s0 + b[j]) + eps                 ([DIAG] sigma, x + eps_hc)
 *   post[j] = 2 * sigmoid(m[hc + j] * s1 + b[hc + j])         ([DIAG] 2 sigma)
 *   c[j][k] = m[2hc + j*hc + k] * s2 + b[2hc + j*hc + k]
 * First round ([DIAG] "First Sinkhorn Round"): row softmax with the row
 * maximum subtracted, then + eps on every entry, then each column divided by
 * (its sum + eps).  Then (iters - 1) rounds ([DIAG] "Sinkhorn Round"): each
 * row divided by (its sum + eps), then each column divided by (its sum + eps).
 * sigmoid(z) = 1 / (1 + exp(-z)).  Division is true division.
 * mixes: [n, mix]; hc_scale: [3]; hc_base: [mix];
 * pre, post: [n, hc]; comb: [n, hc, hc] (row j = input stream, column k = output stream). */
static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

int hco_split_sinkhorn(const double *mixes, const float *hc_scale, const float *hc_base,
                       int64_t n, int hc, int iters, double eps,
                       double *pre, double *post, double *comb)
{
    if (n < 0 || hc <= 0 || iters < 1 || !hc_scale || !hc_base ||
        (n > 0 && (!mixes || !pre || !post || !comb)))
        return HCO_EINVAL;
    const int mix = (2 + hc) * hc;
    double *c = (double *)malloc(sizeof(double) * (size_t)hc * (size_t)hc);
    double *sum = (double *)malloc(sizeof(double) * (size_t)hc);
    if (!c || !sum) {
        free(c);
        free(sum);
        return HCO_ENOMEM;
    }
    const double s0 = hc_scale[0], s1 = hc_scale[1], s2 = hc_scale[2];
    for (int64_t t = 0; t < n; ++t) {
        const double *m = mixes + t * mix;
        for (int j = 0; j < hc; ++j)
            pre[t * hc + j] = sigmoid(m[j] * s0 + (double)hc_base[j]) + eps;
        for (int j = 0; j < hc; ++j)
            post[t * hc + j] = 2.0 * sigmoid(m[hc + j] * s1 + (double)hc_base[hc + j]);
        for (int j = 0; j < hc; ++j)
            for (int k = 0; k < hc; ++k) {
                int i = 2 * hc + j * hc + k;
                c[j * hc + k] = m[i] * s2 + (double)hc_base[i];
            }
        /* first round: softmax along each row, + eps */
        for (int j = 0; j < hc; ++j) {
            double mx = c[j * hc];
            for (int k = 1; k < hc; ++k)
                if (c[j * hc + k] > mx)
                    mx = c[j * hc + k];
            double s = 0.0;
            for (int k = 0; k < hc; ++k) {
                c[j * hc + k] = exp(c[j * hc + k] - mx);
                s += c[j * hc + k];
            }
            for (int k = 0; k < hc; ++k)
                c[j * hc + k] = c[j * hc + k] / s + eps;
        }
        /* first round: column normalisation */
        for (int k = 0; k < hc; ++k) {
            sum[k] = 0.0;
            for (int j = 0; j < hc; ++j)
                sum[k] += c[j * hc + k];
        }
        for (int j = 0; j < hc; ++j)
            for (int k = 0; k < hc; ++k)
                c[j * hc + k] = c[j * hc + k] / (sum[k] + eps);
        /* the later rounds: rows, then columns */
        for (int it = 1; it < iters; ++it) {
            for (int j = 0; j < hc; ++j) {
                sum[j] = 0.0;
                for (int k = 0; k < hc; ++k)
                    sum[j] += c[j * hc + k];
            }
            for (int j = 0; j < hc; ++j)
                for (int k = 0; k < hc; ++k)
                    c[j * hc + k] = c[j * hc + k] / (sum[j] + eps);
            for (int k = 0; k < hc; ++k) {
                sum[k] = 0.0;
                for (int j = 0; j < hc; ++j)
                    sum[k] += c[j * hc + k];
            }
            for (int j = 0; j < hc; ++j)
                for (int k = 0; k < hc; ++k)
                    c[j * hc + k] = c[j * hc + k] / (sum[k] + eps);
        }
        memcpy(comb + t * hc * hc, c, sizeof(double) * (size_t)hc * (size_t)hc);
    }
    free(c);
    free(sum);
    return HCO_OK;
}

/* ------------------------------------------------------------------------ */
/* a4: [BLOCK] Block.hc_pre.  h[t, c] = bf16( sum_s pre_mix[t, s] * x[t, s, c] ),
 * the sum over the hc streams in fp32 in the pages (fp64 here), then the
 * cast back to the stream dtype ([DIAG] "Cast" FP32 -> BF16). */
int hco_pre(const uint16_t *x, const double *pre_mix, int64_t n, int hc, int d, uint16_t *h)
{
    if (n < 0 || hc <= 0 || d <= 0 || (n > 0 && (!x || !pre_mix || !h)))
        return HCO_EINVAL;
    for (int64_t t = 0; t < n; ++t)
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int s = 0; s < hc; ++s)
                acc += pre_mix[t * hc + s] * hco_bf16_to_double(x[(t * hc + s) * d + c]);
            h[t * d + c] = hco_bf16_from_double(acc);
        }
    return HCO_OK;
}

/* a5: RMSNorm ([RMS]; instantiated as attn_norm / ffn_norm on [BLOCK] with
 * eps = norm_eps).  ms = mean_c h[c]^2; out[c] = bf16( (h[c] / sqrt(ms + eps)) * w[c] ).
 * h is the bf16 hc_pre output; w is fp32. */
int hco_rmsnorm(const uint16_t *h, const float *w, int64_t n, int d, double eps, uint16_t *out)
{
    if (n < 0 || d <= 0 || (n > 0 && (!h || !w || !out)))
        return HCO_EINVAL;
    for (int64_t t = 0; t < n; ++t) {
        double ss = 0.0;
        for (int c = 0; c < d; ++c) {
            double v = hco_bf16_to_double(h[t * d + c]);
            ss += v * v;
        }
        double rs = 1.0 / sqrt(ss / (double)d + eps);
        for (int c = 0; c < d; ++c) {
            double v = hco_bf16_to_double(h[t * d + c]);
            out[t * d + c] = hco_bf16_from_double((v * rs) * (double)w[c]);
        }
    }
    return HCO_OK;
}

/* a6: [BLOCK] Block.hc_post.
 * y[t, k, c] = bf16( post[t, k] * f[t, c] + sum_j comb[t, j, k] * residual[t, j, c] ).
 * Column k of comb feeds output stream k (the broadcast in the pages sums
 * over the input-stream axis j). */
int hco_post(const uint16_t *f, const uint16_t *residual, const double *post, const double *comb,
             int64_t n, int hc, int d, uint16_t *y)
{
    if (n < 0 || hc <= 0 || d <= 0 || (n > 0 && (!f || !residual || !post || !comb || !y)))
        return HCO_EINVAL;
    for (int64_t t = 0; t < n; ++t)
        for (int k = 0; k < hc; ++k)
            for (int c = 0; c < d; ++c) {
                double acc = post[t * hc + k] * hco_bf16_to_double(f[t * d + c]);
                for (int j = 0; j < hc; ++j)
                    acc += comb[(t * hc + j) * hc + k] *
                           hco_bf16_to_double(residual[(t * hc + j) * d + c]);
                y[(t * hc + k) * d + c] = hco_bf16_from_double(acc);
            }
    return HCO_OK;
}

/* ------------------------------------------------------------------------ */
/* One sublayer side of [BLOCK] Block.forward ([DIAG] "Single-Pass mHC"):
 * the coefficients (pre, post, comb) come from this side's x (a1-a3); the
 * sublayer input is x collapsed under the pre_mix handed in from the previous
 * side (a4), normalised (a5); the sublayer output f is expanded back with this
 * side's post and comb (a6).  The pre computed here is returned for the next
 * side.  Here f is an input (the sublayer body is not on the path).
 * Outputs: h_norm [n, d] bf16, y [n, hc, d] bf16, pre/post [n, hc], comb [n, hc, hc], mixes [n, mix]. */
int hco_block_step(const uint16_t *x, const double *pre_mix, const uint16_t *f,
                   const float *hc_fn, const float *hc_scale, const float *hc_base,
                   const float *norm_w, int64_t n, int hc, int d, int iters, double eps,
                   double norm_eps, uint16_t *h_norm, uint16_t *y, double *pre,
                   double *post, double *comb, double *mixes)
{
    if (n < 0 || hc <= 0 || d <= 0 || iters < 1)
        return HCO_EINVAL;
    if (n == 0)
        return HCO_OK;
    int rc;
    rc = hco_mixes(x, hc_fn, n, hc, d, norm_eps, mixes);
    if (rc)
        return rc;
    rc = hco_split_sinkhorn(mixes, hc_scale, hc_base, n, hc, iters, eps, pre, post, comb);
    if (rc)
        return rc;
    uint16_t *h = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)n * (size_t)d);
    if (!h)
        return HCO_ENOMEM;
    rc = hco_pre(x, pre_mix, n, hc, d, h);
    if (!rc)
        rc = hco_rmsnorm(h, norm_w, n, d, norm_eps, h_norm);
    free(h);
    if (rc)
        return rc;
    return hco_post(f, x, post, comb, n, hc, d, y);
}

/* ------------------------------------------------------------------------ */
/* [MX] E4M3 element: sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
 * exponent field 0 holds the subnormals m * 2^-9; the largest finite value is
 * 1.75 * 2^8 = 448 (field 15, mantissa 6).  "Nearest" ties to even (the
 * pages do not say; IEEE default).  |v| <= 448 (the cast clamps first). */
uint8_t hco_e4m3_from_double(double v)
{
    uint8_t sign = signbit(v) ? 0x80u : 0u;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);
    int ex = e - 1; /* a in [2^ex, 2^(ex+1)) */
    if (ex < -6)
        ex = -6; /* subnormals share the spacing of the smallest normal binade */
    double ulp = ldexp(1.0, ex - 3); /* 3 mantissa bits */
    double r = round_half_even(a / ulp) * ulp;
    if (r == 0.0)
        return sign;
    frexp(r, &e);
    ex = e - 1;
    if (ex < -6) /* subnormal: r = m * 2^-9, m in 1..7 */
        return (uint8_t)(sign | (uint8_t)(r / ldexp(1.0, -9)));
    int mant = (int)((r / ldexp(1.0, ex) - 1.0) * 8.0); /* exact */
    return (uint8_t)(sign | (uint8_t)((ex + 7) << 3) | (uint8_t)mant);
}

/* [MX] The cast of bf16 rows, d a multiple of 32.  Per group of 32 channels:
 * amax = the largest |x| (exact), kept at or above 1e-4; the scale is the
 * smallest power of two at or above amax / 448, where 1e-4 and the division
 * are fp32 (the reading taken: the scale is decided in the kernel's fp32);
 * scales[g] = log2(scale) + 127 (UE8M0); codes[c] = E4M3 of x[c] / scale
 * (exact in double), clamped to [-448, 448].
 * in: [rows, d] bf16 bits; codes: [rows, d]; scales: [rows, d/32]. */
int hco_mxfp8(const uint16_t *in, int64_t rows, int d, uint8_t *codes, uint8_t *scales)
{
    if (rows < 0 || d <= 0 || d % 32 != 0 || (rows > 0 && (!in || !codes || !scales)))
        return HCO_EINVAL;
    const int groups = d / 32;
    for (int64_t t = 0; t < rows; ++t) {
        for (int g = 0; g < groups; ++g) {
            const uint16_t *xg = in + t * d + 32 * g;
            float amax = 0.0f;
            for (int i = 0; i < 32; ++i) {
                float a = (float)fabs(hco_bf16_to_double(xg[i]));
                if (a > amax)
                    amax = a;
            }
            if (amax < 1e-4f)
                amax = 1e-4f;
            volatile float q = amax / 448.0f; /* fp32 division, correctly rounded */
            int e;
            float m = frexpf(q, &e); /* q = m * 2^e, m in [0.5, 1) */
            int ex = (m == 0.5f) ? e - 1 : e; /* smallest power of two >= q is 2^ex */
            scales[t * groups + g] = (uint8_t)(ex + 127);
            for (int i = 0; i < 32; ++i) {
                double v = ldexp(hco_bf16_to_double(xg[i]), -ex); /* exact */
                if (v > 448.0)
                    v = 448.0;
                if (v < -448.0)
                    v = -448.0;
                codes[t * d + 32 * g + i] = hco_e4m3_from_double(v);
            }
        }
    }
    return HCO_OK;
}

/* ------------------------------------------------------------------------ */
/* f3: the backward of one side step.  The pages give no backward pass; this
 * is the derivative of a1-a6 exactly as defined above ([BLOCK], [COMB]),
 * token by token, with the parameter gradients summed over tokens in index
 * order.  Inputs are doubles (for the bf16 tensors: their exact values).
 * rnd = 1: the forward's three bf16 casts (h, h_norm, y) are applied as in
 * hco_block_step, and gradients pass through a cast unchanged (its
 * derivative is taken as 1, as for a dtype cast in autograd); rnd = 0: no
 * cast anywhere, so the result is the exact derivative of that unrounded
 * forward (which the pins check with finite differences). */

static double rnd_bf16(double v, int rnd) { return rnd ? hco_bf16_to_double(hco_bf16_from_double(v)) : v; }

/* Sinkhorn with every intermediate kept: S = the row softmax of L; P[0] =
 * S + eps; then steps k = 1 .. 2*iters - 1, a column step for odd k and a row
 * step for even k, each dividing by (sum + eps).  P holds 2*iters matrices. */
static void sinkhorn_ckpt(const double *L, int hc, int iters, double eps, double *S, double *P)
{
    const int q = hc * hc;
    for (int j = 0; j < hc; ++j) {
        double mx = L[j * hc];
        for (int k = 1; k < hc; ++k)
            if (L[j * hc + k] > mx)
                mx = L[j * hc + k];
        double s = 0.0;
        for (int k = 0; k < hc; ++k) {
            S[j * hc + k] = exp(L[j * hc + k] - mx);
            s += S[j * hc + k];
        }
        for (int k = 0; k < hc; ++k) {
            S[j * hc + k] = S[j * hc + k] / s;
            P[j * hc + k] = S[j * hc + k] + eps;
        }
    }
    for (int st = 1; st < 2 * iters; ++st) {
        const double *a = P + (st - 1) * q;
        double *b = P + st * q;
        for (int i = 0; i < hc; ++i) {
            double s = 0.0;
            for (int o = 0; o < hc; ++o)
                s += (st & 1) ? a[o * hc + i] : a[i * hc + o]; /* odd: column i; even: row i */
            for (int o = 0; o < hc; ++o) {
                int idx = (st & 1) ? o * hc + i : i * hc + o;
                b[idx] = a[idx] / (s + eps);
            }
        }
    }
}

/* Reverse of sinkhorn_ckpt: g (the gradient of the last matrix) -> gL. */
static void sinkhorn_back(const double *S, const double *P, int hc, int iters, double eps,
                          double *g, double *gL)
{
    const int q = hc * hc;
    for (int st = 2 * iters - 1; st >= 1; --st) {
        const double *a = P + (st - 1) * q; /* the step's input */
        const double *b = P + st * q;       /* its output */
        for (int i = 0; i < hc; ++i) {
            double s = 0.0, dot = 0.0;
            for (int o = 0; o < hc; ++o) {
                int idx = (st & 1) ? o * hc + i : i * hc + o;
                s += a[idx];
                dot += g[idx] * b[idx];
            }
            /* out = in / D: d(out_o)/d(in_o') = (delta - out_o) / D along the line */
            for (int o = 0; o < hc; ++o) {
                int idx = (st & 1) ? o * hc + i : i * hc + o;
                g[idx] = (g[idx] - dot) / (s + eps);
            }
        }
    }
    /* P[0] = softmax(L) + eps, row by row */
    for (int j = 0; j < hc; ++j) {
        double dot = 0.0;
        for (int k = 0; k < hc; ++k)
            dot += g[j * hc + k] * S[j * hc + k];
        for (int k = 0; k < hc; ++k)
            gL[j * hc + k] = S[j * hc + k] * (g[j * hc + k] - dot);
    }
}

/* The side step on double inputs (any hc), the casts applied when rnd = 1.
 * x [n, hc, d], pre_mix [n, hc], f [n, d], hc_fn [mix, hc*d], hc_scale [3],
 * hc_base [mix], norm_w [d] -> h_norm [n, d], y [n, hc, d], pre, post [n, hc],
 * comb [n, hc, hc]. */
int hco_side_f64(const double *x, const double *pre_mix, const double *f, const double *hc_fn,
                 const double *hc_scale, const double *hc_base, const double *norm_w, int64_t n,
                 int hc, int d, int iters, double eps, double norm_eps, int rnd, double *h_norm,
                 double *y, double *pre, double *post, double *comb)
{
    if (n < 0 || hc <= 0 || hc > 64 || d <= 0 || iters < 1)
        return HCO_EINVAL;
    const int mix = (2 + hc) * hc, q = hc * hc;
    const int64_t K = (int64_t)hc * d;
    double *m = malloc(sizeof(double) * mix), *S = malloc(sizeof(double) * q),
           *P = malloc(sizeof(double) * (size_t)(2 * iters) * q), *h = malloc(sizeof(double) * d);
    if (!m || !S || !P || !h) {
        free(m); free(S); free(P); free(h);
        return HCO_ENOMEM;
    }
    for (int64_t t = 0; t < n; ++t) {
        const double *xt = x + t * K;
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k)
            ss += xt[k] * xt[k];
        const double r = 1.0 / sqrt(ss / (double)K + norm_eps);
        for (int i = 0; i < mix; ++i) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += xt[k] * hc_fn[i * K + k];
            m[i] = acc * r;
        }
        for (int j = 0; j < hc; ++j) {
            pre[t * hc + j] = sigmoid(m[j] * hc_scale[0] + hc_base[j]) + eps;
            post[t * hc + j] = 2.0 * sigmoid(m[hc + j] * hc_scale[1] + hc_base[hc + j]);
        }
        double L[64 * 64];
        for (int i = 0; i < q; ++i)
            L[i] = m[2 * hc + i] * hc_scale[2] + hc_base[2 * hc + i];
        sinkhorn_ckpt(L, hc, iters, eps, S, P);
        memcpy(comb + t * q, P + (size_t)(2 * iters - 1) * q, sizeof(double) * q);
        double sh = 0.0;
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int s = 0; s < hc; ++s)
                acc += pre_mix[t * hc + s] * xt[(int64_t)s * d + c];
            h[c] = rnd_bf16(acc, rnd);
            sh += h[c] * h[c];
        }
        const double rs = 1.0 / sqrt(sh / (double)d + norm_eps);
        for (int c = 0; c < d; ++c)
            h_norm[t * d + c] = rnd_bf16((h[c] * rs) * norm_w[c], rnd);
        for (int k = 0; k < hc; ++k)
            for (int c = 0; c < d; ++c) {
                double acc = post[t * hc + k] * f[t * d + c];
                for (int j = 0; j < hc; ++j)
                    acc += comb[t * q + j * hc + k] * xt[(int64_t)j * d + c];
                y[(t * hc + k) * d + c] = rnd_bf16(acc, rnd);
            }
    }
    free(m); free(S); free(P); free(h);
    return HCO_OK;
}

/* The backward of hco_side_f64.  Upstream gradients g_hn [n, d], g_y
 * [n, hc, d], g_pre [n, hc] (NULL: zero).  Out: g_x [n, hc, d], g_pm [n, hc],
 * g_f [n, d] per token; g_fn [mix, hc*d], g_scale [3], g_base [mix], g_w [d]
 * summed over the tokens. */
int hco_side_backward_f64(const double *x, const double *pre_mix, const double *f,
                          const double *hc_fn, const double *hc_scale, const double *hc_base,
                          const double *norm_w, int64_t n, int hc, int d, int iters, double eps,
                          double norm_eps, const double *g_hn, const double *g_y,
                          const double *g_pre, int rnd, double *g_x, double *g_pm, double *g_f,
                          double *g_fn, double *g_scale, double *g_base, double *g_w)
{
    if (n < 0 || hc <= 0 || hc > 64 || d <= 0 || iters < 1)
        return HCO_EINVAL;
    const int mix = (2 + hc) * hc, q = hc * hc;
    const int64_t K = (int64_t)hc * d;
    double *a = malloc(sizeof(double) * mix), *m = malloc(sizeof(double) * mix),
           *gm = malloc(sizeof(double) * mix), *S = malloc(sizeof(double) * q),
           *P = malloc(sizeof(double) * (size_t)(2 * iters) * q), *h = malloc(sizeof(double) * d),
           *gh = malloc(sizeof(double) * d), *pre = malloc(sizeof(double) * hc),
           *post = malloc(sizeof(double) * hc), *gpost = malloc(sizeof(double) * hc),
           *gcomb = malloc(sizeof(double) * q), *gL = malloc(sizeof(double) * q);
    if (!a || !m || !gm || !S || !P || !h || !gh || !pre || !post || !gpost || !gcomb || !gL) {
        free(a); free(m); free(gm); free(S); free(P); free(h); free(gh); free(pre); free(post);
        free(gpost); free(gcomb); free(gL);
        return HCO_ENOMEM;
    }
    memset(g_fn, 0, sizeof(double) * (size_t)mix * (size_t)K);
    memset(g_scale, 0, sizeof(double) * 3);
    memset(g_base, 0, sizeof(double) * mix);
    memset(g_w, 0, sizeof(double) * d);
    for (int64_t t = 0; t < n; ++t) {
        const double *xt = x + t * K;
        double *gxt = g_x + t * K;
        /* forward, as hco_side_f64 */
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k)
            ss += xt[k] * xt[k];
        const double r = 1.0 / sqrt(ss / (double)K + norm_eps);
        for (int i = 0; i < mix; ++i) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += xt[k] * hc_fn[i * K + k];
            a[i] = acc;
            m[i] = acc * r;
        }
        double L[64 * 64];
        for (int i = 0; i < q; ++i)
            L[i] = m[2 * hc + i] * hc_scale[2] + hc_base[2 * hc + i];
        sinkhorn_ckpt(L, hc, iters, eps, S, P);
        const double *comb = P + (size_t)(2 * iters - 1) * q;
        for (int j = 0; j < hc; ++j)
            post[j] = 2.0 * sigmoid(m[hc + j] * hc_scale[1] + hc_base[hc + j]);
        double sh = 0.0;
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int s = 0; s < hc; ++s)
                acc += pre_mix[t * hc + s] * xt[(int64_t)s * d + c];
            h[c] = rnd_bf16(acc, rnd);
            sh += h[c] * h[c];
        }
        const double rs = 1.0 / sqrt(sh / (double)d + norm_eps);
        /* a6: y_k = post_k f + sum_j comb[j][k] x_j */
        for (int k = 0; k < hc; ++k) {
            gpost[k] = 0.0;
            for (int c = 0; c < d; ++c)
                gpost[k] += f[t * d + c] * g_y[(t * hc + k) * d + c];
        }
        for (int j = 0; j < hc; ++j)
            for (int k = 0; k < hc; ++k) {
                double acc = 0.0;
                for (int c = 0; c < d; ++c)
                    acc += xt[(int64_t)j * d + c] * g_y[(t * hc + k) * d + c];
                gcomb[j * hc + k] = acc;
            }
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int k = 0; k < hc; ++k)
                acc += post[k] * g_y[(t * hc + k) * d + c];
            g_f[t * d + c] = acc;
        }
        for (int j = 0; j < hc; ++j)
            for (int c = 0; c < d; ++c) {
                double acc = 0.0;
                for (int k = 0; k < hc; ++k)
                    acc += comb[j * hc + k] * g_y[(t * hc + k) * d + c];
                gxt[(int64_t)j * d + c] = acc;
            }
        /* a5: h_norm = (h * rs) * w, rs = 1/sqrt(sum h^2 / d + eps) */
        double T = 0.0;
        for (int c = 0; c < d; ++c) {
            const double gu = norm_w[c] * g_hn[t * d + c];
            g_w[c] += (h[c] * rs) * g_hn[t * d + c];
            gh[c] = gu;
            T += h[c] * gu;
        }
        for (int c = 0; c < d; ++c)
            gh[c] = rs * gh[c] - rs * rs * rs / (double)d * h[c] * T;
        /* a4: h = sum_s pre_mix[s] x_s */
        for (int s = 0; s < hc; ++s) {
            double acc = 0.0;
            for (int c = 0; c < d; ++c) {
                acc += xt[(int64_t)s * d + c] * gh[c];
                gxt[(int64_t)s * d + c] += pre_mix[t * hc + s] * gh[c];
            }
            g_pm[t * hc + s] = acc;
        }
        /* a2-a3: pre, post, comb from m */
        for (int j = 0; j < hc; ++j) {
            const double sp = sigmoid(m[j] * hc_scale[0] + hc_base[j]);
            const double gz = (g_pre ? g_pre[t * hc + j] : 0.0) * sp * (1.0 - sp);
            gm[j] = gz * hc_scale[0];
            g_scale[0] += gz * m[j];
            g_base[j] += gz;
            const double sq = sigmoid(m[hc + j] * hc_scale[1] + hc_base[hc + j]);
            const double gq = gpost[j] * 2.0 * sq * (1.0 - sq);
            gm[hc + j] = gq * hc_scale[1];
            g_scale[1] += gq * m[hc + j];
            g_base[hc + j] += gq;
        }
        sinkhorn_back(S, P, hc, iters, eps, gcomb, gL);
        for (int i = 0; i < q; ++i) {
            gm[2 * hc + i] = gL[i] * hc_scale[2];
            g_scale[2] += gL[i] * m[2 * hc + i];
            g_base[2 * hc + i] += gL[i];
        }
        /* a1: m = a * r, a = x . hc_fn^T, r = 1/sqrt(sum x^2 / K + norm_eps) */
        double gr = 0.0;
        for (int i = 0; i < mix; ++i)
            gr += gm[i] * a[i];
        const double cr = -gr * r * r * r / (double)K;
        for (int64_t k = 0; k < K; ++k) {
            double acc = cr * xt[k];
            for (int i = 0; i < mix; ++i)
                acc += gm[i] * r * hc_fn[i * K + k];
            gxt[k] += acc;
        }
        for (int i = 0; i < mix; ++i) {
            const double ga = gm[i] * r;
            for (int64_t k = 0; k < K; ++k)
                g_fn[i * K + k] += ga * xt[k];
        }
    }
    free(a); free(m); free(gm); free(S); free(P); free(h); free(gh); free(pre); free(post);
    free(gpost); free(gcomb); free(gL);
    return HCO_OK;
}
