/*
 * hc.h -- C ABI of libhc, the GB300 (sm_103a) implementation of the
 * hyper-connection residual path of a DeepSeek-V4.1-style block.
 *
 * The residual of a token is hc parallel streams of width d (hc = 4,
 * d = 5120 in the released configuration).  Each sublayer side runs:
 *   a1  mixes   = (x_flat . hc_fn^T) * rsqrt(mean(x_flat^2) + norm_eps)
 *   a2  pre     = sigmoid(mixes[0:hc] * s0 + b) + eps,  post = 2 sigmoid(mixes[hc:2hc] * s1 + b)
 *   a3  comb    = Sinkhorn(row softmax + eps of mixes[2hc:] * s2 + b), iters rounds
 *   a4  h       = bf16(sum_s pre_mix[s] * x[s])
 *   a5  h_norm  = bf16(RMSNorm(h) * w)
 *   a6  y[k]    = bf16(post[k] * f + sum_j comb[j][k] * x[j])
 * Sources: DeepSeek-V4.1 "Block(layer_id, args)" page, Code section
 * (Block.hc_mixes, hc_pre, hc_post, forward); DeepSeek-V4.1 "Stream
 * combination" page, Code section (hc_split_sinkhorn); DeepSeek V4.1 Flash
 * diagram (Cast, sigma, 2 sigma, x + eps_hc, First Sinkhorn Round, Sinkhorn
 * Round, Single-Pass mHC blocks); RMSNorm per the DeepSeek-R1 dossier's
 * RMSNorm records (the V4.1 body is not on the pages).
 *
 * Conventions for every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The
 *    library never allocates, frees or retains caller memory, keeps no
 *    state between calls, and never reads or writes outside the extents
 *    stated below.
 *  - Layouts are dense row-major with the innermost index last:
 *      x, residual, y   [n, hc, d]   bf16 (uint16_t bit patterns)
 *      f, h_norm        [n, d]       bf16
 *      hc_fn            [(2+hc)*hc, hc*d] fp32  (row i, column s*d + c)
 *      hc_base          [(2+hc)*hc] fp32,  hc_scale [3] fp32,  norm_w [d] fp32
 *      mixes            [n, (2+hc)*hc] fp32: [pre 0:hc | post hc:2hc | comb 2hc:, row-major j*hc+k]
 *      pre, post, pre_mix  [n, hc] fp32;  comb [n, hc, hc] fp32 (row j = input stream, column k = output stream)
 *  - Every pointer must be 16-byte aligned (HC_ERR_MISALIGNED otherwise).
 *  - Work is enqueued on `stream` (0 = legacy default stream) and is
 *    asynchronous; results are ready when the stream reaches that point.
 *  - Arguments are validated on the host before any launch; an invalid call
 *    launches nothing and returns a non-zero status.  n == 0 is valid and
 *    does nothing.  A failed launch returns HC_ERR_CUDA and records the CUDA
 *    error code for hc_last_cuda_error() (per host thread).
 *  - Compiled stream counts: hc = 2, 4 or 8 (the pages' kernel takes any
 *    hc_mult; the released model uses 4), with d a positive multiple of 64,
 *    d <= 16384; anything else returns HC_ERR_UNSUPPORTED.  The tensor-core
 *    paths of hc_mixes / hc_block_step and the chain (hc_chain_*) serve
 *    hc = 4 with d a multiple of 1024 up to 7168; other shapes run on the
 *    whole-token kernels (the chain refuses them).  The
 *    backward serves all three (tensor-core kernels at hc = 4, plain
 *    per-token kernels at 2 and 8); its no-workspace entry serves hc = 4.
 *  - Output ranges must not overlap input ranges or each other
 *    (HC_ERR_ALIAS), except where an entry point says otherwise.
 */
#ifndef HC_H_
#define HC_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    HC_OK = 0,
    HC_ERR_INVALID_ARG = 1,  /* null pointer, negative size, iters < 1, non-finite or negative eps */
    HC_ERR_UNSUPPORTED = 2,  /* hc not 2, 4 or 8, or d not a multiple of 64 in [64, 16384] */
    HC_ERR_MISALIGNED = 3,   /* a pointer that is not 16-byte aligned */
    HC_ERR_ALIAS = 4,        /* an output range overlaps an input or another output */
    HC_ERR_CUDA = 5,         /* a CUDA runtime call failed; see hc_last_cuda_error() */
    HC_ERR_TIMEOUT = 6       /* a kernel's bounded barrier wait ran out (reported by hc_consume_device_error) */
} hc_status;

/* Static, never-freed description of a status code. */
const char *hc_status_string(hc_status status);

/* The cudaError_t value behind the last HC_ERR_CUDA on this host thread (0 if none). */
int hc_last_cuda_error(void);

/* Library version as major*10000 + minor*100 + patch. */
int hc_version(void);

/*
 * Synchronise `stream`, then report and clear the library's device-side
 * error flag.  Kernels never spin without bound: a barrier wait that runs out
 * (a peer that never arrives) records a flag and the kernel returns early
 * with its outputs incomplete.  Returns HC_ERR_TIMEOUT if any kernel on this
 * device set the flag since the last call, HC_ERR_CUDA if synchronising
 * failed, HC_OK otherwise.  Not part of the method: a health check.
 */
hc_status hc_consume_device_error(cudaStream_t stream);

/*
 * Self-test of the path above: launches one warp that waits on a barrier
 * nothing ever arrives on.  The bounded wait gives up after about half a
 * minute, records the device flag and the kernel returns, leaving the
 * context usable; the next hc_consume_device_error(stream) returns
 * HC_ERR_TIMEOUT.
 * Returns HC_ERR_CUDA if the launch failed, HC_OK otherwise.  Not part of
 * the method.
 */
hc_status hc_selftest_barrier_timeout(cudaStream_t stream);

/*
 * a1-a3 (DeepSeek-V4.1 Block page, Block.hc_mixes, and the "Stream
 * combination" page's hc_split_sinkhorn): from the streams x of n tokens,
 * the 24 mix numbers (one rsqrt statistic over all hc*d values per token,
 * applied after the projection), then pre, post and the Sinkhorn comb.
 *   x          [n, hc, d] bf16            in
 *   hc_fn      [(2+hc)*hc, hc*d] fp32     in
 *   hc_scale   [3] fp32, hc_base [(2+hc)*hc] fp32  in
 *   pre, post  [n, hc] fp32  out;  comb [n, hc, hc] fp32  out
 *   mixes_out  [n, (2+hc)*hc] fp32 out, optional (NULL: not written)
 *   sinkhorn_iters >= 1 (20 in the released model); eps = hc_eps (1e-6);
 *   norm_eps (1e-20).
 */
hc_status hc_mixes(const uint16_t *x, const float *hc_fn, const float *hc_scale,
                   const float *hc_base, int64_t n, int hc, int d, int sinkhorn_iters,
                   float eps, float norm_eps, float *pre, float *post, float *comb,
                   float *mixes_out, cudaStream_t stream);

/*
 * a2-a3 only ("Stream combination" page, hc_split_sinkhorn kernel and
 * wrapper): mixes [n, (2+hc)*hc] fp32 -> pre [n, hc], post [n, hc],
 * comb [n, hc, hc] (all fp32).  pre = sigmoid(m*s0 + b) + eps;
 * post = 2 sigmoid(m*s1 + b); comb = row softmax + eps, one column
 * normalisation, then (iters - 1) rounds of row and column normalisation,
 * each dividing by (sum + eps).  d is not involved.
 */
hc_status hc_split_sinkhorn(const float *mixes, const float *hc_scale, const float *hc_base,
                            int64_t n, int hc, int sinkhorn_iters, float eps, float *pre,
                            float *post, float *comb, cudaStream_t stream);

/*
 * a4 + a5 (Block page, Block.hc_pre then attn_norm / ffn_norm): collapse the
 * streams under pre_mix in fp32, round to bf16, then RMSNorm over d with
 * eps = norm_eps and fp32 gain norm_w, rounding the result to bf16.
 *   x [n, hc, d] bf16, pre_mix [n, hc] fp32, norm_w [d] fp32  in
 *   out [n, d] bf16  out
 */
hc_status hc_pre_norm(const uint16_t *x, const float *pre_mix, const float *norm_w, int64_t n,
                      int hc, int d, float norm_eps, uint16_t *out, cudaStream_t stream);

/*
 * a6 (Block page, Block.hc_post): y[t,k,:] = bf16(post[t,k] * f[t,:] +
 * sum_j comb[t,j,k] * residual[t,j,:]), in fp32.
 *   f [n, d] bf16, residual [n, hc, d] bf16, post [n, hc], comb [n, hc, hc] fp32  in
 *   y [n, hc, d] bf16  out (must not overlap any input)
 */
hc_status hc_post(const uint16_t *f, const uint16_t *residual, const float *post,
                  const float *comb, int64_t n, int hc, int d, uint16_t *y,
                  cudaStream_t stream);

/*
 * One fused side step a1-a6 (Block page, Block.forward; the diagram's
 * "Single-Pass mHC" block): coefficients from this side's x; the sublayer
 * input read with pre_mix handed in from the previous side; the sublayer
 * output f (given) expanded with this side's post and comb.
 *   x [n, hc, d] bf16, pre_mix [n, hc] fp32, f [n, d] bf16, hc_fn, hc_scale,
 *   hc_base, norm_w (as above)                                        in
 *   h_norm [n, d] bf16     out: RMSNorm(hc_pre(x, pre_mix)) -- the sublayer input
 *   y [n, hc, d] bf16      out: hc_post(f, x, post, comb) -- the next residual
 *   pre_out [n, hc] fp32   out: this side's pre (the next side's pre_mix)
 *   post_out [n, hc], comb_out [n, hc, hc] fp32  out, optional (NULL: not written)
 * In a model f depends on h_norm; this fused form takes f as an input (the
 * sublayer body is not part of this path).
 */
hc_status hc_block_step(const uint16_t *x, const float *pre_mix, const uint16_t *f,
                        const float *hc_fn, const float *hc_scale, const float *hc_base,
                        const float *norm_w, int64_t n, int hc, int d, int sinkhorn_iters,
                        float eps, float norm_eps, uint16_t *h_norm, uint16_t *y,
                        float *pre_out, float *post_out, float *comb_out,
                        cudaStream_t stream);

/*
 * The backward of one side step a1-a6 (hc = 2, 4 or 8).  The pages give no backward
 * pass; this is the derivative of hc_block_step's definition (Block page,
 * Code section; "Stream combination" page), with the three bf16 casts (h,
 * h_norm, y) passing gradients through unchanged (as a dtype cast does in
 * autograd) and the forward's rounded h used where the forward used it.
 * Every gradient tensor is fp32.
 *   x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w as hc_block_step     in
 *   g_h_norm [n, d], g_y [n, hc, d]: the gradients of h_norm and y        in
 *   g_pre [n, hc]: the gradient of pre (the next side's pre_mix); NULL: 0 in
 *   g_x [n, hc, d], g_pre_mix [n, hc], g_f [n, d]                        out
 *   g_hc_fn [mix, hc*d], g_hc_scale [3], g_hc_base [mix], g_norm_w [d]:
 *   summed over the n tokens (overwritten, not accumulated)             out
 *   workspace: device scratch of at least
 *   hc_block_step_backward_workspace_bytes(n, hc, d) bytes, 16-byte
 *   aligned, owned by the caller (the library allocates nothing); at hc = 4
 *   that is 4 * (156 n + B (24 * 4d + d + 32) + 160 d) bytes, B = ceil(n / 1024):
 *   a 156-float record per token, then per block of 1,024 tokens the partial
 *   sums of g_hc_fn, g_norm_w and g_hc_base / g_hc_scale, then hc_fn split
 *   into three bf16 parts for the tensor cores (80 rows of 4d bf16)
 * Results are deterministic: the token sums run in a fixed order.
 * sinkhorn_iters must be in [1, 128] (HC_ERR_INVALID_ARG otherwise).
 */
size_t hc_block_step_backward_workspace_bytes(int64_t n, int hc, int d);

/*
 * hc_block_step_backward without a caller workspace: the scratch is a fixed
 * 64 MiB array in device memory that is part of the library's module, so the
 * call allocates nothing.  hc = 4 only.  Inputs whose workspace would not fit
 * (for d = 5120, more than 24,576 tokens) return HC_ERR_UNSUPPORTED.  There is one such
 * array per process and device: calls must not overlap in time (for
 * instance, issue them on one stream).  Results equal
 * hc_block_step_backward's bit for bit.
 */
hc_status hc_block_step_backward_no_workspace(
    const uint16_t *x, const float *pre_mix, const uint16_t *f, const float *hc_fn,
    const float *hc_scale, const float *hc_base, const float *norm_w, int64_t n, int hc, int d,
    int sinkhorn_iters, float eps, float norm_eps, const float *g_h_norm, const float *g_y,
    const float *g_pre, float *g_x, float *g_pre_mix, float *g_f, float *g_hc_fn, float *g_hc_scale,
    float *g_hc_base, float *g_norm_w, cudaStream_t stream);

hc_status hc_block_step_backward(const uint16_t *x, const float *pre_mix, const uint16_t *f,
                                 const float *hc_fn, const float *hc_scale, const float *hc_base,
                                 const float *norm_w, int64_t n, int hc, int d, int sinkhorn_iters,
                                 float eps, float norm_eps, const float *g_h_norm, const float *g_y,
                                 const float *g_pre, float *g_x, float *g_pre_mix, float *g_f,
                                 float *g_hc_fn, float *g_hc_scale, float *g_hc_base,
                                 float *g_norm_w, void *workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

/*
 * The MXFP8 cast (DeepSeek V4.1 Flash diagram, block "Cast to MXFP8"): the
 * rounding the released code runs in front of every FP8/FP4-weight
 * projection, here for the sublayer input h_norm.  The channels of a row are
 * cut into groups of 32.  Per group, scale = the smallest power of two at or
 * above max(amax, 1e-4) / 448, amax the largest |x| of the group, the
 * division in fp32 (correctly rounded); every channel is written as the E4M3
 * number (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no infinity)
 * nearest to x / scale, ties to even, after clamping x / scale to
 * [-448, 448].  The value a code stands for is its E4M3 value times the
 * group's scale.  NaN or infinite inputs are outside the cast's definition.
 *
 * hc_mxfp8_cast: bf16 rows of any origin.
 *   in [rows, d] bf16, d a multiple of 32 (else HC_ERR_UNSUPPORTED)     in
 *   codes [rows, d] uint8: the E4M3 byte of every channel             out
 *   scales [rows, d/32] uint8: log2(scale) + 127 per group (UE8M0)     out
 *   in and codes 16-byte aligned; scales byte-aligned.
 *
 * hc_pre_norm_mxfp8: a4 + a5 as hc_pre_norm computes them, then the cast of
 * the bf16 h_norm in the same pass (nothing written to HBM in between).
 *   x, pre_mix, norm_w as hc_pre_norm                                  in
 *   h_norm_out [n, d] bf16, optional (NULL: not written); when given it
 *   equals hc_pre_norm's output bit for bit                            out
 *   codes [n, d], scales [n, d/32] as for hc_mxfp8_cast of h_norm      out
 */
hc_status hc_mxfp8_cast(const uint16_t *in, int64_t rows, int d, uint8_t *codes, uint8_t *scales,
                        cudaStream_t stream);

hc_status hc_pre_norm_mxfp8(const uint16_t *x, const float *pre_mix, const float *norm_w, int64_t n,
                            int hc, int d, float norm_eps, uint16_t *h_norm_out, uint8_t *codes,
                            uint8_t *scales, cudaStream_t stream);

/*
 * A chain of fused side steps, fused across sides (the Block page's
 * Block.forward: the streams a side reads are the y the previous side wrote,
 * and each side reads its sublayer input with the previous side's pre).  The
 * results equal, bit for bit, those of calling hc_block_step side after side;
 * each launch reads its side's streams from HBM once.  Supported when d is a
 * multiple of 1024 and d <= 7168, with hc = 4 (HC_ERR_UNSUPPORTED otherwise).
 *
 * State buffers.  A state buffer is hc_chain_state_bytes(n, hc, d) bytes of
 * device memory owned by the caller (16-byte aligned).  It starts with the
 * coefficient rows, HC_STATE_FLOATS = 32 fp32 per token:
 *   [0:4] post, [4:20] comb (row-major j*hc+k), [20] RMSNorm scale
 *   rsqrt(mean(h^2) + norm_eps), [21:24] zero, [24:28] pre (the side's pre:
 *   the next side's pre_mix), [28:32] pre_mix (the one the side reads with);
 * the rest is the kernels' scratch for one launch (partial sums of the
 * cross-slice reductions, their arrival flags and the launch's epoch;
 * nothing in it needs clearing).  The caller keeps two buffers in rotation: side i reads the rows
 * of side i and writes the buffer of side i + 1 (the two may not overlap:
 * HC_ERR_ALIAS).  No cited passage has a counterpart for the state: it
 * carries one side's coefficients to the next launch.
 *
 * Two orders of work are served:
 *  - given the sublayer outputs f up front (the benchmark form): every
 *    hc_chain_side launch writes side i's h_norm and y;
 *  - model order (f_i = sublayer(h_norm_i)): hc_chain_side writes side i's y
 *    and side i + 1's bf16 h (h_pre_out, hc_pre of that y with side i's pre)
 *    with its RMSNorm statistic in the next state; hc_chain_norm then turns
 *    that h into h_norm_{i+1} (and / or its MXFP8 cast) for the sublayer, whose
 *    output is the next launch's f.  hc_chain_begin writes the first side's h
 *    the same way.  Every h_norm equals hc_block_step's bit for bit.
 *
 * hc_chain_begin: a1-a3 of the first side and its RMSNorm statistic.
 *   x [n, hc, d] bf16, pre_mix [n, hc] fp32, hc_fn, hc_scale, hc_base of the
 *   first side                                                       in
 *   state_out, state_bytes   out: state buffer of the first side
 *   pre_out [n, hc] fp32     out, optional (NULL: not written): its pre
 *   h_pre_out [n, d] bf16    out, optional: its bf16 h = hc_pre(x, pre_mix)
 *
 * hc_chain_side: a4-a6 of side i from its state, fused with a1-a3 of side
 * i + 1 on the y it produces.
 *   x [n, hc, d] bf16 (side i's streams), f [n, d] bf16, state_in (side i's
 *   state buffer; its first n rows are read), norm_w [d] (side i),
 *   hc_fn_next, hc_scale_next, hc_base_next (side i + 1; all three NULL for
 *   the last side)                                                    in
 *   y [n, hc, d] bf16        out: as hc_block_step's
 *   h_norm [n, d] bf16       out, optional: side i's, as hc_block_step's
 *   state_out, state_bytes   out: state buffer of side i + 1 (unused for the last side)
 *   pre_out [n, hc] fp32     out, optional: side i + 1's pre
 *   h_pre_out [n, d] bf16    out, optional: side i + 1's bf16 h; needs the
 *   next side's weights and excludes h_norm (HC_ERR_INVALID_ARG)
 *
 * hc_chain_norm: a5 in model order.  h_norm = bf16((h * rs) * norm_w) with
 * rs the RMSNorm scale in the state's rows (what hc_block_step computes).
 *   h_pre [n, d] bf16, state (n rows), norm_w [d] fp32                 in
 *   h_norm [n, d] bf16, optional                                       out
 *   codes [n, d], scales [n, d/32] uint8, optional pair: the MXFP8 cast of
 *   h_norm as hc_mxfp8_cast computes it                                out
 *   At least one of h_norm and codes; d a multiple of 64.
 *
 * Launch notes.  The chain kernels run one CTA on each of 16 * floor(SMs / 16)
 * SMs; hc_chain_begin and hc_chain_side with the next side's weights launch
 * cooperatively: they need that many SMs free to start, and a CTA waits
 * (bounded) on flags other CTAs write into the state buffer.
 * The flags carry an epoch that a one-thread kernel, enqueued just before
 * each hc_chain_begin / hc_chain_side launch, writes into the state buffer
 * from a device counter; so the chain, like every other entry point, can be
 * recorded into a CUDA graph and replayed (after one call outside the
 * capture, which sets the kernels' attributes and caches the device's SM and
 * cluster occupancy).
 */
#define HC_STATE_FLOATS 32

size_t hc_chain_state_bytes(int64_t n, int hc, int d);

hc_status hc_chain_begin(const uint16_t *x, const float *pre_mix, const float *hc_fn,
                         const float *hc_scale, const float *hc_base, int64_t n, int hc, int d,
                         int sinkhorn_iters, float eps, float norm_eps, float *state_out,
                         size_t state_bytes, float *pre_out, uint16_t *h_pre_out,
                         cudaStream_t stream);

hc_status hc_chain_side(const uint16_t *x, const uint16_t *f, const float *state_in,
                        const float *norm_w, const float *hc_fn_next, const float *hc_scale_next,
                        const float *hc_base_next, int64_t n, int hc, int d, int sinkhorn_iters,
                        float eps, float norm_eps, uint16_t *h_norm, uint16_t *y,
                        float *state_out, size_t state_bytes, float *pre_out, uint16_t *h_pre_out,
                        cudaStream_t stream);

hc_status hc_chain_norm(const uint16_t *h_pre, const float *state, const float *norm_w, int64_t n,
                        int d, uint16_t *h_norm, uint8_t *codes, uint8_t *scales,
                        cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* HC_H_ */
