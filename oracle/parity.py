"""Parity tolerances between the CUDA path and the oracle -- TEST INFRASTRUCTURE.

Used by tests/, __graft_entry__.smoke() and bench.py only.

fp32 outputs (pre, post, comb): |delta| <= 1e-5 absolute.

bf16 outputs (y, h_norm): |delta| <= 1 bf16 ulp(ref) + 1e-3 |ref| + a,
where `a` is the absolute error the fp32 arithmetic itself can produce
before the final rounding, derived from the operation:

  y[k] = post[k] f + sum_j comb[j][k] x[j]
    The GPU mixes with its own fp32 coefficients, which differ from the
    oracle's fp64 ones by dc (measured per token, <= 1e-5 by the fp32 check),
    and rounds 5 times in fp32: a = dc (|f| + sum_j |x[j]|) + 6 u S with
    S = |post[k] f| + sum_j |comb[j][k] x[j]| and u = 2^-24.
  h_norm = bf16((bf16(sum_s pm[s] x[s]) * rs) * w)
    The GPU sums the hc products in fp32 with hc roundings (a product, then
    fused multiply-adds), so its h is within hc u S_h of the exact sum, with
    S_h = sum_s |pm[s] x[s]|.  Only where the exact h lies that close to a
    bf16 rounding midpoint (within (hc + 1) u S_h) can the fp32 sum round to
    another bf16 value than the exact h does; there, and only there, the two
    rounded h differ by at most (hc + 1) u S_h + one bf16 spacing of h (more
    than one spacing only under cancellation, S_h >> |h|), scaled by rs |w|
    on the way out.  Every element also gets 4 u |ref| for the fp32 products
    (h rs) w:
    a = [h near a midpoint] (spacing_bf16(h) + (hc + 1) u S_h) rs |w| + 4 u |ref|.
    Everywhere else the bound is 1 ulp + 1e-3 |ref| + 4 u |ref|, so an h
    rounded the wrong way (truncated, toward zero) or an h_norm two ulps off
    fails it.

So `a` matters only where a result is tiny next to the terms it is summed
from, or (h_norm) where h sits on a bf16 rounding midpoint.
"""
import numpy as np

from . import bf16_to_f64

FP32_ATOL = 1e-5
BF16_REL = 1e-3
U32 = 2.0 ** -24


def _bits(t):
    if hasattr(t, "detach"):
        import torch
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return np.asarray(t, dtype=np.uint16)


def _np64(t):
    if hasattr(t, "detach"):
        return t.detach().cpu().double().numpy()
    return np.asarray(t, dtype=np.float64)


def bf16_ulp(ref_bits):
    """Spacing of bf16 numbers at |ref| (toward larger magnitude)."""
    rb = np.asarray(ref_bits, dtype=np.uint16)
    r = bf16_to_f64(rb)
    nxt = bf16_to_f64((rb & np.uint16(0x7FFF)) + np.uint16(1))
    return np.abs(nxt - np.abs(r))


def check_fp32(name, got, ref, atol=FP32_ATOL):
    g = _np64(got)
    err = np.abs(g - np.asarray(ref, dtype=np.float64))
    worst = float(err.max()) if err.size else 0.0
    assert np.all(np.isfinite(g)), "%s has non-finite values" % name
    assert worst <= atol, "%s: max |delta| %.3g > %.3g at %s" % (
        name, worst, atol, np.unravel_index(np.argmax(err), err.shape))
    return worst


def check_bf16(name, got, ref_bits, rel=BF16_REL, abs_allow=None):
    """Returns the number of elements whose bits differ at all (rounding flips)."""
    gb = _bits(got)
    rb = np.asarray(ref_bits, dtype=np.uint16)
    assert gb.shape == rb.shape, (gb.shape, rb.shape)
    g = bf16_to_f64(gb)
    r = bf16_to_f64(rb)
    tol = bf16_ulp(rb) + rel * np.abs(r)
    if abs_allow is not None:
        tol = tol + abs_allow
    err = np.abs(g - r)
    bad = ~(err <= tol)
    if bad.any():
        i = np.unravel_index(np.argmax(bad), bad.shape)
        raise AssertionError("%s: %d of %d elements outside tolerance; first at %s: got %r ref %r "
                             "(tol %r)" % (name, int(bad.sum()), bad.size, i, g[i], r[i], tol[i]))
    return int(np.count_nonzero(gb != rb))


def y_allowance(f_bits, x_bits, post_ref, comb_ref, post_got=None, comb_got=None):
    """Absolute allowance for y [n, hc, d] (see the module docstring)."""
    f = bf16_to_f64(_bits(f_bits))                   # [n, d]
    x = bf16_to_f64(_bits(x_bits))                   # [n, hc, d]
    post = np.asarray(post_ref, np.float64)          # [n, hc]
    comb = np.asarray(comb_ref, np.float64)          # [n, hc, hc]
    if post_got is not None:
        dc = np.maximum(np.max(np.abs(_np64(post_got) - post), axis=1),
                        np.max(np.abs(_np64(comb_got) - comb), axis=(1, 2)))
    else:
        dc = np.zeros(post.shape[0])
    ax = np.abs(x)
    S = np.abs(post)[:, :, None] * np.abs(f)[:, None, :] + np.einsum("tjk,tjd->tkd", np.abs(comb), ax)
    return dc[:, None, None] * (np.abs(f)[:, None, :] + ax.sum(axis=1)[:, None, :]) + 6 * U32 * S


def _bf16_mag(bits):
    """|value| of bf16 bit patterns (the sign bit dropped)."""
    return bf16_to_f64(np.asarray(bits, dtype=np.uint16) & np.uint16(0x7FFF))


def h_midpoint_window(x_bits, pre_mix):
    """For h = sum_s pm[s] x[s]: a mask of the elements whose exact h lies
    within the fp32 error window (hc + 1) u S_h of a bf16 rounding midpoint
    (where an fp32 evaluation may round differently), the bf16 spacing of h
    on the side of that midpoint, and the window itself.  The rounded h is
    the oracle's own hc_pre (fp64 sum, one round to nearest even)."""
    from . import pre as oracle_pre
    xb = _bits(x_bits)
    x = bf16_to_f64(xb)                              # [n, hc, d]
    hc = x.shape[1]
    pm = np.asarray(pre_mix, np.float64)             # [n, hc]
    terms = pm[:, :, None] * x
    a = np.abs(terms.sum(axis=1))                    # |h|
    S_h = np.abs(terms).sum(axis=1)
    hb = oracle_pre(xb, pm) & np.uint16(0x7FFF)      # bits of |bf16(h)|
    mag = _bf16_mag(hb)
    up = _bf16_mag(hb + np.uint16(1))                # the next bf16 magnitude above
    dn = np.where(hb == 0, -up, _bf16_mag(np.maximum(hb, np.uint16(1)) - np.uint16(1)))
    d_up = np.abs(a - 0.5 * (mag + up))
    d_dn = np.abs(a - 0.5 * (mag + dn))
    window = (hc + 1) * U32 * S_h
    near = np.minimum(d_up, d_dn) <= window
    spacing = np.where(d_up <= d_dn, up - mag, mag - dn)
    return near, spacing, window


def h_norm_allowance(x_bits, pre_mix, norm_w, h_norm_ref_bits, eps=1e-20):
    """Absolute allowance for h_norm [n, d] (see the module docstring)."""
    from . import pre as oracle_pre
    pm = np.asarray(pre_mix, np.float64)             # [n, hc]
    w = np.abs(np.asarray(norm_w, np.float64))       # [d]
    hb = bf16_to_f64(oracle_pre(_bits(x_bits), pm))
    rs = 1.0 / np.sqrt(np.mean(hb * hb, axis=1, keepdims=True) + eps)
    near, spacing, window = h_midpoint_window(x_bits, pm)
    ref = np.abs(bf16_to_f64(_bits(h_norm_ref_bits)))
    return np.where(near, (spacing + window) * rs * w[None, :], 0.0) + 4 * U32 * ref
