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
    The fp32 sum of 4 products rounds 4 times before its bf16 rounding, so
    h can land on the other side of a bf16 rounding boundary, off by up to
    5 u S_h with S_h = sum_s |pm[s] x[s]|; scaled by rs |w| on the way out:
    a = (ulp_bf16(h) + 5 u S_h) rs |w| + 4 u |ref|.

Away from cancellation `a` is far below 1e-3 |ref|; it only matters where the
result is tiny compared to the terms it is summed from.
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


def h_norm_allowance(x_bits, pre_mix, norm_w, h_norm_ref_bits, eps=1e-20):
    """Absolute allowance for h_norm [n, d] (see the module docstring)."""
    x = bf16_to_f64(_bits(x_bits))                   # [n, hc, d]
    pm = np.asarray(pre_mix, np.float64)             # [n, hc]
    w = np.abs(np.asarray(norm_w, np.float64))       # [d]
    terms = pm[:, :, None] * x
    h = terms.sum(axis=1)
    S_h = np.abs(terms).sum(axis=1)
    from . import bf16_from_f64
    hb = bf16_to_f64(bf16_from_f64(h)) if h.size <= 200000 else h
    rs = 1.0 / np.sqrt(np.mean(hb * hb, axis=1, keepdims=True) + eps)
    ulp_h = np.abs(h) * 2.0 ** -7 + 1e-40
    ref = np.abs(bf16_to_f64(_bits(h_norm_ref_bits)))
    return (ulp_h + 5 * U32 * S_h) * rs * w[None, :] + 4 * U32 * ref
