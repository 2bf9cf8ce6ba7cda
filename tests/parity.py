"""Parity helpers: compare CUDA outputs with the oracle.

Tolerances (stated for this path): |delta| <= 1e-5 absolute on fp32
pre / post / comb; on bf16 outputs |delta| <= 1 bf16 ulp(ref) + 1e-3 |ref|,
where ulp(ref) is the spacing of bf16 numbers at |ref| (toward larger
magnitude).
"""
import numpy as np
import torch

import oracle

FP32_ATOL = 1e-5
BF16_REL = 1e-3


def bits(t):
    if isinstance(t, torch.Tensor):
        return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return np.asarray(t, dtype=np.uint16)


def bf16_ulp(ref_bits):
    r = oracle.bf16_to_f64(ref_bits)
    nxt = oracle.bf16_to_f64((ref_bits & np.uint16(0x7FFF)) + np.uint16(1))
    return np.abs(nxt - np.abs(r))


def check_fp32(name, got, ref, atol=FP32_ATOL):
    g = got.detach().cpu().double().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    err = np.abs(g - np.asarray(ref, dtype=np.float64))
    worst = float(err.max()) if err.size else 0.0
    assert np.all(np.isfinite(g)), "%s has non-finite values" % name
    assert worst <= atol, "%s: max |delta| %.3g > %.3g at %s" % (
        name, worst, atol, np.unravel_index(np.argmax(err), err.shape))
    return worst


def check_bf16(name, got, ref_bits, rel=BF16_REL):
    gb = bits(got)
    rb = np.asarray(ref_bits, dtype=np.uint16)
    assert gb.shape == rb.shape, (gb.shape, rb.shape)
    g = oracle.bf16_to_f64(gb)
    r = oracle.bf16_to_f64(rb)
    tol = bf16_ulp(rb) + rel * np.abs(r)
    err = np.abs(g - r)
    bad = ~(err <= tol)
    if bad.any():
        i = np.unravel_index(np.argmax(bad), bad.shape)
        raise AssertionError("%s: %d of %d elements outside 1 ulp + %g rel; first at %s: got %r ref %r"
                             % (name, int(bad.sum()), bad.size, rel, i, g[i], r[i]))
    # report how many differ at all (rounding flips), for information
    return int(np.count_nonzero(gb != rb))
