"""The bf16 tolerance used against the CUDA path (oracle/parity.py) stays
tight.  Its absolute allowance is at the level of fp32 rounding except where
the arithmetic itself can flip a bf16 rounding (y: cancellation; h_norm: an h
on a bf16 midpoint).  Errors that a wrong kernel would make are caught: an
element two ulps off, and an h rounded toward zero (truncated) instead of to
nearest before the RMSNorm."""
import numpy as np
import pytest

import oracle
from oracle import parity
from hyper_connection_residual_mixes_gb300 import inputs


def _case(n=4, d=256, seed=21):
    case = inputs.tiny(seed=seed, n=n, d=d)
    p = case.params[0]
    xb, fb = inputs.bf16_bits_np(case.x), inputs.bf16_bits_np(case.fs[0])
    pm = case.pre_mix.numpy().astype(np.float64)
    ref = oracle.block_step(xb, pm, fb, *(t.numpy() for t in p.astuple()))
    return case, p, xb, fb, pm, ref


def test_allowance_is_small_away_from_cancellation():
    case, p, xb, fb, pm, ref = _case()
    ya = parity.y_allowance(fb, xb, ref["post"], ref["comb"], ref["post"] + 1e-7, ref["comb"] + 1e-7)
    y = np.abs(oracle.bf16_to_f64(ref["y"]))
    big = y > 0.1
    assert np.median(ya[big] / y[big]) < 1e-5
    ha = parity.h_norm_allowance(xb, pm, p.norm_w.numpy(), ref["h_norm"])
    h = np.abs(oracle.bf16_to_f64(ref["h_norm"]))
    nz = h > 0
    # away from bf16 midpoints of h the allowance is the fp32 rounding term alone
    assert np.median(ha[nz] / h[nz]) <= 4 * parity.U32 * (1 + 1e-12)


def test_h_midpoint_window_is_rare_and_correct():
    """The extra allowance goes only to elements whose exact h lies within
    (hc + 1) u S_h of a bf16 rounding midpoint: few of them, and each one is
    checked against the definition directly."""
    case, p, xb, fb, pm, ref = _case(n=8, d=1024, seed=3)
    near, spacing, window = parity.h_midpoint_window(xb, pm)
    assert near.mean() < 1e-3
    x = oracle.bf16_to_f64(xb)
    h = np.einsum("ts,tsd->td", pm, x)
    S = np.einsum("ts,tsd->td", np.abs(pm), np.abs(x))
    # brute force on a sample: distance to the midpoints between the bf16
    # neighbours of h (found by rounding h up and down by a bisection-free
    # route: the two bf16 values bracketing h)
    rng = np.random.default_rng(0)
    idx = rng.choice(h.size, 400, replace=False)
    for i in idx:
        t, c = divmod(int(i), h.shape[1])
        v = abs(h[t, c])
        b = int(oracle.bf16_from_f64(np.array([v]))[0])
        lo_b, hi_b = (b - 1, b) if oracle.bf16_to_f64(np.array([b], np.uint16))[0] > v else (b, b + 1)
        lo, hi = oracle.bf16_to_f64(np.array([max(lo_b, 0), hi_b], np.uint16))
        mids = [0.5 * (lo + hi)]
        if lo_b > 0:
            mids.append(0.5 * (lo + oracle.bf16_to_f64(np.array([lo_b - 1], np.uint16))[0]))
        mids.append(0.5 * (hi + oracle.bf16_to_f64(np.array([hi_b + 1], np.uint16))[0]))
        dist = min(abs(v - m) for m in mids)
        assert near[t, c] == (dist <= 5 * parity.U32 * S[t, c]), (t, c, dist, S[t, c])
        assert window[t, c] == 5 * parity.U32 * S[t, c]


def test_cancelled_h_keeps_the_fp32_window():
    """Where h cancels to far below its terms (here h ~ 1e-7 from O(1) terms),
    an fp32 sum may be off by many bf16 spacings of h; the allowance of such an
    element covers the whole fp32 error window, so an h_norm computed from any
    h inside that window passes."""
    n, d = 1, 64
    x = np.zeros((n, 4, d))
    x[0, 0, :] = 1.0
    x[0, 1, :] = -1.0
    x[0, 2, 0::2] = 1.0      # odd columns cancel to -0.75 * 2^-22, even ones do not
    xb = oracle.bf16_from_f64(x)
    pm = np.array([[0.75, 0.75 * (1 + 2.0 ** -22), 1.0, 0.0]])
    w = np.ones(d)
    ref = oracle.rmsnorm(oracle.pre(xb, pm), w)
    ha = parity.h_norm_allowance(xb, pm, w, ref)
    near, spacing, window = parity.h_midpoint_window(xb, pm)
    h = np.einsum("ts,tsd->td", pm, oracle.bf16_to_f64(xb))
    # an h off by the full window, rounded and normalised as the kernel would
    worst = oracle.rmsnorm(oracle.bf16_from_f64(h + window), w)
    c = 1
    assert abs(h[0, c]) < 2e-7
    assert near[0, c] and window[0, c] > 10 * spacing[0, c]
    parity.check_bf16("h_norm", worst[:, c:c + 1], ref[:, c:c + 1], abs_allow=ha[:, c:c + 1])


def test_two_ulp_error_is_caught():
    case, p, xb, fb, pm, ref = _case()
    y = ref["y"].copy()
    y64 = np.abs(oracle.bf16_to_f64(y))
    i = np.unravel_index(np.argmax(y64 > 1.0), y.shape)
    bad = y.copy()
    bad[i] = bad[i] + np.uint16(2)  # two ulps away from zero
    ya = parity.y_allowance(fb, xb, ref["post"], ref["comb"], ref["post"], ref["comb"])
    parity.check_bf16("y", y, ref["y"], abs_allow=ya)
    with pytest.raises(AssertionError):
        parity.check_bf16("y", bad, ref["y"], abs_allow=ya)


def test_two_ulp_h_norm_error_is_caught():
    case, p, xb, fb, pm, ref = _case()
    ha = parity.h_norm_allowance(xb, pm, p.norm_w.numpy(), ref["h_norm"])
    parity.check_bf16("h_norm", ref["h_norm"], ref["h_norm"], abs_allow=ha)
    near, _, _ = parity.h_midpoint_window(xb, pm)
    h64 = np.abs(oracle.bf16_to_f64(ref["h_norm"]))
    cand = np.argwhere((h64 > 0.5) & ~near)
    assert len(cand) > 0
    for t, c in cand[:50]:
        bad = ref["h_norm"].copy()
        bad[t, c] = bad[t, c] + np.uint16(2)  # two ulps away from zero
        with pytest.raises(AssertionError):
            parity.check_bf16("h_norm", bad, ref["h_norm"], abs_allow=ha)


def _h_toward_zero(xb, pm):
    """h = sum_s pm[s] x[s] rounded to bf16 toward zero (a truncating kernel)."""
    rne = oracle.pre(xb, pm)
    h = np.einsum("ts,tsd->td", pm, oracle.bf16_to_f64(xb))
    away = np.abs(oracle.bf16_to_f64(rne)) > np.abs(h)
    return np.where(away, rne - np.uint16(1), rne).astype(np.uint16)


def test_h_rounded_toward_zero_is_caught():
    """An RMSNorm fed an h that was rounded toward zero (or truncated) instead
    of to nearest fails the h_norm check."""
    case, p, xb, fb, pm, ref = _case(n=8, d=1024, seed=3)
    w = p.norm_w.numpy()
    ha = parity.h_norm_allowance(xb, pm, w, ref["h_norm"])
    wrong = oracle.rmsnorm(_h_toward_zero(xb, pm), w)
    assert np.count_nonzero(wrong != ref["h_norm"]) > wrong.size // 10
    with pytest.raises(AssertionError):
        parity.check_bf16("h_norm", wrong, ref["h_norm"], abs_allow=ha)
    # the same inputs through the exact path pass
    parity.check_bf16("h_norm", oracle.rmsnorm(oracle.pre(xb, pm), w), ref["h_norm"], abs_allow=ha)


def test_fp32_check():
    parity.check_fp32("c", np.array([1.0, 2.0]), np.array([1.0 + 9e-6, 2.0]))
    with pytest.raises(AssertionError):
        parity.check_fp32("c", np.array([1.0, 2.0]), np.array([1.0 + 2e-5, 2.0]))
