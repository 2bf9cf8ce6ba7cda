"""The bf16 tolerance used against the CUDA path (oracle/parity.py) stays
tight: its absolute allowance is negligible away from cancellation, and a
perturbation of two bf16 ulps of a typical element is still caught."""
import numpy as np
import pytest
import torch

import oracle
from oracle import parity
from hyper_connection_residual_mixes_gb300 import inputs


def _case():
    case = inputs.tiny(seed=21, n=4, d=256)
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
    assert np.median(ha[h > 0.1] / h[h > 0.1]) < 1e-2


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


def test_fp32_check():
    parity.check_fp32("c", np.array([1.0, 2.0]), np.array([1.0 + 9e-6, 2.0]))
    with pytest.raises(AssertionError):
        parity.check_fp32("c", np.array([1.0, 2.0]), np.array([1.0 + 2e-5, 2.0]))
