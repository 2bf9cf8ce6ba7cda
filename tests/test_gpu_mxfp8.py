"""GPU: the MXFP8 cast (DeepSeek V4.1 Flash diagram, block "Cast to MXFP8")
against the CPU oracle, byte for byte.

Codes and scales are bytes, so they must match exactly.  Both sides decide
the scale in fp32 (the division by 448) and round the elements to the
nearest E4M3 value, ties to even.  The fused hc_pre_norm_mxfp8 is compared on
its own h_norm: its bf16 h_norm must equal hc_pre_norm's bit for bit, and its
codes and scales must equal the oracle's cast of that h_norm (h_norm itself is
checked against the oracle within the bf16 tolerance in test_gpu_parity.py)."""
import numpy as np
import pytest
import torch

import oracle
import hyper_connection_residual_mixes_gb300 as hcg
from hyper_connection_residual_mixes_gb300 import _lib, inputs
from hyper_connection_residual_mixes_gb300 import build as hc_build

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hc_build.build()
    _lib.load()


def _rows(seed, rows, d):
    """bf16 rows with the structure the cast has to handle: outliers (x50),
    all-zero groups, groups below the 1e-4 floor, very large groups and
    negative zeros."""
    g = torch.Generator().manual_seed(seed)
    x = inputs.streams(g, rows, 1, d, outlier_p=0.01).reshape(rows, d).float()
    groups = x.view(rows, d // 32, 32)
    pick = torch.rand(rows, d // 32, generator=g)
    groups[pick < 0.03] = 0.0
    groups[(pick >= 0.03) & (pick < 0.06)] *= 1e-6
    groups[(pick >= 0.06) & (pick < 0.08)] *= 1e30
    x = x.to(torch.bfloat16)
    neg0 = torch.rand(rows, d, generator=g) < 0.002
    x[neg0] = -0.0
    return x


def _check(codes, scales, ref_codes, ref_scales):
    c, s = codes.cpu().numpy(), scales.cpu().numpy()
    bad_c = int((c != ref_codes).sum())
    bad_s = int((s != ref_scales).sum())
    assert bad_s == 0, "%d of %d scale bytes differ" % (bad_s, s.size)
    assert bad_c == 0, "%d of %d codes differ" % (bad_c, c.size)


@pytest.mark.parametrize("rows,d", [(1, 32), (3, 96), (1000, 5120), (37, 7168), (129, 4096)])
def test_mxfp8_cast_matches_oracle(rows, d):
    x = _rows(100 + d, rows, d)
    codes, scales = hcg.hc_mxfp8_cast(x.to(DEV))
    torch.cuda.synchronize()
    ref_c, ref_s = oracle.mxfp8(oracle.bf16_bits(x))
    _check(codes, scales, ref_c, ref_s)


def test_mxfp8_cast_ties_subnormals_and_extremes():
    # groups built so that x / scale lands exactly on E4M3 midpoints (ties go to
    # even), on E4M3 subnormals, and on bf16's extremes
    vals = torch.arange(0, 0x7F, dtype=torch.uint8).view(torch.float8_e4m3fn).float()
    mids = (vals[1:] + vals[:-1]) / 2
    rows = []
    for ex in (-20, -3, 0, 7, 100):
        for src in (vals, mids):
            for start in range(0, len(src), 31):
                grp = torch.zeros(32)
                chunk = src[start:start + 31]
                grp[:len(chunk)] = chunk * 2.0 ** ex
                grp[31] = 448.0 * 2.0 ** ex          # pins the scale to 2^ex
                rows.append(grp)
    big = torch.zeros(32)
    big[0] = 3.3895e38                               # bf16's largest finite value
    big[1] = -1.0e38
    tiny = torch.zeros(32)
    tiny[:4] = torch.tensor([9.2e-41, -9.2e-41, 1.2e-38, 3.0e-39])   # bf16 subnormals
    rows += [big, tiny]
    x = torch.stack(rows).to(torch.bfloat16)
    codes, scales = hcg.hc_mxfp8_cast(x.to(DEV))
    torch.cuda.synchronize()
    ref_c, ref_s = oracle.mxfp8(oracle.bf16_bits(x))
    _check(codes, scales, ref_c, ref_s)


def test_pre_norm_mxfp8_prefill_equals_pre_norm_then_oracle_cast():
    case = inputs.prefill(device=DEV)
    p = case.params[0]
    codes, scales, h = hcg.hc_pre_norm_mxfp8(case.x, case.pre_mix, p.norm_w, return_h_norm=True)
    h_ref = hcg.hc_pre_norm(case.x, case.pre_mix, p.norm_w)
    codes2, scales2 = hcg.hc_pre_norm_mxfp8(case.x, case.pre_mix, p.norm_w)
    torch.cuda.synchronize()
    assert torch.equal(h.view(torch.int16), h_ref.view(torch.int16))
    assert torch.equal(codes, codes2) and torch.equal(scales, scales2)
    ref_c, ref_s = oracle.mxfp8(oracle.bf16_bits(h.cpu()))
    _check(codes, scales, ref_c, ref_s)
    assert _lib.raw("hc_consume_device_error", None) == 0


@pytest.mark.parametrize("n,d", [(1, 64), (17, 192), (300, 1024), (61, 7168)])
def test_pre_norm_mxfp8_widths(n, d):
    g = torch.Generator().manual_seed(700 + d)
    x = inputs.streams(g, n, 4, d, outlier_p=0.01).to(DEV)
    pm = inputs.pre_mix(g, n).to(DEV)
    w = inputs.side_params(g, d=d).norm_w.to(DEV)
    codes, scales, h = hcg.hc_pre_norm_mxfp8(x, pm, w, return_h_norm=True)
    h_ref = hcg.hc_pre_norm(x, pm, w)
    torch.cuda.synchronize()
    assert torch.equal(h.view(torch.int16), h_ref.view(torch.int16))
    ref_c, ref_s = oracle.mxfp8(oracle.bf16_bits(h.cpu()))
    _check(codes, scales, ref_c, ref_s)


def test_pre_norm_mxfp8_long_prefill_sampled_rows():
    """The full 65,536-token batch in one launch; 1,024 sampled rows checked."""
    case = inputs.long_prefill(device=DEV, materialize_f=False)
    p = case.params[0]
    codes, scales, h = hcg.hc_pre_norm_mxfp8(case.x, case.pre_mix, p.norm_w, return_h_norm=True)
    torch.cuda.synchronize()
    rows = torch.from_numpy(np.sort(np.random.default_rng(11).choice(case.n, 1024, replace=False))).to(DEV)
    hs = h.index_select(0, rows).cpu()
    ref_c, ref_s = oracle.mxfp8(oracle.bf16_bits(hs))
    _check(codes.index_select(0, rows), scales.index_select(0, rows), ref_c, ref_s)
    assert _lib.raw("hc_consume_device_error", None) == 0
