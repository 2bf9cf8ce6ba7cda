"""GPU: the side step's backward (hc_block_step_backward) against the CPU
oracle's (oracle.side_backward, fp64, with the forward's bf16 casts applied
and gradients passed through them unchanged).

Tolerances.  Per-token gradients (g_x, g_f, g_pre_mix) come from fp32 sums of
up to hc*d = 20,480 products, some of which cancel (the RMSNorm statistic's
term against the direct one), and a fp32 Sinkhorn backward of 40 steps:
|err| <= RTOL_TOK * |ref| + ATOL * max|ref|.  The parameter gradients are fp32
sums over all tokens: |err| <= RTOL_PAR * |ref| + ATOL * max|ref|.

The backward also reads the forward's bf16 h.  Where the GPU's fp32 sum of
pre_mix * x and the oracle's fp64 sum round to different bf16 neighbours (one
element in about 30,000), h differs by one bf16 ulp there and that token's
term of g_norm_w moves by 2^-8 of itself.  The main tests draw pre_mix from
powers of two, which makes the sum exact in fp32 (four bf16 products), so no
such flip can occur and every gradient is held to the bounds above;
test_backward_general_pre_mix keeps general pre_mix values and gives g_norm_w
an allowance of a few such flips per column."""
import numpy as np
import pytest
import torch

import oracle
import hyper_connection_residual_mixes_gb300 as hcg
from hyper_connection_residual_mixes_gb300 import _lib, inputs
from hyper_connection_residual_mixes_gb300 import build as hc_build

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")
RTOL_TOK, RTOL_PAR, ATOL = 1e-4, 1e-3, 1e-4


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hc_build.build()
    _lib.load()


def _np(t):
    return t.detach().cpu().numpy()


def _case(seed, n, d, with_pre=True, dyadic=True):
    case = inputs.tiny(seed=seed, n=n, d=d)
    g = torch.Generator().manual_seed(seed + 1)
    if dyadic:   # pre_mix in {1, 1/2, 1/4, 1/8}: the fp32 sum of pre_mix * x is exact
        case.pre_mix.copy_(torch.exp2(-torch.randint(0, 4, tuple(case.pre_mix.shape), generator=g).float()))
    up = dict(g_h_norm=torch.randn((n, d), generator=g), g_y=torch.randn((n, 4, d), generator=g),
              g_pre=torch.randn((n, 4), generator=g) if with_pre else None)
    return case, up


def _run(case, up, iters=20):
    p = case.params[0]
    return hcg.hc_block_step_backward(
        case.x.to(DEV), case.pre_mix.to(DEV), case.fs[0].to(DEV), *p.to(DEV).astuple(),
        up["g_h_norm"].to(DEV), up["g_y"].to(DEV),
        g_pre=up["g_pre"].to(DEV) if up["g_pre"] is not None else None, sinkhorn_iters=iters)


def _ref(case, up, iters=20):
    p = case.params[0]
    return oracle.side_backward(
        oracle.bf16_to_f64(oracle.bf16_bits(case.x)), _np(case.pre_mix).astype(np.float64),
        oracle.bf16_to_f64(oracle.bf16_bits(case.fs[0])), *(_np(t).astype(np.float64) for t in p.astuple()),
        _np(up["g_h_norm"]).astype(np.float64), _np(up["g_y"]).astype(np.float64),
        None if up["g_pre"] is None else _np(up["g_pre"]).astype(np.float64), iters=iters, rounded=True)


def _compare(got, ref, extra=None):
    worst = {}
    for k, r in ref.items():
        g = _np(got[k]).astype(np.float64)
        rt = RTOL_TOK if k in ("g_x", "g_f", "g_pre_mix") else RTOL_PAR
        scale = np.abs(r).max()
        err = np.abs(g - r)
        bound = rt * np.abs(r) + ATOL * scale + (extra.get(k, 0.0) if extra else 0.0)
        worst[k] = float((err / np.maximum(bound, 1e-300)).max())
        assert np.all(err <= bound), "%s: worst err/bound %.3g (max err %.3g, scale %.3g)" % (
            k, worst[k], err.max(), scale)
    return worst


@pytest.mark.parametrize("n,d,iters,with_pre", [(16, 5120, 20, True), (37, 1024, 20, False),
                                                 (3, 64, 1, True), (5, 2048, 7, True),
                                                 (4, 7168, 20, True), (3, 16384, 20, True),
                                                 (1, 5120, 20, True)])
def test_backward_matches_oracle(n, d, iters, with_pre):
    case, up = _case(40 + n, n, d, with_pre)
    got = _run(case, up, iters)
    torch.cuda.synchronize()
    _compare(got, _ref(case, up, iters))
    assert _lib.raw("hc_consume_device_error", None) == 0


def test_backward_across_token_blocks_and_repeatable():
    """1,030 tokens: the parameter sums cross a 1,024-token block; two runs
    give the same bits."""
    case, up = _case(77, 1030, 256)
    a = _run(case, up)
    b = _run(case, up)
    torch.cuda.synchronize()
    for k in a:
        assert torch.equal(a[k], b[k]), k
    _compare(a, _ref(case, up))


def test_backward_zero_upstream_is_zero():
    case, up = _case(5, 8, 1024)
    up = {k: (torch.zeros_like(v) if v is not None else None) for k, v in up.items()}
    got = _run(case, up)
    torch.cuda.synchronize()
    for k, v in got.items():
        assert torch.count_nonzero(v).item() == 0, k


def test_backward_general_pre_mix():
    """General pre_mix values: every gradient but g_norm_w to the same bounds;
    g_norm_w with room for up to four one-ulp flips of h per column."""
    case, up = _case(91, 300, 1024, dyadic=False)
    got = _run(case, up)
    torch.cuda.synchronize()
    ref = _ref(case, up)
    # the largest single term h * rs_h * g_hn of each column, from the oracle's forward
    p = case.params[0]
    fw = oracle.side_f64(oracle.bf16_to_f64(oracle.bf16_bits(case.x)), _np(case.pre_mix).astype(np.float64),
                         oracle.bf16_to_f64(oracle.bf16_bits(case.fs[0])),
                         *(_np(t).astype(np.float64) for t in p.astuple()), rounded=True)
    w = _np(p.norm_w).astype(np.float64)
    u = fw["h_norm"] / w                       # h * rs_h, up to the final cast
    term = np.abs(u * _np(up["g_h_norm"]).astype(np.float64)).max(axis=0)
    _compare(got, ref, extra={"g_norm_w": 4 * 2.0 ** -8 * term * 1.01})


def test_backward_long_prefill_sampled_tokens_and_additivity():
    """The long-prefill size (65,536 tokens x d = 5120) with the workspace
    entry, as the backward bench calls it.  Each token's gradients depend on
    that token alone, so g_x, g_pre_mix and g_f are checked against the oracle
    on sampled tokens (the last one among them).  The parameter gradients are
    sums over all 64 token blocks; the full batch must equal the sum of its
    two halves."""
    case = inputs.long_prefill(device=DEV, materialize_f=False)
    n, d = case.n, case.d
    p = case.params[0]
    f0 = inputs.long_prefill_f(0, n, d, DEV)
    g = torch.Generator(device=DEV).manual_seed(5)
    g_hn = torch.randn((n, d), device=DEV, generator=g)
    g_y = torch.randn((n, 4, d), device=DEV, generator=g)
    g_pre = torch.randn((n, 4), device=DEV, generator=g)
    full = hcg.hc_block_step_backward(case.x, case.pre_mix, f0, *p.astuple(), g_hn, g_y, g_pre)
    half = n // 2
    parts = [hcg.hc_block_step_backward(case.x[a:b], case.pre_mix[a:b], f0[a:b], *p.astuple(), g_hn[a:b],
                                        g_y[a:b], g_pre[a:b]) for a, b in ((0, half), (half, n))]
    torch.cuda.synchronize()
    assert _lib.raw("hc_consume_device_error", None) == 0
    for k in ("g_x", "g_pre_mix", "g_f"):   # per token: the halves give the same bits
        assert torch.equal(full[k][:half], parts[0][k]) and torch.equal(full[k][half:], parts[1][k]), k
    for k in ("g_hc_fn", "g_hc_scale", "g_hc_base", "g_norm_w"):
        a = _np(full[k]).astype(np.float64)
        b = _np(parts[0][k]).astype(np.float64) + _np(parts[1][k]).astype(np.float64)
        # the same 64 block partials, associated differently at the top: rounding only;
        # a dropped or misplaced block moves a sum by a sizeable part of its scale
        assert np.all(np.abs(a - b) <= 1e-5 * np.abs(a) + 1e-4 * np.abs(a).max()), k
    rows = np.sort(np.random.default_rng(17).choice(n - 1, 5, replace=False)).tolist() + [n - 1]
    sel = torch.tensor(rows, device=DEV)
    pick = lambda t: t.index_select(0, sel).cpu()
    ref = oracle.side_backward(
        oracle.bf16_to_f64(oracle.bf16_bits(pick(case.x))), _np(pick(case.pre_mix)).astype(np.float64),
        oracle.bf16_to_f64(oracle.bf16_bits(pick(f0))), *(_np(t).astype(np.float64) for t in p.astuple()),
        _np(pick(g_hn)).astype(np.float64), _np(pick(g_y)).astype(np.float64),
        _np(pick(g_pre)).astype(np.float64), rounded=True)
    for k in ("g_x", "g_pre_mix", "g_f"):
        got = _np(pick(full[k])).astype(np.float64)
        r = ref[k]
        # general pre_mix: an h flip moves g_x / g_pre_mix by at most the term it feeds;
        # the per-token bound of the other tests, with ATOL on each token's own scale
        scale = np.abs(r).reshape(len(rows), -1).max(axis=1).reshape((-1,) + (1,) * (r.ndim - 1))
        err = np.abs(got - r)
        assert np.all(err <= RTOL_TOK * np.abs(r) + 2 * ATOL * scale), (k, float(err.max()))


@pytest.mark.parametrize("iters,eps", [(128, 1e-6), (20, 0.0)])
def test_backward_iteration_limits(iters, eps):
    """128 Sinkhorn rounds (the largest accepted; the per-token kernel keeps
    256 iterates per token in shared memory) and eps = 0."""
    case, up = _case(120 + iters, 6, 256)
    p = case.params[0]
    got = hcg.hc_block_step_backward(
        case.x.to(DEV), case.pre_mix.to(DEV), case.fs[0].to(DEV), *p.to(DEV).astuple(),
        up["g_h_norm"].to(DEV), up["g_y"].to(DEV), g_pre=up["g_pre"].to(DEV), sinkhorn_iters=iters, eps=eps)
    torch.cuda.synchronize()
    ref = oracle.side_backward(
        oracle.bf16_to_f64(oracle.bf16_bits(case.x)), _np(case.pre_mix).astype(np.float64),
        oracle.bf16_to_f64(oracle.bf16_bits(case.fs[0])), *(_np(t).astype(np.float64) for t in p.astuple()),
        _np(up["g_h_norm"]).astype(np.float64), _np(up["g_y"]).astype(np.float64),
        _np(up["g_pre"]).astype(np.float64), iters=iters, eps=eps, rounded=True)
    _compare(got, ref)
    assert _lib.raw("hc_consume_device_error", None) == 0


@pytest.mark.parametrize("hc,n,d,iters", [(2, 5, 256, 20), (8, 5, 256, 20), (2, 37, 1024, 7),
                                          (8, 9, 1024, 1), (8, 1030, 64, 20)])
def test_backward_other_stream_counts(hc, n, d, iters):
    """Two and eight streams (the plain kernels) against the oracle; 1,030
    tokens cross a parameter-sum block."""
    case = inputs.tiny(seed=200 + hc + n, n=n, d=d, hc=hc)
    g = torch.Generator().manual_seed(300 + hc + n)
    case.pre_mix.copy_(torch.exp2(-torch.randint(0, 4, tuple(case.pre_mix.shape), generator=g).float()))
    up = dict(g_h_norm=torch.randn((n, d), generator=g), g_y=torch.randn((n, hc, d), generator=g),
              g_pre=torch.randn((n, hc), generator=g))
    p = case.params[0]
    got = hcg.hc_block_step_backward(
        case.x.to(DEV), case.pre_mix.to(DEV), case.fs[0].to(DEV), *p.to(DEV).astuple(),
        up["g_h_norm"].to(DEV), up["g_y"].to(DEV), g_pre=up["g_pre"].to(DEV), sinkhorn_iters=iters)
    torch.cuda.synchronize()
    assert got["g_x"].shape == (n, hc, d) and got["g_hc_fn"].shape == ((2 + hc) * hc, hc * d)
    ref = oracle.side_backward(
        oracle.bf16_to_f64(oracle.bf16_bits(case.x)), _np(case.pre_mix).astype(np.float64),
        oracle.bf16_to_f64(oracle.bf16_bits(case.fs[0])), *(_np(t).astype(np.float64) for t in p.astuple()),
        _np(up["g_h_norm"]).astype(np.float64), _np(up["g_y"]).astype(np.float64),
        _np(up["g_pre"]).astype(np.float64), iters=iters, rounded=True)
    _compare(got, ref)
    again = hcg.hc_block_step_backward(
        case.x.to(DEV), case.pre_mix.to(DEV), case.fs[0].to(DEV), *p.to(DEV).astuple(),
        up["g_h_norm"].to(DEV), up["g_y"].to(DEV), g_pre=up["g_pre"].to(DEV), sinkhorn_iters=iters)
    torch.cuda.synchronize()
    for k in got:
        assert torch.equal(got[k], again[k]), k
    assert _lib.raw("hc_consume_device_error", None) == 0
