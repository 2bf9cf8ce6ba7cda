"""GPU: the chain of side steps fused across sides (hc_chain_begin /
hc_chain_side) against hc_block_step run side after side.

The fused chain computes each side's coefficients in the previous launch, on
the y it has just produced, with the same per-thread columns and summation
order as hc_block_step; so every output must agree bit for bit.  hc_block_step
itself is checked against the CPU oracle in test_gpu_parity.py; here the chain
is also compared with the oracle directly on sampled tokens."""
import numpy as np
import pytest
import torch

import oracle
import hyper_connection_residual_mixes_gb300 as hcg
from hyper_connection_residual_mixes_gb300 import _lib, inputs
from hyper_connection_residual_mixes_gb300 import build as hc_build
from parity import bits, check_bf16, check_fp32, h_norm_allowance, y_allowance

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hc_build.build()
    _lib.load()


def _steps(x, pm, fs, params):
    """Side by side with hc_block_step: per side (h_norm, y, pre)."""
    out = []
    for f, p in zip(fs, params):
        h, y, pre = hcg.hc_block_step(x, pm, f, *p.astuple())
        out.append((h, y, pre))
        x, pm = y, pre
    return out


def _chain(x, pm, fs, params, states=None):
    """The fused chain: per side (h_norm, y, pre of that side); `states`, when a
    list, receives each side's state rows."""
    S = len(params)
    p0 = params[0]
    pre0 = torch.empty_like(pm)
    state = hcg.hc_chain_begin(x, pm, p0.hc_fn, p0.hc_scale, p0.hc_base, pre_out=pre0)
    pres = [pre0]
    out = []
    for i in range(S):
        p = params[i]
        if i + 1 < S:
            q = params[i + 1]
            pre_next = torch.empty_like(pm)
            h, y, state_next = hcg.hc_chain_side(x, fs[i], state, p.norm_w, q.hc_fn, q.hc_scale, q.hc_base,
                                                 pre_out=pre_next)
            pres.append(pre_next)
        else:
            h, y, state_next = hcg.hc_chain_side(x, fs[i], state, p.norm_w)
        out.append((h, y, pres[i]))
        if states is not None:
            states.append(state)
        x, state = y, state_next
    return out


def _same(tag, a, b):
    if a.dtype == torch.bfloat16:
        a, b = a.view(torch.int16), b.view(torch.int16)
    diff = int((a != b).sum().item())
    assert diff == 0, "%s: %d of %d elements differ" % (tag, diff, a.numel())


def _compare(ref, got):
    assert len(ref) == len(got)
    for i, (r, g) in enumerate(zip(ref, got)):
        for name, a, b in zip(("h_norm", "y", "pre"), r, g):
            _same("side %d %s" % (i, name), a, b)


def test_chain_equals_block_steps_decode():
    case = inputs.decode(device=DEV)
    ref = _steps(case.x, case.pre_mix, case.fs, case.params)
    got = _chain(case.x, case.pre_mix, case.fs, case.params)
    torch.cuda.synchronize()
    _compare(ref, got)
    assert _lib.raw("hc_consume_device_error", None) == 0


def test_chain_equals_block_steps_prefill():
    case = inputs.prefill(device=DEV)
    ref = _steps(case.x, case.pre_mix, case.fs, case.params)
    got = _chain(case.x, case.pre_mix, case.fs, case.params)
    torch.cuda.synchronize()
    _compare(ref, got)


@pytest.mark.parametrize("n,d", [(1361, 1024), (530, 7168), (37, 2048)])
def test_chain_equals_block_steps_widths(n, d):
    """Other widths (1 and 7 column blocks per tile phase), several tiles per
    cluster and ragged tails, three sides."""
    g = torch.Generator().manual_seed(500 + d)
    x = inputs.streams(g, n, 4, d).to(DEV)
    pm = inputs.pre_mix(g, n).to(DEV)
    params = [inputs.side_params(g, d=d).to(DEV) for _ in range(3)]
    fs = [inputs.sublayer_out(g, n, d).to(DEV) for _ in range(3)]
    ref = _steps(x, pm, fs, params)
    got = _chain(x, pm, fs, params)
    torch.cuda.synchronize()
    _compare(ref, got)


def test_chain_long_prefill_first_sides_and_repeatable():
    """The benchmark's shape (65,536 tokens), its first four sides: equal to the
    side-by-side steps, and a second run of the chain gives the same bits."""
    case = inputs.long_prefill(device=DEV, materialize_f=False)
    S = 4
    fs = [inputs.long_prefill_f(s, case.n, case.d, DEV) for s in range(S)]
    params = case.params[:S]
    ref = _steps(case.x, case.pre_mix, fs, params)
    got = _chain(case.x, case.pre_mix, fs, params)
    torch.cuda.synchronize()
    _compare(ref, got)
    del ref
    again = _chain(case.x, case.pre_mix, fs, params)
    torch.cuda.synchronize()
    _compare(got, again)
    assert _lib.raw("hc_consume_device_error", None) == 0


def test_chain_against_oracle_sampled():
    """The chain against the CPU oracle directly, teacher-forced per side on 48
    sampled tokens of the prefill case."""
    case = inputs.prefill(device=DEV)
    states = []
    got = _chain(case.x, case.pre_mix, case.fs, case.params, states)
    torch.cuda.synchronize()
    rows = torch.from_numpy(np.sort(np.random.default_rng(5).choice(case.n, 48, replace=False))).to(DEV)
    sel = lambda t: t.index_select(0, rows).cpu()
    x, pm = case.x, case.pre_mix
    for i, (h, y, pre) in enumerate(got):
        p = case.params[i].to("cpu")
        xs, pms, fsel = sel(x), sel(pm), sel(case.fs[i])
        ref = oracle.block_step(bits(xs), pms.numpy().astype(np.float64), bits(fsel),
                                *(t.numpy() for t in p.astuple()))
        st = sel(states[i])
        post_g, comb_g = st[:, 0:4], st[:, 4:20].reshape(-1, 4, 4)
        check_fp32("side %d pre" % i, sel(pre), ref["pre"])
        check_fp32("side %d post" % i, post_g, ref["post"])
        check_fp32("side %d comb" % i, comb_g, ref["comb"])
        check_bf16("side %d h_norm" % i, sel(h), ref["h_norm"],
                   abs_allow=h_norm_allowance(bits(xs), pms.numpy().astype(np.float64), p.norm_w.numpy(),
                                              ref["h_norm"]))
        check_bf16("side %d y" % i, sel(y), ref["y"],
                   abs_allow=y_allowance(bits(fsel), bits(xs), ref["post"], ref["comb"], post_g, comb_g))
        x, pm = y, pre


def test_chain_equals_block_steps_80_sides_8192_tokens():
    """A full 40-layer stack (80 sides, each with its own parameters and f) at
    8,192 tokens: every side's h_norm, y and pre through the chain equal those
    of 80 hc_block_step calls bit for bit."""
    n = 8192
    case = inputs.long_prefill(device=DEV, n=n, materialize_f=False)
    S = len(case.params)
    assert S == 80
    fs = [inputs.long_prefill_f(s, n, case.d, DEV) for s in range(S)]
    ref = _steps(case.x, case.pre_mix, fs, case.params)
    got = _chain(case.x, case.pre_mix, fs, case.params)
    torch.cuda.synchronize()
    _compare(ref, got)
    assert _lib.raw("hc_consume_device_error", None) == 0


def _chain_model(x, pm, fs, params, sublayer=None, mxfp8=None):
    """The chain in model order: the first launch writes side 0's bf16 h; each
    side's h_norm comes from hc_chain_norm before the side's launch; launch i
    writes y_i and side i + 1's bf16 h.  f_i = sublayer(h_norm_i) when a
    sublayer is given (else fs[i]).  Returns per side (h_norm, y, pre, f)."""
    S = len(params)
    n, d = x.shape[0], x.shape[-1]
    p0 = params[0]
    hp = torch.empty((n, d), dtype=torch.bfloat16, device=x.device)
    pre0 = torch.empty_like(pm)
    state = hcg.hc_chain_begin(x, pm, p0.hc_fn, p0.hc_scale, p0.hc_base, pre_out=pre0, h_pre_out=hp)
    pres = [pre0]
    out = []
    for i in range(S):
        p = params[i]
        if mxfp8 is not None:
            h, codes, scales = hcg.hc_chain_norm(hp, state, p.norm_w, mxfp8=True)
            mxfp8.append((h, codes, scales))
        else:
            h = hcg.hc_chain_norm(hp, state, p.norm_w)
        f = sublayer(h) if sublayer is not None else fs[i]
        if i + 1 < S:
            q = params[i + 1]
            hp = torch.empty_like(hp)
            pre_next = torch.empty_like(pm)
            _, y, st_next = hcg.hc_chain_side(x, f, state, p.norm_w, q.hc_fn, q.hc_scale, q.hc_base,
                                              pre_out=pre_next, h_pre_out=hp)
            pres.append(pre_next)
        else:
            _, y, st_next = hcg.hc_chain_side(x, f, state, p.norm_w, write_h_norm=False)
        out.append((h, y, pres[i], f, state))
        x, state = y, st_next
    return out


@pytest.mark.parametrize("n,d,sides", [(128, 5120, 2), (8192, 5120, 4), (1361, 1024, 3), (530, 7168, 3)])
def test_chain_model_order_equals_block_steps(n, d, sides):
    """Model order with the sublayer outputs given: every side's h_norm (from
    hc_chain_norm), y and pre equal hc_block_step's bit for bit."""
    g = torch.Generator().manual_seed(900 + n + d)
    x = inputs.streams(g, n, 4, d).to(DEV)
    pm = inputs.pre_mix(g, n).to(DEV)
    params = [inputs.side_params(g, d=d).to(DEV) for _ in range(sides)]
    fs = [inputs.sublayer_out(g, n, d).to(DEV) for _ in range(sides)]
    ref = _steps(x, pm, fs, params)
    casts = []
    got = _chain_model(x, pm, fs, params, mxfp8=casts)
    torch.cuda.synchronize()
    _compare(ref, [o[:3] for o in got])
    # the cast in the same pass equals the standalone cast of the same h_norm
    for i, (h, codes, scales) in enumerate(casts):
        c2, s2 = hcg.hc_mxfp8_cast(ref[i][0])
        _same("side %d codes" % i, codes, c2)
        _same("side %d scales" % i, scales, s2)
    assert _lib.raw("hc_consume_device_error", None) == 0


def test_chain_model_order_with_a_sublayer_against_oracle():
    """A stand-in sublayer that depends on its input (f = bf16(2 tanh(h_norm)),
    torch on the GPU): the chain in model order, checked side by side against
    the oracle fed the same x, pre_mix and f."""
    n, d, sides = 300, 2048, 4
    g = torch.Generator().manual_seed(77)
    x = inputs.streams(g, n, 4, d).to(DEV)
    pm = inputs.pre_mix(g, n).to(DEV)
    params = [inputs.side_params(g, d=d).to(DEV) for _ in range(sides)]
    sub = lambda h: (2.0 * torch.tanh(h.float())).to(torch.bfloat16)
    got = _chain_model(x, pm, None, params, sublayer=sub)
    torch.cuda.synchronize()
    xs, pms = x, pm
    for i, (h, y, pre, f, st) in enumerate(got):
        p = params[i].to("cpu")
        rows = st[:n].cpu()
        post_g, comb_g = rows[:, 0:4], rows[:, 4:20].reshape(-1, 4, 4)
        xb, fb = bits(xs.cpu()), bits(f.cpu())
        pmn = pms.cpu().numpy().astype(np.float64)
        ref = oracle.block_step(xb, pmn, fb, *(t.numpy() for t in p.astuple()))
        check_fp32("side %d pre" % i, pre.cpu(), ref["pre"])
        check_fp32("side %d post" % i, post_g, ref["post"])
        check_fp32("side %d comb" % i, comb_g, ref["comb"])
        check_bf16("side %d h_norm" % i, h.cpu(), ref["h_norm"],
                   abs_allow=h_norm_allowance(xb, pmn, p.norm_w.numpy(), ref["h_norm"]))
        check_bf16("side %d y" % i, y.cpu(), ref["y"],
                   abs_allow=y_allowance(fb, xb, ref["post"], ref["comb"], post_g, comb_g))
        xs, pms = y, pre
    assert _lib.raw("hc_consume_device_error", None) == 0
