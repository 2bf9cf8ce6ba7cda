"""GPU parity: every C-ABI entry point against the CPU oracle on the same
seeded inputs.  Small cases are compared element by element; the full-size
workloads are compared on seeded samples of tokens (tokens are independent,
so a sampled token's oracle result is exact), in the launch configuration
the benchmark uses.

Tolerances: |delta| <= 1e-5 on fp32 pre/post/comb; 1 bf16 ulp + 1e-3 rel on
bf16 outputs (tests/parity.py)."""
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


def _np(t):
    return t.detach().cpu().numpy()


def _oracle_side(x, pre_mix, f, params, rows=None):
    """Oracle side step on the given token rows (all when None).  The inputs
    are kept in the result for the tolerance of the bf16 outputs."""
    sel = slice(None) if rows is None else rows
    ref = oracle.block_step(bits(x[sel]), _np(pre_mix[sel]).astype(np.float64), bits(f[sel]),
                            *(_np(t) for t in params.astuple()))
    ref["_in"] = (bits(x[sel]), _np(pre_mix[sel]).astype(np.float64), bits(f[sel]),
                  _np(params.norm_w))
    return ref


def _gpu_side(x, pre_mix, f, params):
    return hcg.hc_block_step(x, pre_mix, f, *params.astuple(), return_post_comb=True)


def _check_side(out, ref, rows=None, tag=""):
    h_norm, y, pre, post, comb = out
    sel = slice(None) if rows is None else rows
    check_fp32(tag + "pre", pre[sel], ref["pre"])
    check_fp32(tag + "post", post[sel], ref["post"])
    check_fp32(tag + "comb", comb[sel], ref["comb"])
    xb, pm, fb, w = ref["_in"]
    check_bf16(tag + "h_norm", h_norm[sel], ref["h_norm"],
               abs_allow=h_norm_allowance(xb, pm, w, ref["h_norm"]))
    check_bf16(tag + "y", y[sel], ref["y"],
               abs_allow=y_allowance(fb, xb, ref["post"], ref["comb"], post[sel], comb[sel]))


# ----------------------------------------------------------------- a2-a3
@pytest.mark.parametrize("n", [1, 5, 127, 128, 129, 1000])
def test_split_sinkhorn_small(n):
    g = torch.Generator().manual_seed(100 + n)
    m = torch.randn((n, 24), generator=g) * 3.0
    scale = torch.rand(3, generator=g) * 1.5 + 0.5
    base = torch.randn(24, generator=g)
    pre, post, comb = hcg.hc_split_sinkhorn(m.to(DEV), scale.to(DEV), base.to(DEV))
    torch.cuda.synchronize()
    rp, rq, rc = oracle.split_sinkhorn(_np(m).astype(np.float64), _np(scale), _np(base))
    check_fp32("pre", pre, rp)
    check_fp32("post", post, rq)
    check_fp32("comb", comb, rc)


@pytest.mark.parametrize("iters", [1, 2, 7, 50])
def test_split_sinkhorn_iters_and_eps(iters):
    g = torch.Generator().manual_seed(7)
    m = torch.randn((300, 24), generator=g) * 2.0
    scale = torch.tensor([1.0, 0.7, 1.6])
    base = torch.randn(24, generator=g)
    for eps in (1e-6, 0.0, 1e-3):
        pre, post, comb = hcg.hc_split_sinkhorn(m.to(DEV), scale.to(DEV), base.to(DEV),
                                                sinkhorn_iters=iters, eps=eps)
        torch.cuda.synchronize()
        rp, rq, rc = oracle.split_sinkhorn(_np(m).astype(np.float64), _np(scale), _np(base),
                                           iters=iters, eps=eps)
        check_fp32("pre", pre, rp)
        check_fp32("post", post, rq)
        check_fp32("comb", comb, rc)


def test_split_sinkhorn_full_stress_config():
    """Sinkhorn-only stress: 2^20 rows of N(0,3) mixes, all rows checked."""
    m, scale, base = inputs.sinkhorn_stress(device="cpu")
    pre, post, comb = hcg.hc_split_sinkhorn(m.to(DEV), scale.to(DEV), base.to(DEV))
    torch.cuda.synchronize()
    rp, rq, rc = oracle.split_sinkhorn(_np(m).astype(np.float64), _np(scale), _np(base))
    check_fp32("pre", pre, rp)
    check_fp32("post", post, rq)
    check_fp32("comb", comb, rc)
    c = _np(comb)
    # page invariants on the fp32 GPU output: columns sum to 1 within 1e-5,
    # entries positive, pre >= eps, post within [0, 2]
    assert np.max(np.abs(c.sum(axis=1) - 1.0)) <= 1e-5
    assert np.all(c > 0)
    assert np.all(_np(pre) >= np.float32(1e-6))
    p = _np(post)
    assert np.all((p >= 0) & (p <= 2))


def test_split_sinkhorn_empty():
    z = torch.empty((0, 24), device=DEV)
    pre, post, comb = hcg.hc_split_sinkhorn(z, torch.ones(3, device=DEV), torch.zeros(24, device=DEV))
    assert pre.shape == (0, 4) and comb.shape == (0, 4, 4)


# ----------------------------------------------------------------- a1-a3
@pytest.mark.parametrize("n,d", [(1, 5120), (16, 5120), (37, 5120), (130, 5120), (1000, 5120), (9, 64),
                                 (21, 1024), (3, 16384)])
def test_mixes(n, d):
    case = inputs.tiny(seed=11 + n, n=n, d=d)
    p = case.params[0]
    pre, post, comb, mixes = hcg.hc_mixes(case.x.to(DEV), p.hc_fn.to(DEV), p.hc_scale.to(DEV),
                                          p.hc_base.to(DEV), return_mixes=True)
    torch.cuda.synchronize()
    rm = oracle.mixes(bits(case.x), _np(p.hc_fn))
    err = np.abs(_np(mixes).astype(np.float64) - rm)
    assert np.all(err <= 1e-5 + 1e-5 * np.abs(rm)), err.max()
    rp, rq, rc = oracle.split_sinkhorn(rm, _np(p.hc_scale), _np(p.hc_base))
    check_fp32("pre", pre, rp)
    check_fp32("post", post, rq)
    check_fp32("comb", comb, rc)


def test_mixes_zero_streams_closed_form():
    # x = 0 gives mixes = 0 exactly, so pre = sigmoid(base) + eps etc.
    n, d = 8, 5120
    x = torch.zeros((n, 4, d), dtype=torch.bfloat16, device=DEV)
    p = inputs.side_params(torch.Generator().manual_seed(3), d=d)
    pre, post, comb, mixes = hcg.hc_mixes(x, p.hc_fn.to(DEV), p.hc_scale.to(DEV),
                                          p.hc_base.to(DEV), return_mixes=True)
    torch.cuda.synchronize()
    assert torch.count_nonzero(mixes).item() == 0
    rp, rq, rc = oracle.split_sinkhorn(np.zeros((n, 24)), _np(p.hc_scale), _np(p.hc_base))
    check_fp32("pre", pre, rp)
    check_fp32("comb", comb, rc)


# ----------------------------------------------------------------- a4-a5, a6
@pytest.mark.parametrize("n,d", [(1, 5120), (16, 5120), (3000, 5120), (33, 64), (5, 16384)])
def test_pre_norm(n, d):
    g = torch.Generator().manual_seed(50 + n)
    x = inputs.streams(g, n, 4, d, outlier_p=0.01)
    pm = inputs.pre_mix(g, n)
    w = torch.rand(d, generator=g) + 0.5
    out = hcg.hc_pre_norm(x.to(DEV), pm.to(DEV), w.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.rmsnorm(oracle.pre(bits(x), _np(pm).astype(np.float64)), _np(w))
    check_bf16("h_norm", out, ref, abs_allow=h_norm_allowance(x, _np(pm), _np(w), ref))


@pytest.mark.parametrize("n,d", [(1, 5120), (16, 5120), (3000, 5120), (33, 64), (5, 16384)])
def test_post(n, d):
    g = torch.Generator().manual_seed(80 + n)
    x = inputs.streams(g, n, 4, d)
    f = inputs.sublayer_out(g, n, d, std=2.0)
    post = torch.rand((n, 4), generator=g) * 2
    comb = torch.rand((n, 4, 4), generator=g)
    y = hcg.hc_post(f.to(DEV), x.to(DEV), post.to(DEV), comb.to(DEV))
    torch.cuda.synchronize()
    ref = oracle.post(bits(f), bits(x), _np(post).astype(np.float64), _np(comb).astype(np.float64))
    check_bf16("y", y, ref, abs_allow=y_allowance(f, x, _np(post), _np(comb)))


# ----------------------------------------------------------------- a1-a6 fused
def test_block_step_tiny_config():
    """Tiny: 16 tokens, one side step, all elements."""
    case = inputs.tiny()
    p = case.params[0]
    out = _gpu_side(case.x.to(DEV), case.pre_mix.to(DEV), case.fs[0].to(DEV), p.to(DEV))
    torch.cuda.synchronize()
    _check_side(out, _oracle_side(case.x, case.pre_mix, case.fs[0], p))


@pytest.mark.parametrize("n,d", [(1, 5120), (3, 5120), (37, 5120), (200, 5120), (70, 64),
                                 (19, 2048), (4, 16384), (301, 8192)])
def test_block_step_shapes(n, d):
    case = inputs.tiny(seed=200 + n, n=n, d=d)
    p = case.params[0]
    out = _gpu_side(case.x.to(DEV), case.pre_mix.to(DEV), case.fs[0].to(DEV), p.to(DEV))
    torch.cuda.synchronize()
    _check_side(out, _oracle_side(case.x, case.pre_mix, case.fs[0], p))


@pytest.mark.parametrize("n,d", [(1361, 1024), (917, 3072), (530, 7168)])
def test_block_step_cluster_widths_many_tiles(n, d):
    """The cluster kernel at other widths: 1, 3 and 7 column blocks per tile
    phase (at d = 7168 the weight fragments fill 504 of the 512 tensor-memory
    columns), with enough tokens that every cluster walks several tiles and
    the last tile is ragged.  All elements checked."""
    case = inputs.tiny(seed=300 + d, n=n, d=d)
    p = case.params[0]
    out = _gpu_side(case.x.to(DEV), case.pre_mix.to(DEV), case.fs[0].to(DEV), p.to(DEV))
    torch.cuda.synchronize()
    _check_side(out, _oracle_side(case.x, case.pre_mix, case.fs[0], p))


def test_mixes_cluster_many_tiles():
    """hc_mixes through the cluster kernel (phase 1 only) over many tiles."""
    n, d = 1361, 1024
    case = inputs.tiny(seed=77, n=n, d=d)
    p = case.params[0]
    pre, post, comb, mixes = hcg.hc_mixes(case.x.to(DEV), p.hc_fn.to(DEV), p.hc_scale.to(DEV),
                                          p.hc_base.to(DEV), return_mixes=True)
    torch.cuda.synchronize()
    rm = oracle.mixes(bits(case.x), _np(p.hc_fn))
    err = np.abs(_np(mixes).astype(np.float64) - rm)
    assert np.all(err <= 1e-5 + 1e-5 * np.abs(rm)), err.max()
    rp, rq, rc = oracle.split_sinkhorn(rm, _np(p.hc_scale), _np(p.hc_base))
    check_fp32("pre", pre, rp)
    check_fp32("post", post, rq)
    check_fp32("comb", comb, rc)


def test_block_step_decode_config_two_sides():
    """Decode batch: 128 tokens, attention side then FFN side (FFN reads
    with the attention side's pre).  Every element; the FFN side is checked
    teacher-forced (oracle fed the GPU's own bf16 y and fp32 pre) and
    free-running."""
    case = inputs.decode()
    pa, pf = case.params
    x = case.x.to(DEV)
    a = _gpu_side(x, case.pre_mix.to(DEV), case.fs[0].to(DEV), pa.to(DEV))
    b = _gpu_side(a[1], a[2], case.fs[1].to(DEV), pf.to(DEV))
    torch.cuda.synchronize()
    ra = _oracle_side(case.x, case.pre_mix, case.fs[0], pa)
    _check_side(a, ra, tag="attn ")
    rb_tf = _oracle_side(a[1].cpu(), a[2].cpu(), case.fs[1], pf)
    _check_side(b, rb_tf, tag="ffn ")
    # free-running: the oracle's own chain
    rb = oracle.block_step(ra["y"], ra["pre"], bits(case.fs[1]), *(_np(t) for t in pf.astuple()))
    check_fp32("ffn pre (free)", b[2], rb["pre"], atol=1e-4)
    check_bf16("ffn y (free)", b[1], rb["y"], rel=1e-2,
               abs_allow=y_allowance(bits(case.fs[1]), ra["y"], rb["post"], rb["comb"], b[3], b[4])
               + 1e-2)


def test_block_step_prefill_config_sampled():
    """Prefill with outliers: 8192 tokens, two sides, 512 sampled tokens per side
    checked teacher-forced."""
    case = inputs.prefill(device=DEV)
    pa, pf = case.params
    a = _gpu_side(case.x, case.pre_mix, case.fs[0], pa)
    b = _gpu_side(a[1], a[2], case.fs[1], pf)
    torch.cuda.synchronize()
    rows = np.sort(np.random.default_rng(3).choice(case.n, 512, replace=False))
    rows_t = torch.from_numpy(rows).to(DEV)
    ra = _oracle_side(case.x.index_select(0, rows_t).cpu(), case.pre_mix.index_select(0, rows_t).cpu(),
                      case.fs[0].index_select(0, rows_t).cpu(), pa.to("cpu"))
    _check_side(tuple(t.index_select(0, rows_t).cpu() for t in a), ra, tag="attn ")
    rb = _oracle_side(a[1].index_select(0, rows_t).cpu(), a[2].index_select(0, rows_t).cpu(),
                      case.fs[1].index_select(0, rows_t).cpu(), pf.to("cpu"))
    _check_side(tuple(t.index_select(0, rows_t).cpu() for t in b), rb, tag="ffn ")


def test_block_step_long_prefill_config_sampled():
    """Long prefill: 65,536 tokens through 40 layers (80 side steps), each side
    with its own parameters and N(0,2) sublayer output, run exactly as the
    benchmark runs it.  64 sampled tokens checked teacher-forced at every side;
    the free-running oracle chain is reported as ulp differences."""
    case = inputs.long_prefill(device=DEV, materialize_f=False)
    n = case.n
    rows = np.sort(np.random.default_rng(4).choice(n, 64, replace=False))
    rows_t = torch.from_numpy(rows).to(DEV)
    x = case.x
    pm = case.pre_mix
    bufs = [torch.empty_like(x), torch.empty_like(x)]
    h_norm = torch.empty((n, case.d), dtype=torch.bfloat16, device=DEV)
    pres = [torch.empty((n, 4), device=DEV), torch.empty((n, 4), device=DEV)]
    post = torch.empty((n, 4), device=DEV)
    comb = torch.empty((n, 4, 4), device=DEV)
    free_y = bits(x.index_select(0, rows_t))
    free_pm = _np(pm.index_select(0, rows_t)).astype(np.float64)
    worst_free = 0
    for side in range(len(case.params)):
        p = case.params[side]
        f = inputs.long_prefill_f(side, n, case.d, DEV)
        y = bufs[side % 2]
        pre = pres[side % 2]
        hcg.hc_block_step(x, pm, f, *p.astuple(), h_norm=h_norm, y=y, pre_out=pre, post_out=post,
                          comb_out=comb)
        sel = lambda t: t.index_select(0, rows_t).cpu()
        fs = sel(f)
        pc = p.to("cpu")
        ref = _oracle_side(sel(x), sel(pm), fs, pc)
        _check_side((sel(h_norm), sel(y), sel(pre), sel(post), sel(comb)), ref,
                    tag="side %d " % side)
        fr = oracle.block_step(free_y, free_pm, bits(fs), *(_np(t) for t in pc.astuple()))
        free_y, free_pm = fr["y"], fr["pre"]
        x, pm = y, pre
    torch.cuda.synchronize()
    gy = oracle.bf16_to_f64(bits(x.index_select(0, rows_t)))
    ry = oracle.bf16_to_f64(free_y)
    rel = np.abs(gy - ry) / np.maximum(np.abs(ry), 1e-3)
    # free-running over 80 sides: rounding flips compound; bounded loosely
    assert np.median(rel) < 1e-2, np.median(rel)


def test_block_step_long_prefill_repeatable_bitwise():
    """The fused step is deterministic: the same side launched twice on the same
    inputs, at the full long-prefill size where the slot ring turns over many
    times, gives the same bits in every output.  A slot reloaded before its
    readers are done shows up here as scattered differences."""
    case = inputs.long_prefill(device=DEV, materialize_f=False)
    n, d = case.n, case.d
    x, pm = case.x, case.pre_mix

    def outs():
        return (torch.empty((n, d), dtype=torch.bfloat16, device=DEV), torch.empty_like(x),
                torch.empty((n, 4), device=DEV), torch.empty((n, 4), device=DEV),
                torch.empty((n, 4, 4), device=DEV))

    for side in range(3):
        p = case.params[side].astuple()
        f = inputs.long_prefill_f(side, n, d, DEV)
        a, b = outs(), outs()
        for o in (a, b):
            hcg.hc_block_step(x, pm, f, *p, h_norm=o[0], y=o[1], pre_out=o[2], post_out=o[3], comb_out=o[4])
        torch.cuda.synchronize()
        for name, u, v in zip(("h_norm", "y", "pre", "post", "comb"), a, b):
            if u.dtype == torch.bfloat16:
                u, v = u.view(torch.int16), v.view(torch.int16)
            diff = int((u != v).sum().item())
            assert diff == 0, "side %d %s: %d elements differ between two identical launches" % (side, name, diff)
        x, pm = a[1], a[2]


def test_block_step_zero_pre_mix_and_outliers():
    """pre_mix = 0 collapses to h = 0, so h_norm = 0 (eps keeps it finite)."""
    n, d = 8, 5120
    g = torch.Generator().manual_seed(9)
    x = inputs.streams(g, n, 4, d, outlier_p=0.05)
    p = inputs.side_params(g, d=d)
    f = inputs.sublayer_out(g, n, d)
    pm = torch.zeros((n, 4))
    out = _gpu_side(x.to(DEV), pm.to(DEV), f.to(DEV), p.to(DEV))
    torch.cuda.synchronize()
    assert torch.count_nonzero(out[0]).item() == 0
    _check_side(out, _oracle_side(x, pm, f, p))


def test_misaligned_device_pointer_rejected():
    n, d = 4, 5120
    x = torch.zeros((n * 4 * d + 8,), dtype=torch.bfloat16, device=DEV)[1:1 + n * 4 * d]
    st = _lib.raw("hc_pre_norm", x.data_ptr(), torch.zeros((n, 4), device=DEV).data_ptr(),
                  torch.ones(d, device=DEV).data_ptr(), n, 4, d, 1e-20,
                  torch.empty((n, d), dtype=torch.bfloat16, device=DEV).data_ptr(), None)
    assert st == 3


def test_no_kernel_reported_a_barrier_timeout():
    """Every bounded wait in the kernels above completed (the device flag is clear)."""
    torch.cuda.synchronize()
    assert _lib.raw("hc_consume_device_error", None) == 0
