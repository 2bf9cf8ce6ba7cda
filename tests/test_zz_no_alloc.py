"""hc_block_step_backward_no_workspace: the backward with the library's own
fixed device scratch, so a call allocates nothing.

Without a GPU: the entry point is exported and refuses what does not fit
before touching the device.  On the GPU: its results equal
hc_block_step_backward's (caller workspace) bit for bit, and a call leaves
the device's free memory unchanged."""
import pytest
import torch

import hyper_connection_residual_mixes_gb300 as hcg
from hyper_connection_residual_mixes_gb300 import _lib, inputs
from hyper_connection_residual_mixes_gb300 import build as hc_build

FAKE = 0x10000
FAKE2 = 0x20000


@pytest.fixture(scope="module")
def lib():
    hc_build.build()
    return _lib.load()


def _raw(lib, n, hc=4, d=5120, iters=20):
    return lib.hc_block_step_backward_no_workspace(
        FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000, FAKE + 0x400000, FAKE + 0x500000,
        FAKE + 0x600000, n, hc, d, iters, 1e-6, 1e-20, FAKE + 0x700000, FAKE + 0x800000, None,
        FAKE2 * 0x100, FAKE2 * 0x200, FAKE2 * 0x300, FAKE2 * 0x400, FAKE2 * 0x500, FAKE2 * 0x600,
        FAKE2 * 0x700, None)


def test_no_workspace_entry_refuses_what_does_not_fit(lib):
    assert _raw(lib, 24577) == 2          # one token beyond the fixed scratch at d = 5120
    assert _raw(lib, 16, hc=2) == 2
    assert _raw(lib, 0) == 0


def _documented_workspace_bytes(n, d):
    """The backward's workspace at four streams as include/hc.h states it:
    156 fp32 per token, then per block of 1,024 tokens the partial sums of
    g_hc_fn (24 x 4d), g_norm_w (d) and g_hc_base / g_hc_scale (32), then the
    three bf16 parts of hc_fn (80 rows of 4d bf16, i.e. 160 d floats)."""
    blocks = -(-n // 1024)
    return 4 * (156 * n + blocks * (24 * 4 * d + d + 32) + 160 * d)


@pytest.mark.parametrize("d", [1024, 2048, 5120])
def test_no_workspace_capacity_edge_at_other_widths(lib, d):
    """The largest batch that fits the fixed 64 MiB scratch, from the documented
    formula: it passes the capacity check, one more token does not.  Both calls
    pass sinkhorn_iters = 0, so the one that passes the capacity check stops at
    argument validation (or, without a GPU, at the scratch lookup) and nothing
    is launched."""
    cap = 64 << 20
    n = 1
    while _documented_workspace_bytes(2 * n, d) <= cap:
        n *= 2
    lo, hi = n, 2 * n                    # fits at lo, not at hi
    while hi - lo > 1:
        mid = (lo + hi) // 2
        lo, hi = (mid, hi) if _documented_workspace_bytes(mid, d) <= cap else (lo, mid)
    assert lib.hc_block_step_backward_workspace_bytes(lo, 4, d) == _documented_workspace_bytes(lo, d)
    assert _raw(lib, lo, d=d, iters=0) != 2
    assert _raw(lib, lo + 1, d=d, iters=0) == 2
    if d == 5120:
        assert lo == 24576


def test_no_workspace_wrapper_checks_every_input():
    """The Python wrapper refuses a wrong dtype, a non-contiguous tensor or a
    wrong shape on any input before it calls the library, exactly as the
    workspace wrapper does (CPU tensors here: the dtype, layout and shape checks
    come before the device check)."""
    n, d = 6, 64
    g = torch.Generator().manual_seed(1)
    x = inputs.streams(g, n, 4, d)
    p = inputs.side_params(g, d=d)
    good = dict(x=x, pre_mix=inputs.pre_mix(g, n), f=inputs.sublayer_out(g, n, d),
                hc_fn=p.hc_fn, hc_scale=p.hc_scale, hc_base=p.hc_base, norm_w=p.norm_w,
                g_h_norm=torch.randn(n, d), g_y=torch.randn(n, 4, d), g_pre=torch.randn(n, 4))
    bad_cases = [
        ("g_y", good["g_y"].to(torch.bfloat16), TypeError),
        ("g_h_norm", good["g_h_norm"].to(torch.bfloat16), TypeError),
        ("pre_mix", torch.randn(4, n).t(), ValueError),            # not contiguous
        ("g_y", torch.randn(n, 4, d + 64), ValueError),             # wrong shape
        ("hc_fn", torch.randn(24, 4 * d + 64), ValueError),
        ("f", good["f"].float(), TypeError),
    ]
    for fn in (hcg.hc_block_step_backward_no_workspace, hcg.hc_block_step_backward):
        for name, t, err in bad_cases:
            kw = dict(good)
            kw[name] = t
            with pytest.raises(err, match=name):
                fn(**kw)
        with pytest.raises(ValueError, match="CUDA"):
            fn(**good)


@pytest.mark.gpu
@pytest.mark.parametrize("n,d", [(300, 1024), (1030, 256), (16, 5120)])
def test_no_workspace_equals_workspace_and_allocates_nothing(n, d):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hc_build.build()
    _lib.load()
    dev = torch.device("cuda:0")
    case = inputs.tiny(seed=3 + n, n=n, d=d, device=dev)
    p = case.params[0]
    g = torch.Generator(device=dev).manual_seed(n)
    g_hn = torch.randn((n, d), device=dev, generator=g)
    g_y = torch.randn((n, 4, d), device=dev, generator=g)
    g_pre = torch.randn((n, 4), device=dev, generator=g)
    args = (case.x, case.pre_mix, case.fs[0], *p.astuple(), g_hn, g_y, g_pre)
    ref = hcg.hc_block_step_backward(*args)
    got = hcg.hc_block_step_backward_no_workspace(*args)   # the module and its scratch are loaded now
    torch.cuda.synchronize()
    for k in ref:
        assert torch.equal(got[k], ref[k]), k
    outs = {k: torch.empty_like(v) for k, v in got.items()}
    free0, _ = torch.cuda.mem_get_info(dev)
    st = _lib.raw("hc_block_step_backward_no_workspace", *(t.data_ptr() for t in args[:7]), n, 4, d, 20,
                  1e-6, 1e-20, g_hn.data_ptr(), g_y.data_ptr(), g_pre.data_ptr(),
                  *(outs[k].data_ptr() for k in ("g_x", "g_pre_mix", "g_f", "g_hc_fn", "g_hc_scale",
                                                   "g_hc_base", "g_norm_w")), None)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(dev)
    assert st == 0
    assert free1 == free0
    for k in ref:
        assert torch.equal(outs[k], ref[k]), k


@pytest.mark.gpu
def test_no_workspace_at_its_capacity():
    """24,576 tokens at d = 5120, the most the fixed scratch holds: it runs and
    equals the workspace entry bit for bit."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hc_build.build()
    _lib.load()
    dev = torch.device("cuda:0")
    n, d = 24576, 5120
    g = torch.Generator(device=dev).manual_seed(31)
    x = inputs.streams(g, n, 4, d, device=dev)
    pm = inputs.pre_mix(g, n, device=dev)
    f = inputs.sublayer_out(g, n, d, device=dev)
    p = inputs.side_params(g, d=d, device=dev)
    args = (x, pm, f, *p.astuple(), torch.randn((n, d), device=dev, generator=g),
            torch.randn((n, 4, d), device=dev, generator=g))
    ref = hcg.hc_block_step_backward(*args)
    got = hcg.hc_block_step_backward_no_workspace(*args)
    torch.cuda.synchronize()
    for k in ref:
        assert torch.equal(got[k], ref[k]), k
    assert _lib.raw("hc_consume_device_error", None) == 0
