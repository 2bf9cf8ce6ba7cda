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


def _raw(lib, n, hc=4, d=5120):
    return lib.hc_block_step_backward_no_workspace(
        FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000, FAKE + 0x400000, FAKE + 0x500000,
        FAKE + 0x600000, n, hc, d, 20, 1e-6, 1e-20, FAKE + 0x700000, FAKE + 0x800000, None,
        FAKE2 * 0x100, FAKE2 * 0x200, FAKE2 * 0x300, FAKE2 * 0x400, FAKE2 * 0x500, FAKE2 * 0x600,
        FAKE2 * 0x700, None)


def test_no_workspace_entry_refuses_what_does_not_fit(lib):
    assert _raw(lib, 27649) == 2          # one token beyond the fixed scratch at d = 5120
    assert _raw(lib, 16, hc=2) == 2
    assert _raw(lib, 0) == 0


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
    """27,648 tokens at d = 5120, the most the fixed scratch holds: it runs and
    equals the workspace entry bit for bit."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hc_build.build()
    _lib.load()
    dev = torch.device("cuda:0")
    n, d = 27648, 5120
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
