"""GPU: the bounded waits report instead of hanging.

hc_selftest_barrier_timeout launches one warp that waits on an mbarrier that
nothing arrives on.  Its wait runs out (about half a minute), sets the device flag
and the kernel returns.  hc_consume_device_error must then report
HC_ERR_TIMEOUT once, the flag must be clear on the next call, and the context
must still run the library's kernels correctly."""
import pytest
import torch

import hyper_connection_residual_mixes_gb300 as hcg
from hyper_connection_residual_mixes_gb300 import _lib, inputs
from hyper_connection_residual_mixes_gb300 import build as hc_build

pytestmark = pytest.mark.gpu

HC_OK, HC_ERR_TIMEOUT = 0, 6


def test_wait_that_runs_out_is_reported_and_the_context_stays_usable():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hc_build.build()
    _lib.load()
    dev = torch.device("cuda:0")
    torch.cuda.synchronize()
    assert _lib.raw("hc_consume_device_error", None) == HC_OK
    assert _lib.raw("hc_selftest_barrier_timeout", None) == HC_OK
    assert _lib.raw("hc_consume_device_error", None) == HC_ERR_TIMEOUT
    assert _lib.raw("hc_consume_device_error", None) == HC_OK
    # the context still works: a small backward gives the same bits through both entries
    case = inputs.tiny(seed=8, n=20, d=256, device=dev)
    p = case.params[0]
    g = torch.Generator(device=dev).manual_seed(9)
    args = (case.x, case.pre_mix, case.fs[0], *p.astuple(), torch.randn((20, 256), device=dev, generator=g),
            torch.randn((20, 4, 256), device=dev, generator=g))
    a = hcg.hc_block_step_backward(*args)
    b = hcg.hc_block_step_backward_no_workspace(*args)
    torch.cuda.synchronize()
    for k in a:
        assert torch.isfinite(a[k]).all() and torch.equal(a[k], b[k]), k
    assert _lib.raw("hc_consume_device_error", None) == HC_OK
