"""GPU: the side step recorded into a CUDA graph and replayed.

A serving loop issues its small-batch side steps as graph replays; the
kernels must then compute exactly what an eager call computes.  hc_block_step
(the cluster kernel at four streams, the tcgen05 path at eight) and the
backward are captured once and replayed on fresh inputs copied into the
captured buffers; every output must equal the eager call's bit for bit.  So
is the chain, whose cross-CTA flags take a new epoch at every replay (written
on the device into its state buffer just before each launch)."""
import pytest
import torch

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


def _same(a, b):
    assert a.dtype == b.dtype and a.shape == b.shape
    if a.dtype == torch.bfloat16:
        a, b = a.view(torch.int16), b.view(torch.int16)
    elif a.dtype == torch.float32:
        a, b = a.view(torch.int32), b.view(torch.int32)
    assert torch.equal(a, b)


def _inputs(seed, n, hc, d):
    g = torch.Generator(device=DEV).manual_seed(seed)
    x = inputs.streams(g, n, hc, d, device=DEV)
    pm = inputs.pre_mix(g, n, hc, device=DEV)
    fs = [inputs.sublayer_out(g, n, d, device=DEV) for _ in range(2)]
    ps = [inputs.side_params(g, hc, d, device=DEV) for _ in range(2)]
    return x, pm, fs, ps


@pytest.mark.parametrize("n,hc,d", [(16, 4, 5120), (128, 4, 5120), (1000, 4, 1024), (2000, 8, 256)])
def test_block_step_graph_replay(n, hc, d):
    """Two side steps (the decode wiring: the second side reads the first
    side's y with its pre) captured once; each replay on new streams equals
    the eager calls."""
    x, pm, fs, ps = _inputs(70 + n, n, hc, d)
    h = [torch.empty((n, d), dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    y = [torch.empty_like(x) for _ in range(2)]
    pre = [torch.empty_like(pm) for _ in range(2)]

    def two_sides():
        hcg.hc_block_step(x, pm, fs[0], *ps[0].astuple(), h_norm=h[0], y=y[0], pre_out=pre[0])
        hcg.hc_block_step(y[0], pre[0], fs[1], *ps[1].astuple(), h_norm=h[1], y=y[1], pre_out=pre[1])

    two_sides()  # one eager call first: kernel attributes, cached occupancy
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            two_sides()
    torch.cuda.synchronize()
    for rep in range(3):
        x2, pm2, fs2, _ = _inputs(900 + 7 * rep + n, n, hc, d)
        x.copy_(x2), pm.copy_(pm2), fs[0].copy_(fs2[0]), fs[1].copy_(fs2[1])
        graph.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (*h, *y, *pre)]
        two_sides()
        torch.cuda.synchronize()
        for a, b in zip(got, (*h, *y, *pre)):
            _same(a, b)
    assert _lib.raw("hc_consume_device_error", None) == 0


def test_backward_graph_replay():
    """hc_block_step_backward (four streams, its eight launches) captured with
    its workspace and replayed."""
    n, hc, d = 257, 4, 1024
    x, pm, fs, ps = _inputs(81, n, hc, d)
    g = torch.Generator(device=DEV).manual_seed(82)
    g_hn = torch.randn((n, d), device=DEV, generator=g)
    g_y = torch.randn((n, hc, d), device=DEV, generator=g)
    ws = torch.empty(_lib.load().hc_block_step_backward_workspace_bytes(n, hc, d), dtype=torch.uint8,
                     device=DEV)
    eager = hcg.hc_block_step_backward(x, pm, fs[0], *ps[0].astuple(), g_hn, g_y, workspace=ws)
    torch.cuda.synchronize()
    out = {k: torch.empty_like(v) for k, v in eager.items()}

    def bwd():
        r = hcg.hc_block_step_backward(x, pm, fs[0], *ps[0].astuple(), g_hn, g_y, workspace=ws)
        for k in out:
            out[k].copy_(r[k])

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            bwd()
    torch.cuda.synchronize()
    g_y.mul_(-0.5)
    graph.replay()
    torch.cuda.synchronize()
    ref = hcg.hc_block_step_backward(x, pm, fs[0], *ps[0].astuple(), g_hn, g_y, workspace=ws)
    torch.cuda.synchronize()
    for k in ref:
        _same(out[k], ref[k])
    assert _lib.raw("hc_consume_device_error", None) == 0


def test_chain_graph_replay():
    """The chain (its first launch, a side with the next side's weights, the
    last side) captured once; each replay on new streams and sublayer outputs
    equals hc_block_step side after side, bit for bit.  Each replay draws new
    epochs for the cross-CTA flags, while the state buffers still hold the
    flags of the replay before it."""
    n, hc, d = 200, 4, 1024
    x, pm, fs, ps = _inputs(83, n, hc, d)
    p0, p1 = ps
    st = [hcg.chain_state(n, d, DEV) for _ in range(2)]
    h = [torch.empty((n, d), dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    y = [torch.empty_like(x) for _ in range(2)]
    pre = [torch.empty_like(pm) for _ in range(2)]

    def chain():
        hcg.hc_chain_begin(x, pm, p0.hc_fn, p0.hc_scale, p0.hc_base, state_out=st[0], pre_out=pre[0])
        hcg.hc_chain_side(x, fs[0], st[0], p0.norm_w, p1.hc_fn, p1.hc_scale, p1.hc_base, h_norm=h[0], y=y[0],
                          state_out=st[1], pre_out=pre[1])
        hcg.hc_chain_side(y[0], fs[1], st[1], p1.norm_w, h_norm=h[1], y=y[1])

    chain()  # one eager call first
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            chain()
    torch.cuda.synchronize()
    for rep in range(4):
        x2, pm2, fs2, _ = _inputs(950 + 3 * rep, n, hc, d)
        x.copy_(x2), pm.copy_(pm2), fs[0].copy_(fs2[0]), fs[1].copy_(fs2[1])
        graph.replay()
        torch.cuda.synchronize()
        h0, y0, q0 = hcg.hc_block_step(x, pm, fs[0], *p0.astuple())
        h1, y1, q1 = hcg.hc_block_step(y0, q0, fs[1], *p1.astuple())
        torch.cuda.synchronize()
        for a, b in ((h[0], h0), (y[0], y0), (pre[0], q0), (h[1], h1), (y[1], y1), (pre[1], q1)):
            _same(a, b)
    assert _lib.raw("hc_consume_device_error", None) == 0


def test_chain_model_order_graph_replay():
    """The model's inner loop as one CUDA graph: per side, hc_chain_norm (the
    side's h_norm), a stand-in sublayer on it (torch on the GPU), and the
    side's chain launch (y_i and side i + 1's bf16 h), over three sides.
    Replays on new streams equal the same sequence run eagerly, bit for bit."""
    n, hc, d, S = 256, 4, 2048, 3
    g = torch.Generator(device=DEV).manual_seed(85)
    x = inputs.streams(g, n, hc, d, device=DEV)
    pm = inputs.pre_mix(g, n, hc, device=DEV)
    ps = [inputs.side_params(g, hc, d, device=DEV) for _ in range(S)]
    st = [hcg.chain_state(n, d, DEV) for _ in range(2)]
    hp = [torch.empty((n, d), dtype=torch.bfloat16, device=DEV) for _ in range(2)]
    hn = [torch.empty((n, d), dtype=torch.bfloat16, device=DEV) for _ in range(S)]
    fo = [torch.empty((n, d), dtype=torch.bfloat16, device=DEV) for _ in range(S)]
    ys = [torch.empty_like(x) for _ in range(S)]
    pre = [torch.empty_like(pm) for _ in range(S)]

    def model():
        p0 = ps[0]
        hcg.hc_chain_begin(x, pm, p0.hc_fn, p0.hc_scale, p0.hc_base, state_out=st[0], pre_out=pre[0],
                           h_pre_out=hp[0])
        xi = x
        for i in range(S):
            hcg.hc_chain_norm(hp[i % 2], st[i % 2], ps[i].norm_w, h_norm=hn[i])
            fo[i].copy_((2.0 * torch.tanh(hn[i].float())).to(torch.bfloat16))  # the sublayer stand-in
            if i + 1 < S:
                q = ps[i + 1]
                hcg.hc_chain_side(xi, fo[i], st[i % 2], ps[i].norm_w, q.hc_fn, q.hc_scale, q.hc_base, y=ys[i],
                                  state_out=st[(i + 1) % 2], pre_out=pre[i + 1], h_pre_out=hp[(i + 1) % 2])
            else:
                hcg.hc_chain_side(xi, fo[i], st[i % 2], ps[i].norm_w, y=ys[i], write_h_norm=False)
            xi = ys[i]

    model()  # one eager call first
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            model()
    torch.cuda.synchronize()
    for rep in range(3):
        g2 = torch.Generator(device=DEV).manual_seed(990 + rep)
        x.copy_(inputs.streams(g2, n, hc, d, device=DEV))
        pm.copy_(inputs.pre_mix(g2, n, hc, device=DEV))
        graph.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (*hn, *fo, *ys, *pre)]
        model()
        torch.cuda.synchronize()
        for a, b in zip(got, (*hn, *fo, *ys, *pre)):
            _same(a, b)
    assert _lib.raw("hc_consume_device_error", None) == 0
