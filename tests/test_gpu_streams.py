"""GPU: stream counts other than four (hc = 2 and hc = 8) against the oracle.

The pages' split + Sinkhorn kernel is written for any hc_mult (Stream
combination page, Code section: the kernel's hc parameter); the released
model uses 4.  The standalone paths (hc_split_sinkhorn, hc_mixes,
hc_pre_norm, hc_pre_norm_mxfp8, hc_post and hc_block_step through the
whole-token kernel below 128 tokens, through the token-tiled projection from
128 tokens on) are compiled for 2, 4 and 8 streams; the cluster kernel and the
chain stay at 4 (other counts are refused with HC_ERR_UNSUPPORTED).  The
tiled cases include four streams at widths the cluster kernel does not serve
(3072, and 5184, whose 20,736 columns leave a ragged last stage) and ragged
last token tiles.  Tolerances are those of test_gpu_parity.py."""
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


@pytest.mark.parametrize("hc", [2, 8])
@pytest.mark.parametrize("iters", [1, 20])
def test_split_sinkhorn_hc(hc, iters):
    mix = (2 + hc) * hc
    g = torch.Generator().manual_seed(900 + hc + iters)
    m = torch.randn((777, mix), generator=g) * 3.0
    scale = torch.rand(3, generator=g) * 1.5 + 0.5
    base = torch.randn(mix, generator=g)
    pre, post, comb = hcg.hc_split_sinkhorn(m.to(DEV), scale.to(DEV), base.to(DEV), hc_mult=hc,
                                            sinkhorn_iters=iters)
    torch.cuda.synchronize()
    assert comb.shape == (777, hc, hc)
    rp, rq, rc = oracle.split_sinkhorn(_np(m).astype(np.float64), _np(scale), _np(base), hc=hc,
                                       iters=iters)
    check_fp32("pre", pre, rp)
    check_fp32("post", post, rq)
    check_fp32("comb", comb, rc)


@pytest.mark.parametrize("hc,n,d", [(2, 37, 5120), (8, 37, 5120), (2, 9, 64), (8, 5, 1024),
                                    (2, 300, 5120), (8, 200, 5120), (8, 129, 64), (2, 1000, 1024),
                                    (4, 300, 3072), (4, 257, 5184), (8, 160, 2048)])
def test_mixes_hc(hc, n, d):
    case = inputs.tiny(seed=40 + n, n=n, d=d, hc=hc)
    p = case.params[0]
    pre, post, comb, mixes = hcg.hc_mixes(case.x.to(DEV), p.hc_fn.to(DEV), p.hc_scale.to(DEV),
                                          p.hc_base.to(DEV), return_mixes=True)
    torch.cuda.synchronize()
    rm = oracle.mixes(bits(case.x), _np(p.hc_fn))
    err = np.abs(_np(mixes).astype(np.float64) - rm)
    assert np.all(err <= 1e-5 + 1e-5 * np.abs(rm)), err.max()
    rp, rq, rc = oracle.split_sinkhorn(rm, _np(p.hc_scale), _np(p.hc_base), hc=hc)
    check_fp32("pre", pre, rp)
    check_fp32("post", post, rq)
    check_fp32("comb", comb, rc)


@pytest.mark.parametrize("hc,n,d", [(2, 300, 5120), (8, 300, 5120), (8, 7, 64)])
def test_pre_norm_and_post_hc(hc, n, d):
    g = torch.Generator().manual_seed(60 + hc)
    x = inputs.streams(g, n, hc, d, outlier_p=0.01)
    pm = inputs.pre_mix(g, n, hc)
    w = torch.rand(d, generator=g) + 0.5
    out = hcg.hc_pre_norm(x.to(DEV), pm.to(DEV), w.to(DEV))
    f = inputs.sublayer_out(g, n, d, std=2.0)
    post = torch.rand((n, hc), generator=g) * 2
    comb = torch.rand((n, hc, hc), generator=g)
    y = hcg.hc_post(f.to(DEV), x.to(DEV), post.to(DEV), comb.to(DEV))
    codes, scales, h2 = hcg.hc_pre_norm_mxfp8(x.to(DEV), pm.to(DEV), w.to(DEV), return_h_norm=True)
    torch.cuda.synchronize()
    ref = oracle.rmsnorm(oracle.pre(bits(x), _np(pm).astype(np.float64)), _np(w))
    check_bf16("h_norm", out, ref, abs_allow=h_norm_allowance(x, _np(pm), _np(w), ref))
    ref_y = oracle.post(bits(f), bits(x), _np(post).astype(np.float64), _np(comb).astype(np.float64))
    check_bf16("y", y, ref_y, abs_allow=y_allowance(f, x, _np(post), _np(comb)))
    assert torch.equal(h2.view(torch.int16), out.view(torch.int16))
    rc, rs = oracle.mxfp8(bits(h2.cpu()))
    assert np.array_equal(_np(codes), rc) and np.array_equal(_np(scales), rs)


@pytest.mark.parametrize("hc,n,d", [(2, 16, 5120), (8, 16, 5120), (2, 41, 1024), (8, 9, 2048),
                                    (2, 300, 5120), (8, 160, 5120), (8, 130, 64), (4, 200, 3072),
                                    (4, 131, 5184),
                                    # the tcgen05 a1-a3 kernel (its split weights fit h_norm): ragged
                                    # 128-token tiles and 32-row boxes; K split over CTAs (all but
                                    # the two at d = 64), partial slices of 8 or more stages
                                    (2, 100, 64), (2, 513, 1024), (4, 333, 3072), (4, 700, 5184),
                                    (8, 1925, 256), (4, 321, 64), (2, 4099, 5120),
                                    # at least one 128-token tile per CTA slot: K not split, CTAs
                                    # owning two tiles (the second ragged) and finishing in place
                                    (8, 20011, 64), (4, 40003, 64), (2, 40000, 64)])
def test_block_step_hc(hc, n, d):
    case = inputs.tiny(seed=70 + n + hc, n=n, d=d, hc=hc)
    p = case.params[0]
    h_norm, y, pre, post, comb = hcg.hc_block_step(case.x.to(DEV), case.pre_mix.to(DEV),
                                                   case.fs[0].to(DEV), *p.to(DEV).astuple(),
                                                   return_post_comb=True)
    torch.cuda.synchronize()
    xb, fb = bits(case.x), bits(case.fs[0])
    pm = _np(case.pre_mix).astype(np.float64)
    ref = oracle.block_step(xb, pm, fb, *(_np(t) for t in p.astuple()))
    check_fp32("pre", pre, ref["pre"])
    check_fp32("post", post, ref["post"])
    check_fp32("comb", comb, ref["comb"])
    check_bf16("h_norm", h_norm, ref["h_norm"],
               abs_allow=h_norm_allowance(xb, pm, _np(p.norm_w), ref["h_norm"]))
    check_bf16("y", y, ref["y"], abs_allow=y_allowance(fb, xb, ref["post"], ref["comb"], post, comb))


def test_chain_refuses_other_stream_counts():
    case = inputs.tiny(n=4, hc=2)
    p = case.params[0]
    with pytest.raises(hcg.HcError):
        hcg.hc_chain_begin(case.x.to(DEV), case.pre_mix.to(DEV), p.hc_fn.to(DEV),
                           p.hc_scale.to(DEV), p.hc_base.to(DEV))
