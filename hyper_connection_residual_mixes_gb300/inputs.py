"""Seeded synthetic inputs for the hyper-connection residual path.

This module holds no arithmetic of the method: it only draws random tensors
with the shapes and distributions of the five workloads (tiny, decode batch,
Sinkhorn-only stress, prefill with outliers, long prefill).  Both the CUDA
path and the CPU oracle read the same bytes drawn here.

Distributions (``N(0, s)`` means standard deviation ``s``):
  streams x          bf16  N(0, 1)           (prefill: each entry x50 with probability 0.01)
  hc_fn              fp32  N(0, 0.01)        [(2+hc)*hc, hc*d]
  hc_base            fp32  N(0, 1)           [(2+hc)*hc]
  hc_scale           fp32  U[0.5, 2]         [3]
  pre_mix            fp32  U[0.1, 1]         [n, hc]
  sublayer output f  bf16  N(0, 1)  (long prefill: N(0, 2))
  RMSNorm weight     fp32  U[0.5, 1.5]       [d]
  Sinkhorn stress    fp32  mixes N(0, 3)     [n, (2+hc)*hc]
The parameter shapes follow the DeepSeek-V4.1 Block page (Block.__init__):
hc_fn [mix_hc, hc_mult*dim], hc_base [mix_hc], hc_scale [3], fp32.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

HC = 4
D = 5120
ITERS = 20
EPS = 1e-6
NORM_EPS = 1e-20


def mix_hc(hc: int = HC) -> int:
    return (2 + hc) * hc


@dataclass
class SideParams:
    hc_fn: torch.Tensor     # [mix, hc*d] fp32
    hc_scale: torch.Tensor  # [3] fp32
    hc_base: torch.Tensor   # [mix] fp32
    norm_w: torch.Tensor    # [d] fp32

    def to(self, device):
        return SideParams(*(t.to(device) for t in (self.hc_fn, self.hc_scale, self.hc_base,
                                                    self.norm_w)))

    def astuple(self):
        return (self.hc_fn, self.hc_scale, self.hc_base, self.norm_w)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(shape, std, g, device, dtype=torch.float32):
    return (torch.randn(shape, generator=g, device=device, dtype=torch.float32) * std).to(dtype)


def _uniform(shape, lo, hi, g, device):
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo


def side_params(g: torch.Generator, hc: int = HC, d: int = D, device="cpu",
                fn_std: float = 0.01) -> SideParams:
    m = mix_hc(hc)
    return SideParams(
        hc_fn=_normal((m, hc * d), fn_std, g, device),
        hc_scale=_uniform((3,), 0.5, 2.0, g, device),
        hc_base=_normal((m,), 1.0, g, device),
        norm_w=_uniform((d,), 0.5, 1.5, g, device),
    )


def streams(g, n, hc=HC, d=D, device="cpu", std=1.0, outlier_p=0.0, outlier_scale=50.0):
    """x [n, hc, d] bf16.  With outlier_p > 0 each entry is independently
    scaled by outlier_scale with that probability (seeded Bernoulli mask)."""
    x = torch.randn((n, hc, d), generator=g, device=device, dtype=torch.float32) * std
    if outlier_p > 0.0:
        mask = torch.rand((n, hc, d), generator=g, device=device) < outlier_p
        x = torch.where(mask, x * outlier_scale, x)
    return x.to(torch.bfloat16)


def sublayer_out(g, n, d=D, device="cpu", std=1.0):
    return _normal((n, d), std, g, device, torch.bfloat16)


def pre_mix(g, n, hc=HC, device="cpu"):
    return _uniform((n, hc), 0.1, 1.0, g, device)


@dataclass
class BlockCase:
    """Inputs of one or more side steps of the block."""
    name: str
    x: torch.Tensor                 # [n, hc, d] bf16
    pre_mix: torch.Tensor           # [n, hc] fp32
    fs: list                        # per side: f [n, d] bf16
    params: list                    # per side: SideParams
    hc: int = HC
    d: int = D
    iters: int = ITERS
    eps: float = EPS
    norm_eps: float = NORM_EPS

    @property
    def n(self):
        return self.x.shape[0]


def tiny(device="cpu", seed=0, n=16, d=D, hc=HC) -> BlockCase:
    """Tiny: B=1, T=16: one side step (seed 0)."""
    g = _gen(seed, device)
    x = streams(g, n, hc, d, device)
    p = side_params(g, hc, d, device)
    pm = pre_mix(g, n, hc, device)
    f = sublayer_out(g, n, d, device)
    return BlockCase("tiny", x, pm, [f], [p], hc, d)


def decode(device="cpu", seed=1, n=128, d=D, hc=HC) -> BlockCase:
    """Decode batch: B=128, T=1: attention side then FFN side (seed 1)."""
    g = _gen(seed, device)
    x = streams(g, n, hc, d, device)
    pa = side_params(g, hc, d, device)
    pf = side_params(g, hc, d, device)
    pm = pre_mix(g, n, hc, device)
    fa = sublayer_out(g, n, d, device)
    ff = sublayer_out(g, n, d, device)
    return BlockCase("decode", x, pm, [fa, ff], [pa, pf], hc, d)


def prefill(device="cpu", seed=3, n=8192, d=D, hc=HC) -> BlockCase:
    """Prefill: B=1, T=8192, outliers: attention side then FFN side (seed 3)."""
    g = _gen(seed, device)
    x = streams(g, n, hc, d, device, outlier_p=0.01)
    pa = side_params(g, hc, d, device)
    pf = side_params(g, hc, d, device)
    pm = pre_mix(g, n, hc, device)
    fa = sublayer_out(g, n, d, device)
    ff = sublayer_out(g, n, d, device)
    return BlockCase("prefill", x, pm, [fa, ff], [pa, pf], hc, d)


def long_prefill(device="cpu", seed=4, n=65536, layers=40, d=D, hc=HC,
                 materialize_f=True) -> BlockCase:
    """Long prefill: B=4, T=16384 (65,536 tokens), 40 layers = 80 side steps,
    each side with its own parameters and its own N(0, 2) sublayer output (seed 4).
    With materialize_f=False the f list holds per-side seeds instead of
    tensors (see long_prefill_f)."""
    g = _gen(seed, device)
    x = streams(g, n, hc, d, device)
    pm = pre_mix(g, n, hc, device)
    params = [side_params(g, hc, d, device) for _ in range(2 * layers)]
    fs = []
    for side in range(2 * layers):
        if materialize_f:
            fs.append(long_prefill_f(side, n, d, device, seed))
        else:
            fs.append(None)
    return BlockCase("long_prefill", x, pm, fs, params, hc, d)


def long_prefill_f(side: int, n: int, d: int = D, device="cpu", seed: int = 4):
    """The sublayer stand-in output of one side of the long prefill, drawn
    from its own generator so that any one side can be regenerated alone."""
    g = _gen(seed * 1000003 + 7919 * (side + 1), device)
    return sublayer_out(g, n, d, device, std=2.0)


def sinkhorn_stress(device="cpu", seed=2, n=1 << 20, hc=HC):
    """Sinkhorn-only stress: mixes [n, 24] N(0, 3), hc_scale U[0.5, 2], hc_base N(0, 1)."""
    g = _gen(seed, device)
    m = _normal((n, mix_hc(hc)), 3.0, g, device)
    scale = _uniform((3,), 0.5, 2.0, g, device)
    base = _normal((mix_hc(hc),), 1.0, g, device)
    return m, scale, base


def bf16_bits_np(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (no rounding)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")
