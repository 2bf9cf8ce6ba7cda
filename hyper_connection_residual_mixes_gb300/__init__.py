"""GB300-native hyper-connection residual path (DeepSeek-V4.1-style blocks).

A thin PyTorch binding over libhc.so (C ABI in include/hc.h).  Each function
has the name of the C entry point it calls, checks and marshals tensors
(device, dtype, contiguity, shapes), allocates outputs with PyTorch when they
are not supplied, and enqueues the call on the current CUDA stream.  Every
step of the path runs in the CUDA kernels; there is no CPU or PyTorch
fallback, and calling with CPU tensors raises.

Shapes (hc = 4 streams, d = 5120 in the released model, mix = (2+hc)*hc = 24):
  x, residual, y  [..., hc, d] bf16;  f, h_norm [..., d] bf16
  hc_fn [mix, hc*d] fp32;  hc_base [mix];  hc_scale [3];  norm_w [d] fp32
  pre, post, pre_mix [..., hc] fp32;  comb [..., hc, hc] fp32;  mixes [..., mix] fp32
"""
from __future__ import annotations

import torch

from . import _lib
from ._lib import HcError

__all__ = ["hc_mixes", "hc_split_sinkhorn", "hc_pre_norm", "hc_post", "hc_block_step",
           "hc_chain_begin", "hc_chain_side", "hc_chain_norm", "chain_state", "hc_mxfp8_cast",
           "hc_pre_norm_mxfp8",
           "hc_block_step_backward", "hc_block_step_backward_no_workspace", "STATE_FLOATS",
           "HcError", "library_path", "version"]

HC_EPS = 1e-6
NORM_EPS = 1e-20
SINKHORN_ITERS = 20
STATE_FLOATS = 32  # per-token state row of the chained side steps (HC_STATE_FLOATS)


def library_path() -> str:
    return _lib.LIB_PATH


def version() -> int:
    return _lib.load().hc_version()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(t, name, dtype, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor (libhc has no CPU path)" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))
    return t


def _out(t, name, shape, dtype, device):
    if t is None:
        return torch.empty(shape, dtype=dtype, device=device)
    _check(t, name, dtype, device)
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    return t


def hc_split_sinkhorn(mixes, hc_scale, hc_base, hc_mult=4, sinkhorn_iters=SINKHORN_ITERS,
                      eps=HC_EPS, pre=None, post=None, comb=None, stream=None):
    """a2-a3: mixes [..., (2+hc)*hc] fp32 -> (pre [..., hc], post [..., hc], comb [..., hc, hc])."""
    _check(mixes, "mixes", torch.float32)
    dev = mixes.device
    _check(hc_scale, "hc_scale", torch.float32, dev)
    _check(hc_base, "hc_base", torch.float32, dev)
    lead = tuple(mixes.shape[:-1])
    n = mixes.numel() // mixes.shape[-1] if mixes.dim() else 0
    pre = _out(pre, "pre", lead + (hc_mult,), torch.float32, dev)
    post = _out(post, "post", lead + (hc_mult,), torch.float32, dev)
    comb = _out(comb, "comb", lead + (hc_mult, hc_mult), torch.float32, dev)
    with torch.cuda.device(dev):
        _lib.call("hc_split_sinkhorn", _ptr(mixes), _ptr(hc_scale), _ptr(hc_base), n, hc_mult,
                  sinkhorn_iters, eps, _ptr(pre), _ptr(post), _ptr(comb), _stream(stream))
    return pre, post, comb


def hc_mixes(x, hc_fn, hc_scale, hc_base, sinkhorn_iters=SINKHORN_ITERS, eps=HC_EPS,
             norm_eps=NORM_EPS, pre=None, post=None, comb=None, mixes_out=None,
             return_mixes=False, stream=None):
    """a1-a3: x [..., hc, d] bf16 -> (pre, post, comb) [+ mixes when return_mixes]."""
    _check(x, "x", torch.bfloat16)
    dev = x.device
    hc, d = x.shape[-2], x.shape[-1]
    lead = tuple(x.shape[:-2])
    n = x.numel() // (hc * d) if x.numel() else 0
    mix = (2 + hc) * hc
    _check(hc_fn, "hc_fn", torch.float32, dev)
    _check(hc_scale, "hc_scale", torch.float32, dev)
    _check(hc_base, "hc_base", torch.float32, dev)
    pre = _out(pre, "pre", lead + (hc,), torch.float32, dev)
    post = _out(post, "post", lead + (hc,), torch.float32, dev)
    comb = _out(comb, "comb", lead + (hc, hc), torch.float32, dev)
    if return_mixes:
        mixes_out = _out(mixes_out, "mixes_out", lead + (mix,), torch.float32, dev)
    elif mixes_out is not None:
        _out(mixes_out, "mixes_out", lead + (mix,), torch.float32, dev)
    with torch.cuda.device(dev):
        _lib.call("hc_mixes", _ptr(x), _ptr(hc_fn), _ptr(hc_scale), _ptr(hc_base), n, hc, d,
                  sinkhorn_iters, eps, norm_eps, _ptr(pre), _ptr(post), _ptr(comb),
                  _ptr(mixes_out), _stream(stream))
    if return_mixes:
        return pre, post, comb, mixes_out
    return pre, post, comb


def hc_pre_norm(x, pre_mix, norm_w, norm_eps=NORM_EPS, out=None, stream=None):
    """a4-a5: x [..., hc, d] bf16, pre_mix [..., hc] fp32 -> RMSNorm(hc_pre) [..., d] bf16."""
    _check(x, "x", torch.bfloat16)
    dev = x.device
    hc, d = x.shape[-2], x.shape[-1]
    lead = tuple(x.shape[:-2])
    n = x.numel() // (hc * d) if x.numel() else 0
    _check(pre_mix, "pre_mix", torch.float32, dev)
    _check(norm_w, "norm_w", torch.float32, dev)
    out = _out(out, "out", lead + (d,), torch.bfloat16, dev)
    with torch.cuda.device(dev):
        _lib.call("hc_pre_norm", _ptr(x), _ptr(pre_mix), _ptr(norm_w), n, hc, d, norm_eps,
                  _ptr(out), _stream(stream))
    return out


def _backward_args(x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, g_h_norm, g_y, g_pre):
    """Checks every input of the two backward entry points before anything is
    launched: dtype, contiguity and shape of each tensor first, then that all
    of them are CUDA tensors on x's device.  Returns (device, hc, d, lead, n)."""
    if not isinstance(x, torch.Tensor):
        raise TypeError("x must be a torch.Tensor")
    if x.dim() < 2:
        raise ValueError("x must be [..., hc, d]")
    hc, d = x.shape[-2], x.shape[-1]
    lead = tuple(x.shape[:-2])
    mix = (2 + hc) * hc
    specs = [(x, "x", torch.bfloat16, tuple(x.shape)),
             (pre_mix, "pre_mix", torch.float32, lead + (hc,)),
             (f, "f", torch.bfloat16, lead + (d,)),
             (hc_fn, "hc_fn", torch.float32, (mix, hc * d)),
             (hc_scale, "hc_scale", torch.float32, (3,)),
             (hc_base, "hc_base", torch.float32, (mix,)),
             (norm_w, "norm_w", torch.float32, (d,)),
             (g_h_norm, "g_h_norm", torch.float32, lead + (d,)),
             (g_y, "g_y", torch.float32, tuple(x.shape))]
    if g_pre is not None:
        specs.append((g_pre, "g_pre", torch.float32, lead + (hc,)))
    for t, nm, dt, shape in specs:
        if not isinstance(t, torch.Tensor):
            raise TypeError("%s must be a torch.Tensor" % nm)
        if t.dtype != dt:
            raise TypeError("%s must be %s, got %s" % (nm, dt, t.dtype))
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % nm)
        if tuple(t.shape) != shape:
            raise ValueError("%s has shape %s, expected %s" % (nm, tuple(t.shape), shape))
    dev = x.device
    for t, nm, dt, shape in specs:
        _check(t, nm, dt, dev)
    n = x.numel() // (hc * d) if x.numel() else 0
    return dev, hc, d, lead, n


def _backward_outputs(x, hc_fn, hc_base, dev, hc, d, lead):
    return dict(g_x=torch.empty(tuple(x.shape), dtype=torch.float32, device=dev),
                g_pre_mix=torch.empty(lead + (hc,), dtype=torch.float32, device=dev),
                g_f=torch.empty(lead + (d,), dtype=torch.float32, device=dev),
                g_hc_fn=torch.empty(tuple(hc_fn.shape), dtype=torch.float32, device=dev),
                g_hc_scale=torch.empty(3, dtype=torch.float32, device=dev),
                g_hc_base=torch.empty(tuple(hc_base.shape), dtype=torch.float32, device=dev),
                g_norm_w=torch.empty(d, dtype=torch.float32, device=dev))


_GRAD_KEYS = ("g_x", "g_pre_mix", "g_f", "g_hc_fn", "g_hc_scale", "g_hc_base", "g_norm_w")


def hc_block_step_backward(x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, g_h_norm, g_y,
                           g_pre=None, sinkhorn_iters=SINKHORN_ITERS, eps=HC_EPS, norm_eps=NORM_EPS,
                           workspace=None, stream=None):
    """The backward of hc_block_step (fp32 gradients): returns a dict of
    g_x [..., hc, d], g_pre_mix [..., hc], g_f [..., d] and the parameter
    gradients g_hc_fn, g_hc_scale, g_hc_base, g_norm_w summed over tokens.
    workspace: a uint8 device tensor of at least the size the library asks
    for (allocated here when None)."""
    dev, hc, d, lead, n = _backward_args(x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w,
                                         g_h_norm, g_y, g_pre)
    out = _backward_outputs(x, hc_fn, hc_base, dev, hc, d, lead)
    need = _lib.load().hc_block_step_backward_workspace_bytes(n, hc, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    else:
        _check(workspace, "workspace", torch.uint8, dev)
    with torch.cuda.device(dev):
        _lib.call("hc_block_step_backward", _ptr(x), _ptr(pre_mix), _ptr(f), _ptr(hc_fn),
                  _ptr(hc_scale), _ptr(hc_base), _ptr(norm_w), n, hc, d, sinkhorn_iters, eps,
                  norm_eps, _ptr(g_h_norm), _ptr(g_y), _ptr(g_pre),
                  *(_ptr(out[k]) for k in _GRAD_KEYS),
                  _ptr(workspace), workspace.numel(), _stream(stream))
    return out


def hc_block_step_backward_no_workspace(x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, g_h_norm,
                                        g_y, g_pre=None, sinkhorn_iters=SINKHORN_ITERS, eps=HC_EPS,
                                        norm_eps=NORM_EPS, stream=None):
    """hc_block_step_backward with the library's own fixed scratch (no
    workspace argument, nothing allocated by the call); same results.  The
    inputs are checked exactly as hc_block_step_backward checks them."""
    dev, hc, d, lead, n = _backward_args(x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w,
                                         g_h_norm, g_y, g_pre)
    out = _backward_outputs(x, hc_fn, hc_base, dev, hc, d, lead)
    with torch.cuda.device(dev):
        _lib.call("hc_block_step_backward_no_workspace", _ptr(x), _ptr(pre_mix), _ptr(f), _ptr(hc_fn),
                  _ptr(hc_scale), _ptr(hc_base), _ptr(norm_w), n, hc, d, sinkhorn_iters, eps,
                  norm_eps, _ptr(g_h_norm), _ptr(g_y), _ptr(g_pre),
                  *(_ptr(out[k]) for k in _GRAD_KEYS), _stream(stream))
    return out


def hc_mxfp8_cast(x, codes=None, scales=None, stream=None):
    """The MXFP8 cast of bf16 rows x [..., d] (d a multiple of 32) ->
    (E4M3 codes [..., d] uint8, UE8M0 scale bytes [..., d/32] uint8)."""
    _check(x, "x", torch.bfloat16)
    dev = x.device
    d = x.shape[-1]
    lead = tuple(x.shape[:-1])
    rows = x.numel() // d if x.numel() else 0
    codes = _out(codes, "codes", lead + (d,), torch.uint8, dev)
    scales = _out(scales, "scales", lead + (d // 32,), torch.uint8, dev)
    with torch.cuda.device(dev):
        _lib.call("hc_mxfp8_cast", _ptr(x), rows, d, _ptr(codes), _ptr(scales), _stream(stream))
    return codes, scales


def hc_pre_norm_mxfp8(x, pre_mix, norm_w, norm_eps=NORM_EPS, h_norm=None, codes=None, scales=None,
                      return_h_norm=False, stream=None):
    """a4-a5 then the MXFP8 cast of h_norm in one pass: x [..., hc, d] bf16,
    pre_mix [..., hc] -> (codes [..., d] uint8, scales [..., d/32] uint8)
    [+ h_norm [..., d] bf16 when return_h_norm or h_norm is given]."""
    _check(x, "x", torch.bfloat16)
    dev = x.device
    hc, d = x.shape[-2], x.shape[-1]
    lead = tuple(x.shape[:-2])
    n = x.numel() // (hc * d) if x.numel() else 0
    _check(pre_mix, "pre_mix", torch.float32, dev)
    _check(norm_w, "norm_w", torch.float32, dev)
    if return_h_norm or h_norm is not None:
        h_norm = _out(h_norm, "h_norm", lead + (d,), torch.bfloat16, dev)
    codes = _out(codes, "codes", lead + (d,), torch.uint8, dev)
    scales = _out(scales, "scales", lead + (d // 32,), torch.uint8, dev)
    with torch.cuda.device(dev):
        _lib.call("hc_pre_norm_mxfp8", _ptr(x), _ptr(pre_mix), _ptr(norm_w), n, hc, d, norm_eps,
                  _ptr(h_norm) if h_norm is not None else None, _ptr(codes), _ptr(scales),
                  _stream(stream))
    if h_norm is not None:
        return codes, scales, h_norm
    return codes, scales


def hc_post(f, residual, post, comb, y=None, stream=None):
    """a6: f [..., d] bf16, residual [..., hc, d] bf16, post [..., hc], comb [..., hc, hc] -> y."""
    _check(residual, "residual", torch.bfloat16)
    dev = residual.device
    hc, d = residual.shape[-2], residual.shape[-1]
    n = residual.numel() // (hc * d) if residual.numel() else 0
    _check(f, "f", torch.bfloat16, dev)
    _check(post, "post", torch.float32, dev)
    _check(comb, "comb", torch.float32, dev)
    y = _out(y, "y", tuple(residual.shape), torch.bfloat16, dev)
    with torch.cuda.device(dev):
        _lib.call("hc_post", _ptr(f), _ptr(residual), _ptr(post), _ptr(comb), n, hc, d, _ptr(y),
                  _stream(stream))
    return y


def hc_block_step(x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w,
                  sinkhorn_iters=SINKHORN_ITERS, eps=HC_EPS, norm_eps=NORM_EPS,
                  h_norm=None, y=None, pre_out=None, post_out=None, comb_out=None,
                  return_post_comb=False, stream=None):
    """Fused side step a1-a6.  Returns (h_norm, y, pre_out) or, with
    return_post_comb, (h_norm, y, pre_out, post_out, comb_out)."""
    _check(x, "x", torch.bfloat16)
    dev = x.device
    hc, d = x.shape[-2], x.shape[-1]
    lead = tuple(x.shape[:-2])
    n = x.numel() // (hc * d) if x.numel() else 0
    for t, nm, dt in ((pre_mix, "pre_mix", torch.float32), (f, "f", torch.bfloat16),
                      (hc_fn, "hc_fn", torch.float32), (hc_scale, "hc_scale", torch.float32),
                      (hc_base, "hc_base", torch.float32), (norm_w, "norm_w", torch.float32)):
        _check(t, nm, dt, dev)
    h_norm = _out(h_norm, "h_norm", lead + (d,), torch.bfloat16, dev)
    y = _out(y, "y", tuple(x.shape), torch.bfloat16, dev)
    pre_out = _out(pre_out, "pre_out", lead + (hc,), torch.float32, dev)
    if return_post_comb:
        post_out = _out(post_out, "post_out", lead + (hc,), torch.float32, dev)
        comb_out = _out(comb_out, "comb_out", lead + (hc, hc), torch.float32, dev)
    with torch.cuda.device(dev):
        _lib.call("hc_block_step", _ptr(x), _ptr(pre_mix), _ptr(f), _ptr(hc_fn), _ptr(hc_scale),
                  _ptr(hc_base), _ptr(norm_w), n, hc, d, sinkhorn_iters, eps, norm_eps,
                  _ptr(h_norm), _ptr(y), _ptr(pre_out), _ptr(post_out), _ptr(comb_out),
                  _stream(stream))
    if return_post_comb:
        return h_norm, y, pre_out, post_out, comb_out
    return h_norm, y, pre_out


def chain_state(n, d, device, hc=4):
    """A state buffer of the chain for n tokens of width d: an fp32 tensor of
    hc_chain_state_bytes / 128 rows of 32 floats.  Its first n rows are the
    coefficient rows (state[:n]); the rows after them are the kernels' scratch."""
    nbytes = _lib.load().hc_chain_state_bytes(n, hc, d)
    if nbytes == 0:
        raise ValueError("the chain does not serve n=%d, hc=%d, d=%d" % (n, hc, d))
    return torch.empty(((nbytes + 127) // 128, STATE_FLOATS), dtype=torch.float32, device=device)


def _state_or_new(state, name, n, d, hc, dev):
    """The caller's state buffer (checked), a new one, or None where the chain
    does not serve the shape (the library then refuses the call)."""
    if state is not None:
        return _state_arg(state, name, n, d, hc, dev)
    return chain_state(n, d, dev, hc) if _lib.load().hc_chain_state_bytes(n, hc, d) else None


def _state_arg(state, name, n, d, hc, dev):
    _check(state, name, torch.float32, dev)
    need = _lib.load().hc_chain_state_bytes(n, hc, d)
    if state.dim() != 2 or state.shape[1] != STATE_FLOATS or state.numel() * 4 < need:
        raise ValueError("%s must be a chain_state(n, d) buffer (%d bytes, rows of %d floats)"
                         % (name, need, STATE_FLOATS))
    return state


def hc_chain_begin(x, pre_mix, hc_fn, hc_scale, hc_base, sinkhorn_iters=SINKHORN_ITERS,
                   eps=HC_EPS, norm_eps=NORM_EPS, state_out=None, pre_out=None, h_pre_out=None,
                   stream=None):
    """a1-a3 of the first side of a chain and its RMSNorm statistic.  Returns
    the state buffer of the first side (chain_state; its first n rows are the
    coefficient rows) and fills pre_out [n, hc] and h_pre_out [n, d] (the
    side's bf16 h, for hc_chain_norm) when given."""
    _check(x, "x", torch.bfloat16)
    dev = x.device
    hc, d = x.shape[-2], x.shape[-1]
    lead = tuple(x.shape[:-2])
    n = x.numel() // (hc * d) if x.numel() else 0
    for t, nm in ((pre_mix, "pre_mix"), (hc_fn, "hc_fn"), (hc_scale, "hc_scale"), (hc_base, "hc_base")):
        _check(t, nm, torch.float32, dev)
    state_out = _state_or_new(state_out, "state_out", n, d, hc, dev)
    if pre_out is not None:
        pre_out = _out(pre_out, "pre_out", lead + (hc,), torch.float32, dev)
    if h_pre_out is not None:
        h_pre_out = _out(h_pre_out, "h_pre_out", lead + (d,), torch.bfloat16, dev)
    with torch.cuda.device(dev):
        _lib.call("hc_chain_begin", _ptr(x), _ptr(pre_mix), _ptr(hc_fn), _ptr(hc_scale), _ptr(hc_base),
                  n, hc, d, sinkhorn_iters, eps, norm_eps, _ptr(state_out),
                  state_out.numel() * 4 if state_out is not None else 0,
                  _ptr(pre_out), _ptr(h_pre_out), _stream(stream))
    return state_out


def hc_chain_side(x, f, state_in, norm_w, hc_fn_next=None, hc_scale_next=None, hc_base_next=None,
                  sinkhorn_iters=SINKHORN_ITERS, eps=HC_EPS, norm_eps=NORM_EPS, h_norm=None, y=None,
                  state_out=None, pre_out=None, h_pre_out=None, write_h_norm=True, stream=None):
    """a4-a6 of side i from its state, fused with a1-a3 of side i + 1 on the y it
    produces.  Returns (h_norm, y, state_out): h_norm is None when it is not
    written (write_h_norm=False, or model order with h_pre_out given);
    state_out is None for the last side (no next-side weights).  h_pre_out
    [n, d] receives side i + 1's bf16 h (model order)."""
    _check(x, "x", torch.bfloat16)
    dev = x.device
    hc, d = x.shape[-2], x.shape[-1]
    lead = tuple(x.shape[:-2])
    n = x.numel() // (hc * d) if x.numel() else 0
    _check(f, "f", torch.bfloat16, dev)
    _check(state_in, "state_in", torch.float32, dev)
    _check(norm_w, "norm_w", torch.float32, dev)
    nxt = hc_fn_next is not None
    if nxt:
        for t, nm in ((hc_fn_next, "hc_fn_next"), (hc_scale_next, "hc_scale_next"),
                      (hc_base_next, "hc_base_next")):
            _check(t, nm, torch.float32, dev)
        state_out = _state_or_new(state_out, "state_out", n, d, hc, dev)
        if pre_out is not None:
            pre_out = _out(pre_out, "pre_out", lead + (hc,), torch.float32, dev)
        if h_pre_out is not None:
            h_pre_out = _out(h_pre_out, "h_pre_out", lead + (d,), torch.bfloat16, dev)
    else:
        state_out = pre_out = None
        if h_pre_out is not None:
            raise ValueError("h_pre_out needs the next side's weights")
    if h_pre_out is not None or not write_h_norm:
        if h_norm is not None:
            raise ValueError("h_norm is not written in model order (h_pre_out) or with write_h_norm=False")
    else:
        h_norm = _out(h_norm, "h_norm", lead + (d,), torch.bfloat16, dev)
    y = _out(y, "y", tuple(x.shape), torch.bfloat16, dev)
    with torch.cuda.device(dev):
        _lib.call("hc_chain_side", _ptr(x), _ptr(f), _ptr(state_in), _ptr(norm_w), _ptr(hc_fn_next),
                  _ptr(hc_scale_next), _ptr(hc_base_next), n, hc, d, sinkhorn_iters, eps, norm_eps,
                  _ptr(h_norm), _ptr(y), _ptr(state_out), state_out.numel() * 4 if state_out is not None else 0,
                  _ptr(pre_out), _ptr(h_pre_out), _stream(stream))
    return h_norm, y, state_out


def hc_chain_norm(h_pre, state, norm_w, h_norm=None, codes=None, scales=None, mxfp8=False,
                  return_h_norm=True, stream=None):
    """a5 of the chain in model order: h_norm = bf16((h * rs) * norm_w) from the
    bf16 h a chain launch wrote and the statistic in its state.  Returns
    h_norm, or with mxfp8 (or codes / scales given) (h_norm or None, codes,
    scales) -- the MXFP8 cast of h_norm."""
    _check(h_pre, "h_pre", torch.bfloat16)
    dev = h_pre.device
    d = h_pre.shape[-1]
    lead = tuple(h_pre.shape[:-1])
    n = h_pre.numel() // d if h_pre.numel() else 0
    _check(state, "state", torch.float32, dev)
    _check(norm_w, "norm_w", torch.float32, dev)
    if state.dim() != 2 or state.shape[1] != STATE_FLOATS or state.shape[0] < n:
        raise ValueError("state must hold the %d coefficient rows of the chain" % n)
    cast = mxfp8 or codes is not None or scales is not None
    if return_h_norm or h_norm is not None or not cast:
        h_norm = _out(h_norm, "h_norm", lead + (d,), torch.bfloat16, dev)
    if cast:
        codes = _out(codes, "codes", lead + (d,), torch.uint8, dev)
        scales = _out(scales, "scales", lead + (d // 32,), torch.uint8, dev)
    with torch.cuda.device(dev):
        _lib.call("hc_chain_norm", _ptr(h_pre), _ptr(state), _ptr(norm_w), n, d, _ptr(h_norm),
                  _ptr(codes), _ptr(scales), _stream(stream))
    if cast:
        return h_norm, codes, scales
    return h_norm
