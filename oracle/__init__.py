"""CPU oracle for the hyper-connection residual path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library and its Python binding never import, link or call it, and it shares
no code with them.

The arithmetic lives in ``hc_oracle.c`` (plain single-threaded C, IEEE double
precision, bf16 round-to-nearest-even only where the pages store bf16).  This
module compiles it with gcc on first use and marshals numpy arrays through
ctypes.  Every function cites the page passage it follows in the C source:

* DeepSeek-V4.1 "Block(layer_id, args)" page, Code section -- hc_mixes,
  hc_pre, hc_post and the two-sided forward wiring.
* DeepSeek-V4.1 "Stream combination" page, Code section -- the split of the
  24 mix numbers and the Sinkhorn rounds.
* DeepSeek V4.1 Flash diagram -- the Cast, sigma, 2 sigma, x + eps_hc,
  First Sinkhorn Round and Sinkhorn Round blocks, and the Cast to MXFP8
  block (groups of 32, UE8M0 scale, E4M3 elements).
* DeepSeek-R1 dossier, RMSNorm records -- the RMSNorm body (the V4.1 body is
  not on the pages).

Pins: tests/test_oracle_pins.py.  Every function here is pinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hc_oracle.c")
_LIB = os.path.join(_HERE, "libhc_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile hc_oracle.c into libhc_oracle.so (gcc, -O2, no FP contraction)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c99",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i64, i32, f64 = ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.hco_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.hco_bf16_to_double.restype = f64
        lib.hco_bf16_from_double.argtypes = [f64]
        lib.hco_bf16_from_double.restype = ctypes.c_uint16
        lib.hco_mixes.argtypes = [P, P, i64, i32, i32, f64, P]
        lib.hco_split_sinkhorn.argtypes = [P, P, P, i64, i32, i32, f64, P, P, P]
        lib.hco_pre.argtypes = [P, P, i64, i32, i32, P]
        lib.hco_rmsnorm.argtypes = [P, P, i64, i32, f64, P]
        lib.hco_post.argtypes = [P, P, P, P, i64, i32, i32, P]
        lib.hco_block_step.argtypes = [P, P, P, P, P, P, P, i64, i32, i32, i32, f64, f64,
                                       P, P, P, P, P, P]
        lib.hco_side_f64.argtypes = [P, P, P, P, P, P, P, i64, i32, i32, i32, f64, f64, i32,
                                     P, P, P, P, P]
        lib.hco_side_backward_f64.argtypes = [P, P, P, P, P, P, P, i64, i32, i32, i32, f64, f64,
                                              P, P, P, i32, P, P, P, P, P, P, P]
        lib.hco_e4m3_from_double.argtypes = [f64]
        lib.hco_e4m3_from_double.restype = ctypes.c_uint8
        lib.hco_mxfp8.argtypes = [P, i64, i32, P, P]
        for name in ("hco_mixes", "hco_split_sinkhorn", "hco_pre", "hco_rmsnorm",
                     "hco_post", "hco_block_step", "hco_mxfp8", "hco_side_f64",
                     "hco_side_backward_f64"):
            getattr(lib, name).restype = i32
        _lib = lib
        return lib


def _arr(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, name):
    if rc != 0:
        raise RuntimeError("oracle %s failed with code %d" % (name, rc))


def bf16_bits(a) -> np.ndarray:
    """Accepts a uint16 array of bf16 bit patterns (returned unchanged) or a
    torch bfloat16 tensor (its bits are taken, no rounding)."""
    if hasattr(a, "view") and hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        import torch  # local: only when torch tensors are handed in
        return a.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    a = np.asarray(a)
    if a.dtype != np.uint16:
        raise TypeError("bf16 data must be passed as uint16 bit patterns")
    return a


def bf16_to_f64(bits) -> np.ndarray:
    """Exact value of bf16 bit patterns ('Cast' BF16 -> FP32 keeps every value)."""
    b = np.ascontiguousarray(bf16_bits(bits)).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_from_f64(v) -> np.ndarray:
    """Round doubles to bf16 bit patterns (nearest, ties to even)."""
    lib = _load()
    v = np.asarray(v, dtype=np.float64)
    flat = v.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)
    for i in range(flat.size):
        out[i] = lib.hco_bf16_from_double(float(flat[i]))
    return out.reshape(v.shape)


def mixes(x, hc_fn, norm_eps=1e-20):
    """a1: x [n, hc, d] bf16 bits, hc_fn [(2+hc)*hc, hc*d] fp32 -> mixes [n, mix] fp64."""
    x = bf16_bits(x)
    n, hc, d = x.shape
    mix = (2 + hc) * hc
    xa, xp = _arr(x, np.uint16)
    wa, wp = _arr(hc_fn, np.float32)
    assert wa.shape == (mix, hc * d)
    out = np.empty((n, mix), dtype=np.float64)
    _check(_load().hco_mixes(xp, wp, n, hc, d, float(norm_eps),
                             out.ctypes.data_as(ctypes.c_void_p)), "mixes")
    return out


def split_sinkhorn(mixes_, hc_scale, hc_base, hc=4, iters=20, eps=1e-6):
    """a2+a3: mixes [n, (2+hc)*hc] -> (pre [n,hc], post [n,hc], comb [n,hc,hc]) fp64."""
    ma, mp = _arr(mixes_, np.float64)
    n = ma.shape[0]
    assert ma.shape[1] == (2 + hc) * hc
    sa, sp = _arr(hc_scale, np.float32)
    ba, bp = _arr(hc_base, np.float32)
    pre = np.empty((n, hc)); post = np.empty((n, hc)); comb = np.empty((n, hc, hc))
    V = ctypes.c_void_p
    _check(_load().hco_split_sinkhorn(mp, sp, bp, n, hc, int(iters), float(eps),
                                      pre.ctypes.data_as(V), post.ctypes.data_as(V),
                                      comb.ctypes.data_as(V)), "split_sinkhorn")
    return pre, post, comb


def pre(x, pre_mix):
    """a4: x [n, hc, d] bf16 bits, pre_mix [n, hc] -> h [n, d] bf16 bits."""
    x = bf16_bits(x)
    n, hc, d = x.shape
    xa, xp = _arr(x, np.uint16)
    pa, pp = _arr(pre_mix, np.float64)
    h = np.empty((n, d), dtype=np.uint16)
    _check(_load().hco_pre(xp, pp, n, hc, d, h.ctypes.data_as(ctypes.c_void_p)), "pre")
    return h


def rmsnorm(h, w, eps=1e-20):
    """a5: h [n, d] bf16 bits, w [d] fp32 -> [n, d] bf16 bits."""
    h = bf16_bits(h)
    n, d = h.shape
    ha, hp = _arr(h, np.uint16)
    wa, wp = _arr(w, np.float32)
    out = np.empty((n, d), dtype=np.uint16)
    _check(_load().hco_rmsnorm(hp, wp, n, d, float(eps), out.ctypes.data_as(ctypes.c_void_p)),
           "rmsnorm")
    return out


def side_f64(x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, iters=20, eps=1e-6,
             norm_eps=1e-20, rounded=True):
    """The side step on double inputs x [n, hc, d], pre_mix [n, hc], f [n, d]
    (and the parameters): dict of h_norm, y, pre, post, comb (doubles).  With
    rounded=True the three bf16 casts are applied, as in block_step."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    n, hc, d = x.shape
    args = [_arr(a, np.float64) for a in (x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w)]
    out = dict(h_norm=np.empty((n, d)), y=np.empty((n, hc, d)), pre=np.empty((n, hc)),
               post=np.empty((n, hc)), comb=np.empty((n, hc, hc)))
    V = ctypes.c_void_p
    _check(_load().hco_side_f64(*(p for _, p in args), n, hc, d, int(iters), float(eps),
                                float(norm_eps), int(bool(rounded)),
                                *(out[k].ctypes.data_as(V) for k in ("h_norm", "y", "pre", "post",
                                                                     "comb"))), "side_f64")
    return out


def side_backward(x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, g_h_norm, g_y, g_pre=None,
                  iters=20, eps=1e-6, norm_eps=1e-20, rounded=True):
    """Backward of side_f64 for upstream gradients g_h_norm [n, d], g_y
    [n, hc, d], g_pre [n, hc] (None: zero) -> dict of g_x, g_pre_mix, g_f
    (per token) and g_hc_fn, g_hc_scale, g_hc_base, g_norm_w (summed over
    tokens), all doubles."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    n, hc, d = x.shape
    mix = (2 + hc) * hc
    args = [_arr(a, np.float64) for a in (x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w,
                                          g_h_norm, g_y)]
    gp = _arr(g_pre, np.float64) if g_pre is not None else (None, None)
    out = dict(g_x=np.empty((n, hc, d)), g_pre_mix=np.empty((n, hc)), g_f=np.empty((n, d)),
               g_hc_fn=np.empty((mix, hc * d)), g_hc_scale=np.empty(3), g_hc_base=np.empty(mix),
               g_norm_w=np.empty(d))
    V = ctypes.c_void_p
    _check(_load().hco_side_backward_f64(*(p for _, p in args[:7]), n, hc, d, int(iters), float(eps),
                                         float(norm_eps), args[7][1], args[8][1], gp[1],
                                         int(bool(rounded)),
                                         *(out[k].ctypes.data_as(V) for k in
                                           ("g_x", "g_pre_mix", "g_f", "g_hc_fn", "g_hc_scale",
                                            "g_hc_base", "g_norm_w"))), "side_backward")
    return out


def e4m3_from_f64(v) -> np.ndarray:
    """E4M3 bytes of doubles within [-448, 448] (nearest, ties to even)."""
    lib = _load()
    v = np.asarray(v, dtype=np.float64)
    flat = v.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    for i in range(flat.size):
        out[i] = lib.hco_e4m3_from_double(float(flat[i]))
    return out.reshape(v.shape)


def e4m3_to_f64(codes) -> np.ndarray:
    """Value of E4M3 bytes (field 0: m * 2^-9; else (1 + m/8) * 2^(e-7))."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    return sign * mag


def mxfp8(x):
    """The MXFP8 cast of bf16 rows [rows, d] (d a multiple of 32) ->
    (E4M3 codes [rows, d] uint8, UE8M0 scale bytes [rows, d/32] uint8)."""
    x = bf16_bits(x)
    rows, d = x.shape
    xa, xp = _arr(x, np.uint16)
    codes = np.empty((rows, d), dtype=np.uint8)
    scales = np.empty((rows, d // 32), dtype=np.uint8)
    _check(_load().hco_mxfp8(xp, rows, d, codes.ctypes.data_as(ctypes.c_void_p),
                             scales.ctypes.data_as(ctypes.c_void_p)), "mxfp8")
    return codes, scales


def post(f, residual, post_, comb):
    """a6: f [n, d], residual [n, hc, d] bf16 bits, post [n, hc], comb [n, hc, hc] -> y [n, hc, d]."""
    residual = bf16_bits(residual)
    f = bf16_bits(f)
    n, hc, d = residual.shape
    fa, fp = _arr(f, np.uint16)
    ra, rp = _arr(residual, np.uint16)
    pa, pp = _arr(post_, np.float64)
    ca, cp = _arr(comb, np.float64)
    y = np.empty((n, hc, d), dtype=np.uint16)
    _check(_load().hco_post(fp, rp, pp, cp, n, hc, d, y.ctypes.data_as(ctypes.c_void_p)), "post")
    return y


def block_step(x, pre_mix, f, hc_fn, hc_scale, hc_base, norm_w, iters=20, eps=1e-6,
               norm_eps=1e-20):
    """One side step a1-a6.  Returns dict with h_norm, y (bf16 bits), pre, post, comb, mixes (fp64)."""
    x = bf16_bits(x)
    f = bf16_bits(f)
    n, hc, d = x.shape
    mix = (2 + hc) * hc
    xa, xp = _arr(x, np.uint16)
    pa, pp = _arr(pre_mix, np.float64)
    fa, fp = _arr(f, np.uint16)
    wa, wp = _arr(hc_fn, np.float32)
    sa, sp = _arr(hc_scale, np.float32)
    ba, bp = _arr(hc_base, np.float32)
    na, np_ = _arr(norm_w, np.float32)
    out = dict(h_norm=np.empty((n, d), np.uint16), y=np.empty((n, hc, d), np.uint16),
               pre=np.empty((n, hc)), post=np.empty((n, hc)), comb=np.empty((n, hc, hc)),
               mixes=np.empty((n, mix)))
    V = ctypes.c_void_p
    _check(_load().hco_block_step(xp, pp, fp, wp, sp, bp, np_, n, hc, d, int(iters), float(eps),
                                  float(norm_eps),
                                  *(out[k].ctypes.data_as(V) for k in
                                    ("h_norm", "y", "pre", "post", "comb", "mixes"))),
           "block_step")
    return out


def block_layer(x, pre_mix, f_attn, f_ffn, attn_params, ffn_params, iters=20, eps=1e-6,
                norm_eps=1e-20):
    """a7: one Block's two sides (DeepSeek-V4.1 Block page, Block.forward).

    The attention side computes its own (pre, post, comb) from x, reads with
    the pre_mix handed in, writes with its own post/comb.  The FFN side does
    the same on the attention side's output, reading with the attention
    side's pre.  Returns (attention-side dict, FFN-side dict); the FFN side's
    ``pre`` is the next layer's pre_mix and its ``y`` the layer output.
    Each params tuple is (hc_fn, hc_scale, hc_base, norm_w)."""
    a = block_step(x, pre_mix, f_attn, *attn_params, iters=iters, eps=eps, norm_eps=norm_eps)
    b = block_step(a["y"], a["pre"], f_ffn, *ffn_params, iters=iters, eps=eps, norm_eps=norm_eps)
    return a, b
