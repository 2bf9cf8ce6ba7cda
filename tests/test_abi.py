"""The C ABI without a GPU: the library loads, exports every symbol that
include/hc.h declares, and its host-side validation rejects bad arguments
before any launch (no CUDA call is made on these paths)."""
import ctypes
import os
import re
import subprocess

import pytest

from hyper_connection_residual_mixes_gb300 import _lib
from hyper_connection_residual_mixes_gb300 import build as hc_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hc.h")


@pytest.fixture(scope="module")
def lib():
    hc_build.build()
    return _lib.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(hc_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_five_entry_points():
    names = declared_functions()
    for n in ("hc_mixes", "hc_split_sinkhorn", "hc_pre_norm", "hc_post", "hc_block_step",
              "hc_status_string", "hc_last_cuda_error", "hc_version"):
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\s[TW]\s+(\w+)$", out, flags=re.M))
    for name in declared_functions():
        assert name in exported, "%s declared in hc.h but not exported" % name
        getattr(lib, name)  # resolvable through ctypes too
    # the binding knows every declared entry point, with the same name
    assert set(declared_functions()) == set(_lib.SIGNATURES)


def test_status_strings(lib):
    for code, name in _lib.STATUS.items():
        s = lib.hc_status_string(code).decode()
        assert s.startswith(name)
    assert lib.hc_last_cuda_error() == 0
    assert lib.hc_version() >= 100


FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first
FAKE2 = 0x20000


def _block(**kw):
    a = dict(x=FAKE, pre_mix=FAKE + 0x100000, f=FAKE + 0x200000, hc_fn=FAKE + 0x300000,
             hc_scale=FAKE + 0x400000, hc_base=FAKE + 0x500000, norm_w=FAKE + 0x600000,
             n=16, hc=4, d=5120, iters=20, eps=1e-6, norm_eps=1e-20, h_norm=FAKE2 * 0x100,
             y=FAKE2 * 0x200, pre_out=FAKE2 * 0x300, post_out=None, comb_out=None, stream=None)
    a.update(kw)
    return _lib.raw("hc_block_step", a["x"], a["pre_mix"], a["f"], a["hc_fn"], a["hc_scale"],
                    a["hc_base"], a["norm_w"], a["n"], a["hc"], a["d"], a["iters"], a["eps"],
                    a["norm_eps"], a["h_norm"], a["y"], a["pre_out"], a["post_out"],
                    a["comb_out"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(n=-1), 1),
    (dict(hc=3), 2),
    (dict(hc=0), 1),
    (dict(d=5121), 2),
    (dict(d=32), 2),
    (dict(d=32768), 2),
    (dict(d=0), 1),
    (dict(iters=0), 1),
    (dict(eps=-1.0), 1),
    (dict(eps=float("nan")), 1),
    (dict(norm_eps=float("inf")), 1),
    (dict(x=None), 1),
    (dict(pre_out=None), 1),
    (dict(f=None), 1),
    (dict(x=FAKE + 8), 3),
    (dict(post_out=FAKE2 * 0x400 + 4), 3),
    (dict(y=FAKE + 64), 4),                       # y overlaps x
    (dict(pre_out=FAKE2 * 0x100 + 16), 4),        # pre_out overlaps h_norm
])
def test_block_step_validation(lib, kw, expect):
    assert _block(**kw) == expect


def test_block_step_empty_is_ok(lib):
    assert _block(n=0, x=None, y=None) == 0


def test_split_sinkhorn_validation(lib):
    r = lambda **kw: _lib.raw("hc_split_sinkhorn", kw.get("mixes", FAKE), FAKE + 0x1000,
                              FAKE + 0x2000, kw.get("n", 4), kw.get("hc", 4), kw.get("iters", 20),
                              kw.get("eps", 1e-6), kw.get("pre", FAKE2), FAKE2 + 0x1000,
                              FAKE2 + 0x2000, None)
    assert r(n=0) == 0
    assert r(n=-3) == 1
    assert r(hc=3) == 2    # stream counts 2, 4 and 8 are compiled
    assert r(hc=16) == 2
    assert r(iters=0) == 1
    assert r(mixes=None) == 1
    assert r(mixes=FAKE + 4) == 3
    assert r(pre=FAKE + 16) == 4


def test_pre_norm_and_post_validation(lib):
    assert _lib.raw("hc_pre_norm", FAKE, FAKE + 0x100000, FAKE + 0x200000, 2, 4, 5120, 1e-20,
                    FAKE + 0x100, None) == 4  # out overlaps x
    assert _lib.raw("hc_pre_norm", FAKE, FAKE + 0x100000, FAKE + 0x200000, 2, 4, 100, 1e-20,
                    FAKE2 * 0x100, None) == 2
    assert _lib.raw("hc_post", FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000, 2, 4,
                    5120, None, None) == 1
    assert _lib.raw("hc_post", FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000, 2, 4,
                    5120, FAKE + 0x100010, None) == 4
    assert _lib.raw("hc_mixes", FAKE, FAKE + 0x100000, FAKE + 0x200000, FAKE + 0x300000, 2, 4,
                    5120, 20, 1e-6, 1e-20, FAKE2 * 0x100, FAKE2 * 0x200, FAKE2 * 0x300,
                    FAKE2 * 0x300 + 8, None) == 3


def _state_bytes(n=16, d=5120):
    return _lib.load().hc_chain_state_bytes(n, 4, d)


def _side(**kw):
    a = dict(x=FAKE, f=FAKE + 0x100000, state_in=FAKE + 0x200000, norm_w=FAKE + 0x300000,
             fn=FAKE + 0x400000, scale=FAKE + 0x500000, base=FAKE + 0x600000, n=16, hc=4, d=5120,
             iters=20, eps=1e-6, norm_eps=1e-20, h_norm=FAKE2 * 0x100, y=FAKE2 * 0x200,
             state_out=FAKE2 * 0x300, state_bytes=None, pre_out=None, h_pre_out=None, stream=None)
    a.update(kw)
    if a["state_bytes"] is None:
        a["state_bytes"] = _state_bytes(max(a["n"], 0), a["d"])
    return _lib.raw("hc_chain_side", a["x"], a["f"], a["state_in"], a["norm_w"], a["fn"], a["scale"],
                    a["base"], a["n"], a["hc"], a["d"], a["iters"], a["eps"], a["norm_eps"], a["h_norm"],
                    a["y"], a["state_out"], a["state_bytes"], a["pre_out"], a["h_pre_out"], a["stream"])


def _begin(**kw):
    a = dict(x=FAKE, pre_mix=FAKE + 0x100000, fn=FAKE + 0x200000, scale=FAKE + 0x300000,
             base=FAKE + 0x400000, n=16, hc=4, d=5120, iters=20, eps=1e-6, norm_eps=1e-20,
             state_out=FAKE2 * 0x100, state_bytes=None, pre_out=None, h_pre_out=None, stream=None)
    a.update(kw)
    if a["state_bytes"] is None:
        a["state_bytes"] = _state_bytes(max(a["n"], 0), a["d"])
    return _lib.raw("hc_chain_begin", a["x"], a["pre_mix"], a["fn"], a["scale"], a["base"], a["n"],
                    a["hc"], a["d"], a["iters"], a["eps"], a["norm_eps"], a["state_out"], a["state_bytes"],
                    a["pre_out"], a["h_pre_out"], a["stream"])


# Every case below fails validation (or has n == 0), so nothing is launched even
# on a machine with a GPU: the pointers are not real allocations.
@pytest.mark.parametrize("kw,expect", [
    (dict(scale=None), 1),                 # next-side weights come all together or not at all
    (dict(base=None), 1),
    (dict(state_out=None), 1),             # a next side needs a state to write
    (dict(state_bytes=64), 1),             # ... of hc_chain_state_bytes bytes
    (dict(h_pre_out=FAKE2 * 0x400), 1),    # the next side's h excludes this side's h_norm
    (dict(h_norm=None, h_pre_out=FAKE2 * 0x400 + 8), 3),
    (dict(h_norm=None, h_pre_out=FAKE + 0x10), 4),   # it overlaps x
    (dict(d=320), 2),                      # the chain needs d a multiple of 1024 ...
    (dict(d=8192), 2),                     # ... and d <= 7168
    (dict(hc=3), 2),
    (dict(state_in=FAKE + 0x200008), 3),
    (dict(y=FAKE + 64), 4),                # y overlaps x
    (dict(state_out=FAKE + 0x200010), 4),  # state_out overlaps state_in
    (dict(y=None), 1),
    (dict(n=-1), 1),
])
def test_chain_side_validation(lib, kw, expect):
    assert _side(**kw) == expect


def test_chain_side_last_needs_no_state_and_empty_is_ok(lib):
    # the last side: no next weights, no state to write (still validated, then empty)
    assert _side(n=0, fn=None, scale=None, base=None, state_out=None) == 0
    assert _side(n=0) == 0
    # the last side has no next side whose h it could write
    assert _side(fn=None, scale=None, base=None, state_out=None, h_norm=None, h_pre_out=FAKE2 * 0x400) == 1


def test_chain_state_bytes(lib):
    """Coefficient rows (128 bytes per token, rounded up to 256), then 16 x 28
    fp32 partial sums per token, then 16 eight-byte flags per 64-token tile,
    then a 16-byte header (the epoch of the launch that writes the buffer)."""
    for n in (1, 64, 65, 1000, 65536):
        tiles = -(-n // 64)
        assert lib.hc_chain_state_bytes(n, 4, 5120) == ((128 * n + 255) // 256) * 256 + 1792 * n + 128 * tiles + 16
    assert lib.hc_chain_state_bytes(16, 4, 320) == 0      # not served by the chain
    assert lib.hc_chain_state_bytes(16, 2, 5120) == 0
    assert lib.hc_chain_state_bytes(-1, 4, 5120) == 0


@pytest.mark.parametrize("kw,expect", [
    (dict(d=2048 + 64), 2),
    (dict(state_out=None), 1),
    (dict(state_bytes=1024), 1),
    (dict(state_out=FAKE2 * 0x100 + 4), 3),
    (dict(state_out=FAKE + 0x100), 4),     # state_out overlaps x
    (dict(h_pre_out=FAKE + 0x100), 4),     # h_pre_out overlaps x
    (dict(h_pre_out=FAKE2 * 0x200 + 2), 3),
    (dict(iters=0), 1),
])
def test_chain_begin_validation(lib, kw, expect):
    assert _begin(**kw) == expect


def test_binding_rejects_cpu_tensors():
    import torch
    import hyper_connection_residual_mixes_gb300 as hcg
    x = torch.zeros(2, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        hcg.hc_pre_norm(x, torch.zeros(2, 4), torch.ones(64))


def _cast(**kw):
    a = dict(x=FAKE, rows=16, d=5120, codes=FAKE2 * 0x100, scales=FAKE2 * 0x200, stream=None)
    a.update(kw)
    return _lib.raw("hc_mxfp8_cast", a["x"], a["rows"], a["d"], a["codes"], a["scales"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(d=48), 2),                        # groups of 32 channels
    (dict(d=0), 1),
    (dict(rows=-1), 1),
    (dict(codes=None), 1),
    (dict(scales=None), 1),
    (dict(x=FAKE + 2), 3),
    (dict(codes=FAKE2 * 0x100 + 8), 3),
    (dict(codes=FAKE + 0x100), 4),          # codes overlap the input
    (dict(scales=FAKE2 * 0x100 + 0x40), 4),  # scales overlap the codes
])
def test_mxfp8_cast_validation(lib, kw, expect):
    assert _cast(**kw) == expect


def test_mxfp8_cast_empty_and_unaligned_scales_ok(lib):
    assert _cast(rows=0) == 0
    assert _cast(rows=0, scales=FAKE2 * 0x200 + 1) == 0


def _pnq(**kw):
    a = dict(x=FAKE, pre_mix=FAKE + 0x100000, norm_w=FAKE + 0x200000, n=16, hc=4, d=5120,
             norm_eps=1e-20, h_norm=None, codes=FAKE2 * 0x100, scales=FAKE2 * 0x200, stream=None)
    a.update(kw)
    return _lib.raw("hc_pre_norm_mxfp8", a["x"], a["pre_mix"], a["norm_w"], a["n"], a["hc"], a["d"],
                    a["norm_eps"], a["h_norm"], a["codes"], a["scales"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(hc=3), 2),
    (dict(d=96), 2),
    (dict(norm_eps=-1.0), 1),
    (dict(codes=None), 1),
    (dict(scales=None), 1),
    (dict(h_norm=FAKE2 * 0x300 + 4), 3),
    (dict(codes=FAKE + 0x80), 4),            # codes overlap x
    (dict(h_norm=FAKE2 * 0x100), 4),         # h_norm overlaps the codes
    (dict(n=-1), 1),
])
def test_pre_norm_mxfp8_validation(lib, kw, expect):
    assert _pnq(**kw) == expect


def test_pre_norm_mxfp8_empty_is_ok(lib):
    assert _pnq(n=0) == 0
    assert _pnq(n=0, h_norm=FAKE2 * 0x300) == 0


def _bwd(**kw):
    a = dict(x=FAKE, pm=FAKE + 0x100000, f=FAKE + 0x200000, fn=FAKE + 0x300000, sc=FAKE + 0x400000,
             base=FAKE + 0x500000, w=FAKE + 0x600000, n=16, hc=4, d=5120, iters=20, eps=1e-6,
             norm_eps=1e-20, g_hn=FAKE + 0x700000, g_y=FAKE + 0x800000, g_pre=None,
             g_x=FAKE2 * 0x100, g_pm=FAKE2 * 0x200, g_f=FAKE2 * 0x300, g_fn=FAKE2 * 0x400,
             g_sc=FAKE2 * 0x500, g_base=FAKE2 * 0x600, g_w=FAKE2 * 0x700, ws=FAKE2 * 0x800,
             ws_bytes=1 << 30, stream=None)
    a.update(kw)
    return _lib.raw("hc_block_step_backward", a["x"], a["pm"], a["f"], a["fn"], a["sc"], a["base"],
                    a["w"], a["n"], a["hc"], a["d"], a["iters"], a["eps"], a["norm_eps"], a["g_hn"],
                    a["g_y"], a["g_pre"], a["g_x"], a["g_pm"], a["g_f"], a["g_fn"], a["g_sc"],
                    a["g_base"], a["g_w"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(hc=3), 2),                         # the backward is compiled for 2, 4 and 8 streams
    (dict(hc=16), 2),
    (dict(hc=2, ws_bytes=1000), 1),          # the workspace asked for depends on hc
    (dict(hc=8, ws_bytes=1000), 1),
    (dict(iters=0), 1),
    (dict(iters=129), 1),
    (dict(ws=None), 1),
    (dict(ws_bytes=1000), 1),                # smaller than the library asks for
    (dict(g_x=None), 1),
    (dict(g_pre=FAKE2 * 0x900 + 4), 3),
    (dict(g_f=FAKE + 0x200000 + 64), 4),     # g_f overlaps f
    (dict(n=-1), 1),
])
def test_block_step_backward_validation(lib, kw, expect):
    assert _bwd(**kw) == expect


def test_block_step_backward_workspace_size(lib):
    f = lib.hc_block_step_backward_workspace_bytes
    assert f(0, 4, 5120) >= 0
    assert f(1000, 4, 5120) > f(10, 4, 5120) > 0
    assert f(16, 3, 5120) == 0 and f(16, 4, 100) == 0
    assert f(16, 2, 5120) > 0 and f(16, 8, 5120) > f(16, 4, 5120)
    assert _bwd(n=0) == 0 and _bwd(n=0, hc=2) == 0 and _bwd(n=0, hc=8) == 0


def _norm(**kw):
    a = dict(h_pre=FAKE, state=FAKE + 0x100000, norm_w=FAKE + 0x200000, n=16, d=5120,
             h_norm=FAKE2 * 0x100, codes=None, scales=None, stream=None)
    a.update(kw)
    return _lib.raw("hc_chain_norm", a["h_pre"], a["state"], a["norm_w"], a["n"], a["d"], a["h_norm"],
                    a["codes"], a["scales"], a["stream"])


@pytest.mark.parametrize("kw,expect", [
    (dict(h_norm=None), 1),                        # nothing to write
    (dict(codes=FAKE2 * 0x200), 1),                # codes and scales come together
    (dict(scales=FAKE2 * 0x300), 1),
    (dict(d=100), 2),
    (dict(n=-1), 1),
    (dict(h_pre=None), 1),
    (dict(state=FAKE + 0x100004), 3),
    (dict(h_norm=FAKE + 0x100), 4),                # h_norm overlaps h_pre
    (dict(codes=FAKE2 * 0x200, scales=FAKE + 0x200010), 4),  # scales overlap norm_w
    (dict(n=0), 0),
])
def test_chain_norm_validation(lib, kw, expect):
    assert _norm(**kw) == expect
