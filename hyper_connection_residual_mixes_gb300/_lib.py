"""ctypes loader for libhc.so (the C ABI declared in include/hc.h).

Argument marshalling only: no arithmetic of the method happens in Python.
The library must have been built (``__graft_entry__.build()`` or
``python -m hyper_connection_residual_mixes_gb300.build``); a missing
library raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libhc.so")

_lock = threading.Lock()
_lib = None

P = ctypes.c_void_p
I64 = ctypes.c_int64
I32 = ctypes.c_int
F32 = ctypes.c_float

# name -> argtypes, in the order of include/hc.h
SIGNATURES = {
    "hc_status_string": [I32],
    "hc_last_cuda_error": [],
    "hc_version": [],
    "hc_consume_device_error": [P],
    "hc_selftest_barrier_timeout": [P],
    "hc_mixes": [P, P, P, P, I64, I32, I32, I32, F32, F32, P, P, P, P, P],
    "hc_split_sinkhorn": [P, P, P, I64, I32, I32, F32, P, P, P, P],
    "hc_pre_norm": [P, P, P, I64, I32, I32, F32, P, P],
    "hc_mxfp8_cast": [P, I64, I32, P, P, P],
    "hc_block_step_backward_workspace_bytes": [I64, I32, I32],
    "hc_block_step_backward_no_workspace": [P, P, P, P, P, P, P, I64, I32, I32, I32, F32, F32,
                                            P, P, P, P, P, P, P, P, P, P, P],
    "hc_block_step_backward": [P, P, P, P, P, P, P, I64, I32, I32, I32, F32, F32, P, P, P,
                               P, P, P, P, P, P, P, P, ctypes.c_size_t, P],
    "hc_pre_norm_mxfp8": [P, P, P, I64, I32, I32, F32, P, P, P, P],
    "hc_post": [P, P, P, P, I64, I32, I32, P, P],
    "hc_block_step": [P, P, P, P, P, P, P, I64, I32, I32, I32, F32, F32, P, P, P, P, P, P],
    "hc_chain_state_bytes": [I64, I32, I32],
    "hc_chain_begin": [P, P, P, P, P, I64, I32, I32, I32, F32, F32, P, ctypes.c_size_t, P, P, P],
    "hc_chain_side": [P, P, P, P, P, P, P, I64, I32, I32, I32, F32, F32, P, P, P, ctypes.c_size_t,
                      P, P, P],
    "hc_chain_norm": [P, P, P, I64, I32, P, P, P, P],
}

STATUS = {
    0: "HC_OK",
    1: "HC_ERR_INVALID_ARG",
    2: "HC_ERR_UNSUPPORTED",
    3: "HC_ERR_MISALIGNED",
    4: "HC_ERR_ALIAS",
    5: "HC_ERR_CUDA",
    6: "HC_ERR_TIMEOUT",
}


class HcError(RuntimeError):
    def __init__(self, name, status, message, cuda_error=0):
        self.status = status
        self.cuda_error = cuda_error
        super().__init__("%s failed: %s (status %d%s)" % (
            name, message, status, ", cudaError %d" % cuda_error if cuda_error else ""))


def load():
    """Load libhc.so once; raise if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libhc.so is not built (expected at %s); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        for name, argtypes in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = argtypes
            fn.restype = I32
        lib.hc_status_string.restype = ctypes.c_char_p
        lib.hc_block_step_backward_workspace_bytes.restype = ctypes.c_size_t
        lib.hc_chain_state_bytes.restype = ctypes.c_size_t
        _lib = lib
        return lib


def call(name, *args):
    """Call an entry point and raise HcError on a non-zero status."""
    lib = load()
    st = getattr(lib, name)(*args)
    if st != 0:
        msg = lib.hc_status_string(st).decode()
        raise HcError(name, st, msg, lib.hc_last_cuda_error() if st == 5 else 0)
    return st


def raw(name, *args) -> int:
    """Call an entry point and return its status code."""
    return getattr(load(), name)(*args)
