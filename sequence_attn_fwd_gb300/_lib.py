"""Loads libseqattn.so (built in-tree by sequence_attn_fwd_gb300.build) via ctypes.

The library must exist: there is no fallback implementation. Import fails
with a message naming the build command when it is missing.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libseqattn.so")

# Every function the public header include/seqattn.h declares.
EXPORTS = ["attn_fwd", "attn_partial", "lse_merge", "attn_query_device_error",
           "attn_status_string", "attn_last_cuda_error", "attn_ring_fwd_static",
           "attn_debug_expire_wait", "attn_debug_exp2", "attn_partial_blocks", "attn_fwd_varlen", "attn_fwd_fp8", "attn_bwd",
           "attn_ring_fwd_host_workspace_bytes", "attn_ring_fwd_host"]

STATUS = {0: "ATTN_OK", 1: "ATTN_ERR_INVALID_ARG", 2: "ATTN_ERR_UNSUPPORTED",
          3: "ATTN_ERR_CUDA", 4: "ATTN_ERR_TIMEOUT"}


class AttnBlock(ctypes.Structure):
    """attn_block of include/seqattn.h."""
    _fields_ = [("q_row", ctypes.c_longlong), ("kv_row", ctypes.c_longlong), ("o_row", ctypes.c_longlong),
                ("q_pos", ctypes.c_longlong), ("kv_pos", ctypes.c_longlong), ("Sq", ctypes.c_int),
                ("Skv", ctypes.c_int), ("part", ctypes.c_int)]


class AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        name = STATUS.get(status, str(status))
        detail = lib.attn_status_string(status).decode() if lib is not None else ""
        extra = f" (cudaError {lib.attn_last_cuda_error()})" if status == 3 and lib is not None else ""
        super().__init__(f"{what}: {name}: {detail}{extra}")


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing; build it with `python sequence_attn_fwd_gb300/build.py`")
    L = ctypes.CDLL(path)
    P, I, LL, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_float
    L.attn_fwd.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, P]
    L.attn_partial.argtypes = [P, P, P, LL, LL, LL, P, P, I, I, I, I, I, I, I, F, I, P]
    L.lse_merge.argtypes = [P, P, I, P, I, P, I, I, I, I, P]
    L.attn_query_device_error.argtypes = [P]
    L.attn_status_string.argtypes = [I]
    L.attn_status_string.restype = ctypes.c_char_p
    L.attn_last_cuda_error.argtypes = []
    L.attn_ring_fwd_static.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, F, P]
    L.attn_ring_fwd_static.restype = ctypes.c_int
    L.attn_ring_fwd_host_workspace_bytes.argtypes = [I, I, I, I, I, I]
    L.attn_ring_fwd_host_workspace_bytes.restype = ctypes.c_size_t
    L.attn_ring_fwd_host.argtypes = [P, P, P, P, P, P, ctypes.c_size_t, I, I, I, I, I, I, I, F, P]
    L.attn_ring_fwd_host.restype = ctypes.c_int
    L.attn_debug_expire_wait.argtypes = [ctypes.c_uint, P]
    L.attn_debug_expire_wait.restype = ctypes.c_int
    L.attn_debug_exp2.argtypes = [P, P, ctypes.c_longlong, ctypes.c_int, P]
    L.attn_debug_exp2.restype = ctypes.c_int
    L.attn_partial_blocks.argtypes = [P, P, P, P, P, P, I, I, I, I, LL, LL, LL, I, I, I, F, I, P]
    L.attn_partial_blocks.restype = ctypes.c_int
    L.attn_fwd_varlen.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, F, P]
    L.attn_fwd_varlen.restype = ctypes.c_int
    L.attn_fwd_fp8.argtypes = [P, P, P, P, P, I, I, I, I, I, I, F, F, F, F, P]
    L.attn_fwd_fp8.restype = ctypes.c_int
    L.attn_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, I, I, I, I, I, I, F, P]
    L.attn_bwd.restype = ctypes.c_int
    for name in ("attn_fwd", "attn_partial", "lse_merge", "attn_query_device_error",
                 "attn_last_cuda_error"):
        getattr(L, name).restype = ctypes.c_int
    return L


lib = None
lib = load()
