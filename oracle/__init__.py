"""ORACLE -- test infrastructure, not product code.

Python access to the fp64 CPU oracle in ``attn_oracle.c``. Only the tests,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg import this
package; the CUDA path (``sequence_attn_fwd_gb300``) never does.

Functions
---------
attention(q, k, v, causal, scale=None, q_off=0, kv_off=0, rows=None, threads=None)
    Exact attention in fp64 from bf16 inputs ([B,Hq,Sq,D], [B,Hkv,Skv,D]).
    See attn_oracle.c for the definition and the passages it follows.
lse_merge(o_parts, lse_parts)
    fp64 merge of per-chunk partials ([P,...,D], [P,...]).
attention_backward(q, k, v, dout, causal, scale=None, threads=None)
    fp64 gradients (dQ, dK, dV) of attention for the output gradient dO
    (bf16 [B,Hq,S,D]); see attn_oracle.c.
attention_backward_dq_rows(q, k, v, dout, causal, rows, scale=None, threads=None)
    fp64 dQ of selected query rows ([B*Hq, n] indices) only, row by row.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (plain -O2, IEEE semantics, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
                               "-fno-fast-math", "-ffp-contract=off",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        lib.oracle_attention.argtypes = [P, P, P] + [ctypes.c_int] * 6 + [ctypes.c_longlong] * 4 + [
            ctypes.c_int, ctypes.c_double, P, ctypes.c_int, P, P, ctypes.c_int]
        lib.oracle_attention.restype = ctypes.c_int
        lib.oracle_lse_merge.argtypes = [P, P, ctypes.c_int, ctypes.c_longlong, ctypes.c_int, P, P]
        lib.oracle_lse_merge.restype = None
        lib.oracle_attention_backward.argtypes = [P, P, P, P] + [ctypes.c_int] * 6 + [
            ctypes.c_double, P, P, P, ctypes.c_int]
        lib.oracle_attention_backward.restype = ctypes.c_int
        lib.oracle_attention_backward_dq_rows.argtypes = [P, P, P, P] + [ctypes.c_int] * 6 + [
            ctypes.c_double, P, ctypes.c_int, P, ctypes.c_int]
        lib.oracle_attention_backward_dq_rows.restype = ctypes.c_int
        _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _bits(t: torch.Tensor) -> np.ndarray:
    assert t.dtype == torch.bfloat16 and t.device.type == "cpu"
    return np.ascontiguousarray(t.contiguous().view(torch.int16).numpy().view(np.uint16))


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool,
              scale: float | None = None, q_off: int = 0, kv_off: int = 0,
              rows: np.ndarray | None = None, threads: int | None = None):
    """fp64 attention. Returns (O [B,Hq,R,D] float64, lse [B,Hq,R] float64) as numpy,
    R = Sq or rows.shape[1] (rows: [B*Hq, R] int64 query rows per head)."""
    B, Hq, Sq, D = q.shape
    Bk, Hkv, Skv, Dk = k.shape
    assert Bk == B and Dk == D and v.shape == k.shape and Hq % Hkv == 0
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    qb, kb, vb = _bits(q), _bits(k), _bits(v)
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        assert rows.shape[0] == B * Hq
        R = rows.shape[1]
    else:
        R = Sq
    o = np.empty((B, Hq, R, D), dtype=np.float64)
    lse = np.empty((B, Hq, R), dtype=np.float64)
    rc = _load().oracle_attention(
        qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, B, Hq, Hkv, Sq, Skv, D,
        int(q_off), int(kv_off), Sq * D, Skv * D, int(bool(causal)), scale,
        rows.ctypes.data if rows is not None else None, R if rows is not None else 0,
        o.ctypes.data, lse.ctypes.data, int(threads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_attention rejected its arguments")
    return o, lse


def lse_merge(o_parts, lse_parts):
    """fp64 merge. o_parts [P,...,D], lse_parts [P,...] (any float dtype, numpy or torch)."""
    o_parts = np.ascontiguousarray(np.asarray(o_parts, dtype=np.float64))
    lse_parts = np.ascontiguousarray(np.asarray(lse_parts, dtype=np.float64))
    P = o_parts.shape[0]
    D = o_parts.shape[-1]
    assert lse_parts.shape == o_parts.shape[:-1]
    nrows = int(np.prod(lse_parts.shape[1:], dtype=np.int64))
    o = np.empty(o_parts.shape[1:], dtype=np.float64)
    lse = np.empty(lse_parts.shape[1:], dtype=np.float64)
    _load().oracle_lse_merge(o_parts.ctypes.data, lse_parts.ctypes.data, P, nrows, D,
                             o.ctypes.data, lse.ctypes.data)
    return o, lse


def attention_backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, dout: torch.Tensor, causal: bool,
                       scale: float | None = None, threads: int | None = None):
    """fp64 (dQ [B,Hq,S,D], dK [B,Hkv,S,D], dV [B,Hkv,S,D]) as numpy from bf16
    q, dout [B,Hq,S,D] and k, v [B,Hkv,S,D] (the chain rule through the
    definition; attn_oracle.c)."""
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    assert k.shape == (B, Hkv, S, D) and v.shape == k.shape and dout.shape == q.shape and Hq % Hkv == 0
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    qb, kb, vb, db = _bits(q), _bits(k), _bits(v), _bits(dout)
    dq = np.empty((B, Hq, S, D), dtype=np.float64)
    dk = np.empty((B, Hkv, S, D), dtype=np.float64)
    dv = np.empty((B, Hkv, S, D), dtype=np.float64)
    rc = _load().oracle_attention_backward(qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, db.ctypes.data,
                                           B, Hq, Hkv, S, D, int(bool(causal)), scale, dq.ctypes.data,
                                           dk.ctypes.data, dv.ctypes.data, int(threads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_attention_backward rejected its arguments")
    return dq, dk, dv


def attention_backward_dq_rows(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, dout: torch.Tensor,
                               causal: bool, rows: np.ndarray, scale: float | None = None,
                               threads: int | None = None) -> np.ndarray:
    """fp64 dQ [B*Hq, n, D] of the query rows rows[b*Hq + h] (int64 [B*Hq, n])
    of each (batch, query head): the chain rule of attention_backward for one
    row at a time (attn_oracle.c)."""
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    assert k.shape == (B, Hkv, S, D) and v.shape == k.shape and dout.shape == q.shape and Hq % Hkv == 0
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    assert rows.ndim == 2 and rows.shape[0] == B * Hq
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    qb, kb, vb, db = _bits(q), _bits(k), _bits(v), _bits(dout)
    out = np.empty((B * Hq, rows.shape[1], D), dtype=np.float64)
    rc = _load().oracle_attention_backward_dq_rows(qb.ctypes.data, kb.ctypes.data, vb.ctypes.data, db.ctypes.data,
                                                   B, Hq, Hkv, S, D, int(bool(causal)), scale, rows.ctypes.data,
                                                   rows.shape[1], out.ctypes.data, int(threads or default_threads()))
    if rc != 0:
        raise ValueError("oracle_attention_backward_dq_rows rejected its arguments")
    return out
