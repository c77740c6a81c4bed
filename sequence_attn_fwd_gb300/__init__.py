"""Blockwise exact attention and log-sum-exp merge on GB300 (sm_103a).

Thin Python binding over the C ABI of ``libseqattn.so`` (include/seqattn.h):
it checks dtypes, shapes and layouts, marshals pointers and the current CUDA
stream, and raises on a non-zero status. Every step of the computation runs
in the library's CUDA kernels; there is no other implementation to fall back
to, and a missing library is an error.

    o, lse = attn_fwd(q, k, v, causal=True)
    o_i, lse_i = attn_partial(q, k[:, :, a:b], v[:, :, a:b], q_off=0, kv_off=a, causal=True)
    o, lse = lse_merge(o_parts, lse_parts)
    o, lse = ring_attn_fwd(q, k, v, P=8, causal=True)   # P chunks + merge on one GPU
    o, lse = attn_fwd_varlen(q, k, v, cu_seqlens, cu_seqlens, causal=True)  # packed sequences
    o, lse = attn_fwd_fp8(q8, k8, vt8, q_scale, k_scale, v_scale, causal=True)  # e4m3 inputs
    dq, dk, dv = attn_bwd(q, k, v, o, lse, dout, causal=True)   # gradients
    o_h, lse_h = ring_attn_fwd_host(q_h, k_h, v_h, P=8, causal=True)  # host tensors in and out
"""
from __future__ import annotations

import math

import torch

import ctypes

from ._lib import AttnBlock, AttnError, lib

__all__ = ["attn_fwd", "attn_partial", "attn_partial_blocks", "attn_fwd_varlen", "attn_fwd_fp8", "attn_bwd", "lse_merge",
           "ring_attn_fwd", "ring_attn_fwd_static", "ring_attn_fwd_host", "ring_host_workspace_bytes",
           "EmulatedRing",
           "query_device_error", "AttnError", "lib", "RING_SCRATCH_BYTES"]

RING_SCRATCH_BYTES = 64 << 20  # the library's fixed scratch array for ring_attn_fwd_static

ATTN_BF16, ATTN_F32 = 0, 1
ATTN_PARTIAL_SKIP_EMPTY = 1


def _stream_handle(device: torch.device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _check(status: int, what: str) -> None:
    if status != 0:
        raise AttnError(status, what)


def _require(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def _rows_contiguous(t: torch.Tensor) -> bool:
    """[B, H, S, D] with D and S packed (row r of a head at r*D) and heads at a
    uniform stride, so a slice along S of a contiguous tensor qualifies."""
    B, H, S, D = t.shape
    return (t.stride(3) == 1 and (S <= 1 or t.stride(2) == D)
            and (B <= 1 or t.stride(0) == H * t.stride(1)))


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, causal: bool = False,
             scale: float | None = None, out: torch.Tensor | None = None,
             lse: torch.Tensor | None = None):
    """softmax(scale * Q K^T) V for bf16 Q [B,Hq,S,D], K/V [B,Hkv,S,D] (contiguous).

    Returns (O bf16 [B,Hq,S,D], lse fp32 [B,Hq,S]); lse is the natural log."""
    _require(q.dim() == 4 and k.dim() == 4 and v.shape == k.shape, "expected [B,H,S,D] tensors")
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    _require(k.shape[0] == B and k.shape[2] == S and k.shape[3] == D, "K/V shape mismatch")
    for t in (q, k, v):
        _require(t.dtype == torch.bfloat16 and t.is_cuda and t.is_contiguous(),
                 "q, k, v must be contiguous bf16 CUDA tensors")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    _require(out.shape == q.shape and out.dtype == torch.bfloat16 and out.is_contiguous(), "bad out")
    _require(lse.shape == (B, Hq, S) and lse.dtype == torch.float32 and lse.is_contiguous(), "bad lse")
    st = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                      B, Hq, Hkv, S, D, int(bool(causal)), scale, _stream_handle(q.device))
    _check(st, "attn_fwd")
    return out, lse


def attn_partial(q: torch.Tensor, k_chunk: torch.Tensor, v_chunk: torch.Tensor, q_off: int = 0,
                 kv_off: int = 0, causal: bool = False, scale: float | None = None,
                 out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                 skip_empty: bool = False):
    """Attention of Q [B,Hq,Sq,D] against one K/V chunk [B,Hkv,Skv,D].

    The chunk may be a slice along S of a larger contiguous K/V (no copy).
    q_off / kv_off are the global positions of query row 0 and key 0.
    Returns (O_i fp32 [B,Hq,Sq,D] normalised within the chunk, lse_i fp32 [B,Hq,Sq]).
    Rows that see no key get lse = -inf and O = 0, or, with skip_empty, an O row
    left unwritten (lse_merge never reads it)."""
    _require(q.dim() == 4 and k_chunk.dim() == 4 and v_chunk.shape == k_chunk.shape,
             "expected [B,H,S,D] tensors")
    B, Hq, Sq, D = q.shape
    Hkv, Skv = k_chunk.shape[1], k_chunk.shape[2]
    _require(k_chunk.shape[0] == B and k_chunk.shape[3] == D, "K/V shape mismatch")
    _require(q.dtype == torch.bfloat16 and q.is_cuda and q.is_contiguous(), "q must be contiguous bf16")
    for t in (k_chunk, v_chunk):
        _require(t.dtype == torch.bfloat16 and t.is_cuda and _rows_contiguous(t),
                 "k/v chunks must be bf16 with packed rows (a contiguous tensor or an S-slice of one)")
    _require(k_chunk.stride() == v_chunk.stride(), "k and v chunks must share strides")
    head_stride = k_chunk.stride(1) if Hkv > 1 or B > 1 else Skv * D
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty((B, Hq, Sq, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    _require(out.shape == (B, Hq, Sq, D) and out.dtype == torch.float32 and out.is_contiguous(), "bad out")
    _require(lse.shape == (B, Hq, Sq) and lse.dtype == torch.float32 and lse.is_contiguous(), "bad lse")
    st = lib.attn_partial(q.data_ptr(), k_chunk.data_ptr(), v_chunk.data_ptr(), int(q_off), int(kv_off),
                          int(head_stride), out.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Sq, Skv, D,
                          int(bool(causal)), scale, ATTN_PARTIAL_SKIP_EMPTY if skip_empty else 0,
                          _stream_handle(q.device))
    _check(st, "attn_partial")
    return out, lse


def attn_partial_blocks(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, blocks, n_parts: int = 1,
                        o_rows: int | None = None, causal: bool = False, scale: float | None = None,
                        out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                        skip_empty: bool = False):
    """Several attention blocks in one persistent launch (per 64 blocks).

    q bf16 [B,Hq,q_rows,D], k/v bf16 [B,Hkv,kv_rows,D], contiguous; blocks: an
    iterable of (q_row, kv_row, o_row, q_pos, kv_pos, Sq, Skv, part) with the
    meaning of attn_block in include/seqattn.h. Returns the partials (O fp32
    [n_parts,B,Hq,o_rows,D], lse fp32 [n_parts,B,Hq,o_rows]); rows no block
    writes keep their previous contents (uninitialised unless out/lse are given)."""
    _require(q.dim() == 4 and k.dim() == 4 and v.shape == k.shape, "expected [B,H,S,D] tensors")
    B, Hq, q_rows, D = q.shape
    Hkv, kv_rows = k.shape[1], k.shape[2]
    for t in (q, k, v):
        _require(t.dtype == torch.bfloat16 and t.is_cuda and t.is_contiguous(),
                 "q, k, v must be contiguous bf16 CUDA tensors")
    blocks = list(blocks)
    o_rows = q_rows if o_rows is None else int(o_rows)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty((n_parts, B, Hq, o_rows, D), dtype=torch.float32, device=q.device)
    if lse is None:
        lse = torch.empty((n_parts, B, Hq, o_rows), dtype=torch.float32, device=q.device)
    _require(out.shape == (n_parts, B, Hq, o_rows, D) and out.dtype == torch.float32 and out.is_contiguous(),
             "bad out")
    _require(lse.shape == (n_parts, B, Hq, o_rows) and lse.dtype == torch.float32 and lse.is_contiguous(),
             "bad lse")
    arr = (AttnBlock * max(len(blocks), 1))(*[AttnBlock(*map(int, b)) for b in blocks])
    st = lib.attn_partial_blocks(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                 ctypes.addressof(arr), len(blocks), B, Hq, Hkv, q_rows, kv_rows, o_rows,
                                 int(n_parts), D, int(bool(causal)), scale,
                                 ATTN_PARTIAL_SKIP_EMPTY if skip_empty else 0, _stream_handle(q.device))
    _check(st, "attn_partial_blocks")
    return out, lse


def attn_fwd_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens_q, cu_seqlens_k,
                    causal: bool = False, scale: float | None = None, out: torch.Tensor | None = None,
                    lse: torch.Tensor | None = None):
    """Attention over packed variable-length sequences: q bf16 [Hq,total_q,D],
    k/v bf16 [Hkv,total_k,D] (sequence s in rows cu_seqlens[s]..cu_seqlens[s+1]);
    cu_seqlens_* are host sequences of ints (nseq + 1 entries, from 0). Causal
    masks are aligned at the bottom right of each sequence. Returns (O bf16
    [Hq,total_q,D], lse fp32 [Hq,total_q])."""
    _require(q.dim() == 3 and k.dim() == 3 and v.shape == k.shape, "expected [H,total,D] tensors")
    Hq, total_q, D = q.shape
    Hkv, total_k = k.shape[0], k.shape[1]
    for t in (q, k, v):
        _require(t.dtype == torch.bfloat16 and t.is_cuda and t.is_contiguous(),
                 "q, k, v must be contiguous bf16 CUDA tensors")
    cq = [int(x) for x in cu_seqlens_q]
    ck = [int(x) for x in cu_seqlens_k]
    _require(len(cq) == len(ck) and len(cq) >= 1, "cu_seqlens_q and cu_seqlens_k need nseq + 1 entries")
    _require(cq[-1] == total_q and ck[-1] == total_k, "cu_seqlens must end at the packed lengths")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    _require(out.shape == q.shape and out.dtype == torch.bfloat16 and out.is_contiguous(), "bad out")
    _require(lse.shape == (Hq, total_q) and lse.dtype == torch.float32 and lse.is_contiguous(), "bad lse")
    aq = (ctypes.c_longlong * len(cq))(*cq)
    ak = (ctypes.c_longlong * len(ck))(*ck)
    st = lib.attn_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                             ctypes.addressof(aq), ctypes.addressof(ak), len(cq) - 1, Hq, Hkv, D,
                             int(bool(causal)), scale, _stream_handle(q.device))
    _check(st, "attn_fwd_varlen")
    return out, lse


def attn_fwd_fp8(q8: torch.Tensor, k8: torch.Tensor, vt8: torch.Tensor, q_scale: float, k_scale: float,
                 v_scale: float, causal: bool = False, scale: float | None = None,
                 out: torch.Tensor | None = None, lse: torch.Tensor | None = None):
    """Attention on e4m3 inputs with per-tensor scales: q = q_scale*q8,
    k = k_scale*k8, v = v_scale*vt8^T. q8 [B,Hq,S,128], k8 [B,Hkv,S,128] and the
    transposed vt8 [B,Hkv,128,S] are contiguous torch.float8_e4m3fn CUDA
    tensors (S a multiple of 16). Returns (O bf16 [B,Hq,S,128], lse fp32)."""
    _require(q8.dim() == 4 and k8.dim() == 4 and vt8.dim() == 4, "expected 4-d tensors")
    B, Hq, S, D = q8.shape
    Hkv = k8.shape[1]
    _require(k8.shape == (B, Hkv, S, D) and vt8.shape == (B, Hkv, D, S), "K / V^T shape mismatch")
    for t in (q8, k8, vt8):
        _require(t.dtype == torch.float8_e4m3fn and t.is_cuda and t.is_contiguous(),
                 "q8, k8, vt8 must be contiguous float8_e4m3fn CUDA tensors")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty((B, Hq, S, D), dtype=torch.bfloat16, device=q8.device)
    if lse is None:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q8.device)
    _require(out.shape == (B, Hq, S, D) and out.dtype == torch.bfloat16 and out.is_contiguous(), "bad out")
    _require(lse.shape == (B, Hq, S) and lse.dtype == torch.float32 and lse.is_contiguous(), "bad lse")
    st = lib.attn_fwd_fp8(q8.data_ptr(), k8.data_ptr(), vt8.data_ptr(), out.data_ptr(), lse.data_ptr(), B, Hq,
                          Hkv, S, D, int(bool(causal)), scale, float(q_scale), float(k_scale), float(v_scale),
                          _stream_handle(q8.device))
    _check(st, "attn_fwd_fp8")
    return out, lse


def attn_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor, lse: torch.Tensor,
             dout: torch.Tensor, causal: bool = False, scale: float | None = None,
             dq: torch.Tensor | None = None, dk: torch.Tensor | None = None, dv: torch.Tensor | None = None,
             delta: torch.Tensor | None = None):
    """Gradients (dQ, dK, dV) of attn_fwd(q, k, v) for the output gradient dout,
    from the forward's o and lse (bf16 [B,Hq,S,D] q / o / dout, [B,Hkv,S,D]
    k / v with D 64 or 128, fp32 lse [B,Hq,S]). delta is an optional fp32
    [B,Hq,S] workspace."""
    _require(q.dim() == 4 and k.dim() == 4 and v.shape == k.shape, "expected [B,H,S,D] tensors")
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    _require(o.shape == q.shape and dout.shape == q.shape and lse.shape == (B, Hq, S), "shape mismatch")
    for t in (q, k, v, o, dout):
        _require(t.dtype == torch.bfloat16 and t.is_cuda and t.is_contiguous(), "bf16 contiguous CUDA tensors")
    _require(lse.dtype == torch.float32 and lse.is_contiguous(), "lse must be contiguous fp32")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    delta = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device) if delta is None else delta
    st = lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                      delta.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, S, D,
                      int(bool(causal)), scale, _stream_handle(q.device))
    _check(st, "attn_bwd")
    return dq, dk, dv


def quantize_e4m3(x: torch.Tensor, scale: float) -> torch.Tensor:
    """x / scale rounded to e4m3 (nearest even, clamped to +-448): input
    preparation for attn_fwd_fp8 (torch's conversion)."""
    return (x.float() / scale).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)


def lse_merge(o_parts: torch.Tensor, lse_parts: torch.Tensor, out_dtype=torch.bfloat16,
              out: torch.Tensor | None = None, lse: torch.Tensor | None = None):
    """Merge P partials: o_parts fp32 [P,B,H,S,D], lse_parts fp32 [P,B,H,S] -> (O, lse)."""
    _require(o_parts.dim() == 5 and lse_parts.shape == o_parts.shape[:4], "expected [P,B,H,S,D] and [P,B,H,S]")
    P, B, H, S, D = o_parts.shape
    for t in (o_parts, lse_parts):
        _require(t.dtype == torch.float32 and t.is_cuda and t.is_contiguous(), "partials must be contiguous fp32 CUDA")
    _require(out_dtype in (torch.bfloat16, torch.float32), "out_dtype must be bf16 or fp32")
    if out is None:
        out = torch.empty((B, H, S, D), dtype=out_dtype, device=o_parts.device)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=o_parts.device)
    _require(out.shape == (B, H, S, D) and out.dtype == out_dtype and out.is_contiguous(), "bad out")
    _require(lse.shape == (B, H, S) and lse.dtype == torch.float32 and lse.is_contiguous(), "bad lse")
    st = lib.lse_merge(o_parts.data_ptr(), lse_parts.data_ptr(), P, out.data_ptr(),
                       ATTN_BF16 if out_dtype == torch.bfloat16 else ATTN_F32, lse.data_ptr(),
                       B, H, S, D, _stream_handle(o_parts.device))
    _check(st, "lse_merge")
    return out, lse


def ring_attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, P: int, causal: bool = False,
                  scale: float | None = None, o_parts: torch.Tensor | None = None,
                  lse_parts: torch.Tensor | None = None, out: torch.Tensor | None = None,
                  lse: torch.Tensor | None = None, grouped: bool = False):
    """Ring-Attention's per-device arithmetic on one GPU: the keys are split into
    P equal chunks (S % P == 0); chunk j is attended by attn_partial at kv_off =
    j*S/P (a zero-copy view), then the P partials are merged by lse_merge. Rows a
    chunk cannot see are not written in o_parts (their lse is -inf).
    o_parts / lse_parts are optional preallocated fp32 [P,B,Hq,S,D] / [P,B,Hq,S].
    grouped: the P partials in one attn_partial_blocks launch instead of P
    attn_partial launches (same results)."""
    B, Hq, S, D = q.shape
    _require(P >= 1 and S % P == 0, "S must be a multiple of P")
    C = S // P
    if o_parts is None:
        o_parts = torch.empty((P, B, Hq, S, D), dtype=torch.float32, device=q.device)
    if lse_parts is None:
        lse_parts = torch.empty((P, B, Hq, S), dtype=torch.float32, device=q.device)
    if grouped:
        attn_partial_blocks(q, k, v, [(0, j * C, 0, 0, j * C, S, C, j) for j in range(P)], n_parts=P,
                            causal=causal, scale=scale, out=o_parts, lse=lse_parts, skip_empty=True)
    else:
        for j in range(P):
            attn_partial(q, k[:, :, j * C:(j + 1) * C], v[:, :, j * C:(j + 1) * C], 0, j * C, causal, scale,
                         out=o_parts[j], lse=lse_parts[j], skip_empty=True)
    return lse_merge(o_parts, lse_parts, torch.bfloat16, out=out, lse=lse)


class EmulatedRing:
    """P ring devices emulated on one GPU. The blocks each device computes at
    each hop follow ``ring_schedule.hop_blocks`` for the layout ("contiguous":
    the pages' ring, one chunk per device; "zigzag": chunks d and 2P-1-d,
    balanced under the causal mask). K/V chunks are read in place (a "hop"
    moves no bytes on one GPU); each block's fp32 partial has its own slot,
    the slots of a query chunk adjacent, so that chunk's merge reads them as
    one [n, B, Hq, C, D] stack.

    run() launches, hop by hop and device by device, the device's blocks --
    one attn_partial_blocks launch per (hop, device) when fused, else one
    attn_partial per block (device-local contiguous Q chunk) -- then per query
    chunk one lse_merge of its partials; with timing, the launches of each
    (hop, device) are bracketed by CUDA events. output() assembles the
    devices' results into [B,Hq,S,D] / [B,Hq,S] (test glue)."""

    def __init__(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, P: int, layout: str = "zigzag",
                 causal: bool = True, scale: float | None = None, fused: bool = True):
        from . import ring_schedule as rs

        B, Hq, S, D = q.shape
        nc = rs.n_chunks(P, layout)
        _require(S % nc == 0, f"S must be a multiple of {nc} for the {layout} layout with P = {P}")
        _require(q.is_contiguous() and k.is_contiguous() and v.is_contiguous(), "q, k, v must be contiguous")
        self.B, self.Hq, self.S, self.D, self.P, self.layout = B, Hq, S, D, P, layout
        self.causal, self.scale, self.fused = causal, scale, fused
        self.q, self.k, self.v = q, k, v
        self.C = C = S // nc
        self.chunks = rs.device_chunks(P, layout)
        self.blocks = rs.hop_blocks(P, layout, causal)
        qcs = [qc for dc in self.chunks for qc in dc]
        n_parts = {qc: 0 for qc in qcs}
        slot = {}
        for hop in self.blocks:
            for blocks in hop:
                for b in blocks:
                    slot[b] = n_parts[b.q_chunk]
                    n_parts[b.q_chunk] += 1
        first, total = {}, 0
        for qc in sorted(qcs):
            first[qc] = total
            total += n_parts[qc]
        self.n_parts, self.first = n_parts, first
        self.part = {b: first[b.q_chunk] + s for b, s in slot.items()}
        self.o_all = torch.empty((max(total, 1), B, Hq, C, D), dtype=torch.float32, device=q.device)
        self.lse_all = torch.empty((max(total, 1), B, Hq, C), dtype=torch.float32, device=q.device)
        self.q_chunk = {} if fused else {qc: q[:, :, qc * C:(qc + 1) * C].contiguous() for qc in qcs}
        self.o = {qc: torch.empty((B, Hq, C, D), dtype=torch.bfloat16, device=q.device) for qc in qcs}
        self.lse = {qc: torch.empty((B, Hq, C), dtype=torch.float32, device=q.device) for qc in qcs}

    def _launch_device_hop(self, blocks):
        C = self.C
        if self.fused:
            if blocks:
                attn_partial_blocks(self.q, self.k, self.v,
                                    [(b.q_chunk * C, b.kv_chunk * C, 0, b.q_chunk * C, b.kv_chunk * C, C, C,
                                      self.part[b]) for b in blocks],
                                    n_parts=self.o_all.shape[0], o_rows=C, causal=self.causal,
                                    scale=self.scale, out=self.o_all, lse=self.lse_all)
            return
        for b in blocks:
            kc, s = b.kv_chunk, self.part[b]
            attn_partial(self.q_chunk[b.q_chunk], self.k[:, :, kc * C:(kc + 1) * C],
                         self.v[:, :, kc * C:(kc + 1) * C], b.q_chunk * C, kc * C, self.causal, self.scale,
                         out=self.o_all[s], lse=self.lse_all[s])

    def run(self, timing: bool = False, hold_cycles: int = 0):
        """One ring pass. With timing, returns ms[t][d] (the launches of device
        d at hop t) and the merge time of each device; else None. hold_cycles
        > 0 first queues a GPU-side wait of that many clocks, so that every
        launch of the pass is enqueued before the GPU reaches it and the events
        time the GPU work, not the host's launch rate."""
        if hold_cycles > 0:
            torch.cuda._sleep(int(hold_cycles))
        ev = []
        for hop in self.blocks:
            row = []
            for blocks in hop:
                if timing:
                    e0 = torch.cuda.Event(enable_timing=True)
                    e0.record()
                self._launch_device_hop(blocks)
                if timing:
                    e1 = torch.cuda.Event(enable_timing=True)
                    e1.record()
                    row.append((e0, e1))
            ev.append(row)
        merge_ev = []
        for dc in self.chunks:
            if timing:
                e0 = torch.cuda.Event(enable_timing=True)
                e0.record()
            for qc in dc:
                n, f = self.n_parts[qc], self.first[qc]
                if n == 0:  # no visible key (only without keys at all): O = 0, lse = -inf
                    self.o[qc].zero_()
                    self.lse[qc].fill_(-math.inf)
                    continue
                lse_merge(self.o_all[f:f + n], self.lse_all[f:f + n], torch.bfloat16, out=self.o[qc],
                          lse=self.lse[qc])
            if timing:
                e1 = torch.cuda.Event(enable_timing=True)
                e1.record()
                merge_ev.append((e0, e1))
        if not timing:
            return None
        torch.cuda.synchronize()
        hop_ms = [[a.elapsed_time(b) for a, b in row] for row in ev]
        merge_ms = [a.elapsed_time(b) for a, b in merge_ev]
        return hop_ms, merge_ms

    def output(self):
        o = torch.empty((self.B, self.Hq, self.S, self.D), dtype=torch.bfloat16, device=self.k.device)
        lse = torch.empty((self.B, self.Hq, self.S), dtype=torch.float32, device=self.k.device)
        for qc in self.o:
            o[:, :, qc * self.C:(qc + 1) * self.C] = self.o[qc]
            lse[:, :, qc * self.C:(qc + 1) * self.C] = self.lse[qc]
        return o, lse


def ring_attn_fwd_static(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, P: int, causal: bool = False,
                         scale: float | None = None, out: torch.Tensor | None = None,
                         lse: torch.Tensor | None = None):
    """ring_attn_fwd without caller-side scratch: the fp32 partials live in a
    fixed 64 MiB device array inside the library (attn_ring_fwd_static), so
    the C call itself allocates nothing. Meant for callers that cannot allocate
    device memory (a host application whose allocator owns the device memory,
    or loops that cannot afford cudaMalloc/cudaFree). Problems whose partials
    exceed the array are rejected. Calls that overlap on the GPU share the
    array and race; the first call on a device sets up the array's address.
    Here ``out``/``lse`` are allocated through torch only when not given.

    Shapes are checked before anything else (so a mismatch is refused before
    any launch), then dtypes, layouts and devices: q bf16 [B,Hq,S,D], k/v bf16
    [B,Hkv,S,D], out bf16 [B,Hq,S,D] and lse fp32 [B,Hq,S], all contiguous and
    on q's device."""
    _require(q.dim() == 4 and k.dim() == 4 and v.shape == k.shape, "expected [B,H,S,D] tensors")
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    _require(k.shape[0] == B and k.shape[2] == S and k.shape[3] == D, "K/V shape mismatch")
    _require(Hkv > 0 and Hq % Hkv == 0, "Hq must be a multiple of Hkv")
    _require(out is None or tuple(out.shape) == (B, Hq, S, D), "bad out: expected [B,Hq,S,D]")
    _require(lse is None or tuple(lse.shape) == (B, Hq, S), "bad lse: expected [B,Hq,S]")
    for t in (q, k, v):
        _require(t.dtype == torch.bfloat16 and t.is_cuda and t.is_contiguous(),
                 "q, k, v must be contiguous bf16 CUDA tensors")
        _require(t.device == q.device, "q, k, v must be on one device")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    _require(out.dtype == torch.bfloat16 and out.is_contiguous() and out.device == q.device,
             "bad out: must be a contiguous bf16 tensor on q's device")
    _require(lse.dtype == torch.float32 and lse.is_contiguous() and lse.device == q.device,
             "bad lse: must be a contiguous fp32 tensor on q's device")
    st = lib.attn_ring_fwd_static(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                  B, Hq, Hkv, S, D, int(P), int(bool(causal)), scale, _stream_handle(q.device))
    _check(st, "attn_ring_fwd_static")
    return out, lse


def ring_host_workspace_bytes(B: int, Hq: int, Hkv: int, S: int, D: int, P: int) -> int:
    """Device workspace bytes ring_attn_fwd_host needs (attn_ring_fwd_host_workspace_bytes)."""
    n = lib.attn_ring_fwd_host_workspace_bytes(B, Hq, Hkv, S, D, P)
    _require(n > 0, "invalid sizes")
    return int(n)


def ring_attn_fwd_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, P: int, causal: bool = False,
                       scale: float | None = None, out: torch.Tensor | None = None,
                       lse: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                       device: torch.device | None = None, synchronize: bool = True):
    """The ring-emulated forward from host tensors to host tensors
    (attn_ring_fwd_host): Q and each K/V chunk are uploaded on the library's
    copy stream, each chunk's partial starts on the current stream as soon as
    its chunk arrives, then the merge and the downloads of O and lse.
    q, k, v: CPU bf16 [B, H, S, D] (pinned for the copies to overlap);
    out, lse: CPU outputs (pinned ones are allocated when not given);
    workspace: a uint8 CUDA tensor of at least ring_host_workspace_bytes(...)
    bytes (allocated when not given). With synchronize=False the call returns
    once the work is queued on the current stream; the outputs are complete
    when that stream reaches it."""
    _require(q.dim() == 4 and k.dim() == 4 and v.shape == k.shape, "expected [B,H,S,D] tensors")
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    for t in (q, k, v):
        _require(t.dtype == torch.bfloat16 and t.device.type == "cpu" and t.is_contiguous(),
                 "q, k, v must be contiguous bf16 CPU tensors")
    device = device or torch.device("cuda", torch.cuda.current_device())
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    if lse is None:
        lse = torch.empty((B, Hq, S), dtype=torch.float32).pin_memory()
    _require(out.device.type == "cpu" and out.dtype == torch.bfloat16 and out.shape == q.shape
             and out.is_contiguous(), "out must be a contiguous bf16 CPU tensor shaped like q")
    _require(lse.device.type == "cpu" and lse.dtype == torch.float32 and lse.shape == (B, Hq, S)
             and lse.is_contiguous(), "lse must be a contiguous fp32 CPU tensor [B, Hq, S]")
    if B == 0 or S == 0:  # nothing to compute (the C call would return at once)
        _require(P >= 1 and (S == 0 or S % P == 0), "S must be a multiple of P")
        return out, lse
    need = ring_host_workspace_bytes(B, Hq, Hkv, S, D, P)
    if workspace is None:
        # the library's copy stream writes the workspace, which torch's allocator
        # does not track: a workspace allocated here must outlive the work
        _require(synchronize, "pass a workspace when synchronize=False")
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    _require(workspace.is_cuda and workspace.numel() * workspace.element_size() >= need,
             "workspace must be a CUDA tensor of at least ring_host_workspace_bytes(...) bytes")
    st = lib.attn_ring_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                                B, Hq, Hkv, S, D, int(P), int(bool(causal)), scale, _stream_handle(device))
    _check(st, "attn_ring_fwd_host")
    if synchronize:
        torch.cuda.current_stream(device).synchronize()
    return out, lse


def query_device_error(device: torch.device | None = None) -> None:
    """Synchronise the current stream and raise AttnError if a kernel timed out."""
    device = device or torch.device("cuda", torch.cuda.current_device())
    _check(lib.attn_query_device_error(_stream_handle(device)), "device wait")
