"""The C-ABI library builds, loads, exports what include/seqattn.h declares and
rejects bad arguments on the host, before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

from __graft_entry__ import _build_module

build_mod = _build_module()

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "seqattn.h")


@pytest.fixture(scope="module")
def lib():
    path = build_mod.build()
    from sequence_attn_fwd_gb300._lib import load

    return load(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    assert declared_functions() == sorted(["attn_fwd", "attn_partial", "lse_merge", "attn_query_device_error",
                                           "attn_status_string", "attn_last_cuda_error",
                                           "attn_ring_fwd_static", "attn_debug_expire_wait",
                                           "attn_debug_exp2", "attn_partial_blocks", "attn_fwd_varlen",
                                           "attn_fwd_fp8", "attn_bwd",
                                           "attn_ring_fwd_host_workspace_bytes", "attn_ring_fwd_host"])


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    from sequence_attn_fwd_gb300._lib import EXPORTS

    assert sorted(EXPORTS) == declared_functions()


def test_library_is_built_for_sm103a():
    log = open(os.path.join(os.path.dirname(build_mod.LIB), "ptxas.log")).read()
    assert "for 'sm_103a'" in log and "attn_fwd_kernel" in log and "lse_merge_kernel" in log
    assert "tcgen05" in open(os.path.join(build_mod.CSRC, "ptx.cuh")).read()


def test_expire_wait_argument_checks(lib):
    assert lib.attn_debug_expire_wait(0, None) == 1
    assert lib.attn_debug_expire_wait(2_000_000, None) == 1


def test_exp2_hook_argument_checks(lib):
    assert lib.attn_debug_exp2(FAKE, FAKE, -1, 1, None) == 1
    assert lib.attn_debug_exp2(FAKE, FAKE, 4, 2, None) == 1
    assert lib.attn_debug_exp2(0, FAKE, 4, 1, None) == 1
    assert lib.attn_debug_exp2(0, 0, 0, 0, None) == 0


def test_status_strings(lib):
    assert lib.attn_status_string(0) == b"ok"
    assert lib.attn_status_string(4) == b"device-side wait timed out"
    assert lib.attn_status_string(99) == b"unknown status"
    assert lib.attn_last_cuda_error() == 0


FAKE = 1 << 20  # a 16-byte-aligned non-null address; never dereferenced on these paths


def fwd(lib, q=FAKE, B=1, Hq=2, Hkv=2, S=16, D=64, causal=0, scale=0.125):
    return lib.attn_fwd(q, FAKE, FAKE, FAKE, FAKE, B, Hq, Hkv, S, D, causal, ctypes.c_float(scale), None)


def test_attn_fwd_argument_checks(lib):
    assert fwd(lib, Hq=3, Hkv=2) == 1  # Hq % Hkv != 0
    assert fwd(lib, D=96) == 2  # unsupported head dim
    assert fwd(lib, D=256) == 2
    assert fwd(lib, q=0) == 1  # null pointer
    assert fwd(lib, q=FAKE + 8) == 1  # misaligned
    assert fwd(lib, scale=0.0) == 1 and fwd(lib, scale=float("nan")) == 1 and fwd(lib, scale=-1.0) == 1
    assert fwd(lib, causal=2) == 1
    assert fwd(lib, B=-1) == 1 and fwd(lib, S=-5) == 1 and fwd(lib, Hkv=0) == 1
    assert fwd(lib, B=0) == 0 and fwd(lib, S=0) == 0  # empty problems are no-ops
    assert fwd(lib, q=0, S=0) == 0


def test_attn_partial_argument_checks(lib):
    def part(kv_head_stride=0, Sq=16, Skv=16, D=64, o=FAKE, flags=0):
        return lib.attn_partial(FAKE, FAKE, FAKE, 0, 0, kv_head_stride, o, FAKE, 1, 2, 1, Sq, Skv, D, 1,
                                ctypes.c_float(0.125), flags, None)

    assert part(kv_head_stride=16 * 64 - 8) == 1  # stride shorter than a head
    assert part(kv_head_stride=16 * 64 + 4) == 1  # not a multiple of 8 elements
    assert part(o=FAKE + 4) == 1
    assert part(D=32) == 2
    assert part(Sq=0) == 0
    assert part(flags=2) == 1 and part(flags=-1) == 1  # unknown flag bits
    assert part(Sq=0, flags=1) == 0


def test_lse_merge_argument_checks(lib):
    def merge(P=2, o_dtype=0, D=128, S=8, parts=FAKE):
        return lib.lse_merge(parts, FAKE, P, FAKE, o_dtype, FAKE, 1, 2, S, D, None)

    assert merge(P=0) == 1
    assert merge(o_dtype=7) == 1
    assert merge(D=80) == 2
    assert merge(parts=0) == 1
    assert merge(parts=FAKE + 4) == 1
    assert merge(S=0) == 0


def test_attn_block_layout_matches_the_header():
    from sequence_attn_fwd_gb300._lib import AttnBlock

    assert ctypes.sizeof(AttnBlock) == 56  # five int64 and three int32, 8-byte aligned
    text = open(HEADER).read()
    assert "long long q_row, kv_row, o_row;" in text and "int part;" in text


def test_attn_partial_blocks_argument_checks(lib):
    from sequence_attn_fwd_gb300._lib import AttnBlock

    def run(blocks, q_rows=512, kv_rows=512, o_rows=512, n_parts=2, D=128, flags=0):
        arr = (AttnBlock * max(len(blocks), 1))(*[AttnBlock(*b) for b in blocks])
        return lib.attn_partial_blocks(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.addressof(arr), len(blocks), 1, 2, 1,
                                       q_rows, kv_rows, o_rows, n_parts, D, 1, ctypes.c_float(0.1), flags, None)

    ok = (0, 0, 0, 0, 0, 256, 256, 0)
    assert run([]) == 0
    assert run([ok, (0, 0, 200, 0, 0, 100, 100, 0)]) == 1  # output rows 200.. overlap 0..256 in part 0
    assert run([(0, 0, 0, 0, 0, 256, 256, 2)]) == 1  # part out of range
    assert run([(300, 0, 0, 0, 0, 256, 256, 0)]) == 1  # queries past q_rows
    assert run([(0, 300, 0, 0, 0, 256, 256, 0)]) == 1  # keys past kv_rows
    assert run([(0, 0, 300, 0, 0, 256, 256, 0)]) == 1  # outputs past o_rows
    assert run([(0, 0, 0, 0, 0, -1, 256, 0)]) == 1
    assert run([ok], D=96) == 2
    assert run([ok], flags=4) == 1
    assert lib.attn_partial_blocks(FAKE, FAKE, FAKE, FAKE, FAKE, None, 3, 1, 2, 1, 8, 8, 8, 1, 128, 1,
                                   ctypes.c_float(0.1), 0, None) == 1  # null block array


def test_attn_fwd_varlen_argument_checks(lib):
    def run(cq, ck, Hq=2, Hkv=1, D=128):
        aq = (ctypes.c_longlong * len(cq))(*cq)
        ak = (ctypes.c_longlong * len(ck))(*ck)
        return lib.attn_fwd_varlen(FAKE, FAKE, FAKE, FAKE, FAKE, ctypes.addressof(aq), ctypes.addressof(ak),
                                   len(cq) - 1, Hq, Hkv, D, 1, ctypes.c_float(0.1), None)

    assert run([0], [0]) == 0  # no sequence
    assert run([0, 0, 0], [0, 5, 9]) == 0  # no query row
    assert run([1, 5], [0, 5]) == 1  # must start at 0
    assert run([0, 5, 3], [0, 5, 9]) == 1  # decreasing
    assert run([0, 5], [0, 5], Hq=3, Hkv=2) == 1
    assert run([0, 5], [0, 5], D=32) == 2


def test_attn_fwd_fp8_argument_checks(lib):
    def run(S=256, D=128, Hq=2, Hkv=1, qs=1.0, vs=1.0, causal=1):
        return lib.attn_fwd_fp8(FAKE, FAKE, FAKE, FAKE, FAKE, 1, Hq, Hkv, S, D, causal, ctypes.c_float(0.1),
                                ctypes.c_float(qs), ctypes.c_float(1.0), ctypes.c_float(vs), None)

    assert run(D=64) == 2
    assert run(S=100) == 2  # V^T rows must be 16-byte multiples
    assert run(qs=0.0) == 1 and run(vs=float("inf")) == 1
    assert run(Hq=3, Hkv=2) == 1 and run(causal=3) == 1
    assert run(S=0) == 0


def test_attn_bwd_argument_checks(lib):
    def run(S=256, D=128, Hq=2, Hkv=1, B=1, q=FAKE, delta=FAKE, scale=0.1):
        return lib.attn_bwd(q, FAKE, FAKE, FAKE, FAKE, FAKE, delta, FAKE, FAKE, FAKE, B, Hq, Hkv, S, D, 1,
                            ctypes.c_float(scale), None)

    assert run(D=96) == 2 and run(D=32) == 2
    assert run(D=64, q=FAKE + 8) == 1  # D = 64 is accepted: it reaches the alignment checks
    assert run(B=2, Hq=32768, Hkv=1) == 2  # more than 65535 (batch, query head) pairs
    assert run(S=(1 << 30) + 128) == 2
    assert run(Hq=3, Hkv=2) == 1 and run(scale=-1.0) == 1
    assert run(q=FAKE + 8) == 1 and run(delta=FAKE + 2) == 1 and run(q=0) == 1
    assert run(S=0) == 0


def test_ring_host_workspace_layout(lib):
    """Device copies of Q, K, V, the fp32 partials (P > 1 only), O and lse, each
    rounded up to 256 bytes."""
    up = lambda n: (n + 255) // 256 * 256
    B, Hq, Hkv, S, D, P = 2, 8, 2, 1000, 128, 8
    rows, kv = B * Hq * S, B * Hkv * S
    want = up(rows * D * 2) + 2 * up(kv * D * 2) + up(P * rows * D * 4) + up(P * rows * 4) + up(rows * D * 2) + up(rows * 4)
    assert lib.attn_ring_fwd_host_workspace_bytes(B, Hq, Hkv, S, D, P) == want
    assert lib.attn_ring_fwd_host_workspace_bytes(B, Hq, Hkv, S, D, 1) == (
        up(rows * D * 2) + 2 * up(kv * D * 2) + up(rows * D * 2) + up(rows * 4))
    for bad in ((B, Hq, Hkv, S, 96, P), (B, Hq, Hkv, S, D, 0), (B, Hq, Hkv, S, D, 65), (B, 0, Hkv, S, D, P)):
        assert lib.attn_ring_fwd_host_workspace_bytes(*bad) == 0


def test_ring_host_argument_checks(lib):
    def run(S=512, P=4, D=128, ws=FAKE, ws_bytes=1 << 40, q=FAKE, scale=0.1, Hq=4, Hkv=2):
        return lib.attn_ring_fwd_host(q, FAKE, FAKE, FAKE, FAKE, ws, ws_bytes, 1, Hq, Hkv, S, D, P, 1,
                                      ctypes.c_float(scale), None)

    assert run(P=0) == 1 and run(P=65) == 1 and run(S=510) == 1  # S % P != 0
    assert run(D=96) == 2
    assert run(Hq=3) == 1 and run(scale=0.0) == 1 and run(q=0) == 1
    assert run(ws=FAKE + 16) == 1  # workspace not 256-byte aligned
    assert run(ws_bytes=1024) == 1  # workspace too small
    assert run(S=0) == 0


def test_ring_static_argument_checks(lib):
    """attn_ring_fwd_static refuses bad sizes and problems beyond its array
    before any CUDA call."""
    def call(B=1, Hq=4, Hkv=4, S=2048, D=128, P=16):
        return lib.attn_ring_fwd_static(FAKE, FAKE, FAKE, FAKE, FAKE, B, Hq, Hkv, S, D, P, 1,
                                        ctypes.c_float(0.125), None)

    assert call() == 2            # 16 x 4 x 2048 x 129 x 4 bytes > 64 MiB
    assert call(P=0) == 1
    assert call(S=1000, P=16) == 1  # S not a multiple of P
    assert call(D=96, S=256, P=2) == 2
    assert call(B=0, S=256, P=2) == 0  # nothing to compute


def test_ring_static_wrapper_refuses_bad_shapes_before_launch():
    """The Python wrapper checks K/V and given outputs' shapes before anything
    else, so a mismatch never reaches the library (CPU tensors here: the shape
    checks come ahead of the device checks)."""
    import torch

    import sequence_attn_fwd_gb300 as sa

    q = torch.zeros((1, 4, 256, 64), dtype=torch.bfloat16)
    kv = torch.zeros((1, 2, 256, 64), dtype=torch.bfloat16)
    short = torch.zeros((1, 2, 128, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="K/V shape"):
        sa.ring_attn_fwd_static(q, short, short, P=2)
    with pytest.raises(ValueError, match="K/V shape"):
        sa.ring_attn_fwd_static(q, kv[..., :32], kv[..., :32], P=2)
    with pytest.raises(ValueError, match="bad out"):
        sa.ring_attn_fwd_static(q, kv, kv, P=2, out=torch.zeros((1, 4, 128, 64), dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="bad lse"):
        sa.ring_attn_fwd_static(q, kv, kv, P=2, lse=torch.zeros((1, 4, 255), dtype=torch.float32))
    with pytest.raises(ValueError, match="CUDA"):
        sa.ring_attn_fwd_static(q, kv, kv, P=2)  # right shapes, but not on a GPU
