"""The allocation-free ring entry point against the regular one and the oracle.

attn_ring_fwd_static exists for callers that cannot allocate device memory
themselves (a host application whose allocator already owns the device's
memory, or a loop that cannot pay for cudaMalloc/cudaFree and the device
synchronisation they may cause). It keeps the ring's fp32 partials in a
fixed array inside the library. This file is collected last so that a run
stopping at the first failure has run every other test already; it must also
pass on its own in a fresh process (the first call there sets up the array).
"""
import ctypes
import math

import pytest
import torch

import oracle
import workloads
from tests.parity import LSE_TOL, O_TOL, check_lse, check_o

pytestmark = pytest.mark.gpu


def call_static(lib, q, k, v, o, lse, P, causal):
    B, Hq, S, D = q.shape
    return lib.attn_ring_fwd_static(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                    B, Hq, k.shape[1], S, D, P, int(causal), ctypes.c_float(1 / math.sqrt(D)),
                                    torch.cuda.current_stream().cuda_stream)


def test_static_scratch_ring_matches_caller_scratch_ring_and_oracle(cuda_dev):
    """Calls in a row on problems that share the array: the causal call comes
    right after a non-causal one of the same shape, so the partial rows a
    causal chunk cannot see still hold the previous call's finite values (the
    merge must never read them); a third call changes head dim and part count.
    Each result equals the caller-scratch ring within the tolerance and matches
    the oracle on every row. The last call goes through the Python wrapper."""
    import sequence_attn_fwd_gb300 as sa

    lib = sa.lib
    cases = [workloads.Workload("noalloc_a_full", 2, 4, 2, 1024, 128, False, 8, 2024),
             workloads.Workload("noalloc_a_causal", 2, 4, 2, 1024, 128, True, 8, 2024),
             workloads.Workload("noalloc_b", 1, 3, 3, 768, 64, True, 3, 2025)]
    for i, w in enumerate(cases):
        q_h, k_h, v_h = workloads.make_qkv(w)
        q, k, v = (t.cuda() for t in (q_h, k_h, v_h))
        if i < len(cases) - 1:
            o = torch.empty_like(q)
            lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
            assert call_static(lib, q, k, v, o, lse, w.P, w.causal) == 0
        else:
            o, lse = sa.ring_attn_fwd_static(q, k, v, P=w.P, causal=w.causal)
        o_ring, lse_ring = sa.ring_attn_fwd(q, k, v, P=w.P, causal=w.causal)
        torch.cuda.synchronize()
        assert (o.float() - o_ring.float()).abs().max().item() <= O_TOL
        assert torch.equal(torch.isneginf(lse), torch.isneginf(lse_ring))
        assert (lse - lse_ring).abs().max().item() <= LSE_TOL
        o_ref, lse_ref = oracle.attention(q_h, k_h, v_h, w.causal)
        check_o(o, o_ref)
        check_lse(lse, lse_ref)
    sa.query_device_error()


def test_static_scratch_rejects_problems_beyond_the_array(cuda_dev):
    import sequence_attn_fwd_gb300 as sa

    # partials of 16 x 4 x 2048 x 128 fp32 = 64 MiB, plus their lse: over the limit
    w = workloads.Workload("noalloc_big", 1, 4, 4, 2048, 128, True, 16, 7)
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    assert call_static(sa.lib, q, k, v, o, lse, w.P, w.causal) == 2  # ATTN_ERR_UNSUPPORTED
    assert sa.RING_SCRATCH_BYTES == 64 << 20
