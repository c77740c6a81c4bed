"""The backward parity bound (tests/parity.py) against an emulation of the
kernels' arithmetic on the CPU: P formed in fp32 from the fp32 scores and lse
and rounded to bf16, delta formed in fp32 from a bf16 O, dS rounded to bf16,
fp32 products, bf16 results. The emulated gradients must lie within the bound
of every element, and a planted error of a few percent must not. (The bound's
error of P is derived per element from the score accumulation, the exponent
argument's roundings, the given lse and the exponential unit: p_rel_error.)"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import bwd_bound, bwd_ratio


def bf16(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def emulate(q, k, v, dout, o_in, lse_in, causal, scale):
    """dQ, dK, dV with the kernels' roundings (float32 numpy, one head group at a time)."""
    qn, kn, vn, dn = (t.float().numpy() for t in (q, k, v, dout))
    on, ln = o_in.float().numpy(), lse_in.float().numpy()
    B, Hq, S, D = qn.shape
    g = Hq // kn.shape[1]
    dq = np.zeros_like(qn)
    dk = np.zeros_like(kn)
    dv = np.zeros_like(vn)
    mask = np.tril(np.ones((S, S), dtype=bool)) if causal else np.ones((S, S), dtype=bool)
    for b in range(B):
        for h in range(Hq):
            hk = h // g
            s = (qn[b, h] @ kn[b, hk].T).astype(np.float32)
            p = np.where(mask, np.exp2(s * np.float32(scale * math.log2(math.e)) - ln[b, h][:, None] * np.float32(math.log2(math.e))), 0).astype(np.float32)
            delta = (dn[b, h] * on[b, h]).sum(axis=1, keepdims=True, dtype=np.float32)
            dp = (dn[b, h] @ vn[b, hk].T).astype(np.float32)
            pb = bf16(p)
            dsb = bf16(p * (dp - delta))
            dv[b, hk] += pb.T @ dn[b, h]
            dk[b, hk] += dsb.T @ qn[b, h]
            dq[b, h] = dsb @ kn[b, hk]
    return bf16(dq * scale), bf16(dk * scale), bf16(dv)


@pytest.mark.parametrize("causal", [True, False])
def test_emulated_kernel_arithmetic_lies_within_the_bound(causal):
    w = workloads.Workload("bwd_tol", 1, 4, 2, 200, 64, causal, 1, 1010)
    q, k, v = workloads.make_qkv(w)
    dout = workloads.make_dout(w)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
    o_in = torch.from_numpy(o_ref).to(torch.bfloat16)
    lse_in = torch.from_numpy(lse_ref).float()
    got = emulate(q, k, v, dout, o_in, lse_in, causal, w.scale)
    ref = oracle.attention_backward(q, k, v, dout, causal)
    bnd = bwd_bound(q, k, v, dout, causal, w.scale, o_in)
    ratios = [bwd_ratio(torch.from_numpy(x), r, b_) for x, r, b_ in zip(got, ref, bnd)]
    assert max(ratios) <= 1.0, ratios
    # the bound is not loose enough to hide a real error: dV scaled by 1.05 fails
    assert bwd_ratio(torch.from_numpy(got[2] * 1.05), ref[2], bnd[2]) > 1.0
