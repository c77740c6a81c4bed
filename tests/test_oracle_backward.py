"""Pins of the oracle's attention backward (no GPU): its gradients against
central finite differences of a brute-force fp64 forward (a different
computation of the same loss), exact invariants of the softmax Jacobian, and
GQA as the group sum of the expanded problem."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads


def forward_np(q, k, v, causal, scale):
    """O for float64 numpy q [H,S,D], k, v [Hkv,S,D] (brute force, tiny shapes)."""
    H, S, D = q.shape
    g = H // k.shape[0]
    o = np.empty_like(q)
    for h in range(H):
        s = scale * q[h] @ k[h // g].T
        if causal:
            s = np.where(np.tril(np.ones((S, S), dtype=bool)), s, -np.inf)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        o[h] = (p / p.sum(axis=1, keepdims=True)) @ v[h // g]
    return o


def qkvd(Hq, Hkv, S, D, seed):
    q, k, v = workloads.make_qkv(workloads.Workload("bwd", 1, Hq, Hkv, S, D, True, 1, seed))
    d, _, _ = workloads.make_qkv(workloads.Workload("bwd", 1, Hq, Hq, S, D, True, 1, seed + 1))
    return q, k, v, d


@pytest.mark.parametrize("causal", [True, False])
def test_gradients_match_finite_differences(causal):
    Hq, Hkv, S, D = 2, 1, 6, 4
    q, k, v, d = qkvd(Hq, Hkv, S, D, 321)
    scale = 1.0 / math.sqrt(D)
    dq, dk, dv = oracle.attention_backward(q, k, v, d, causal)
    qn, kn, vn, dn = (t[0].double().numpy() for t in (q, k, v, d))
    loss = lambda q_, k_, v_: float((dn * forward_np(q_, k_, v_, causal, scale)).sum())
    eps = 1e-6
    for name, x, grad in (("q", qn, dq[0]), ("k", kn, dk[0]), ("v", vn, dv[0])):
        num = np.empty_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args = {"q": (qn, kn, vn), "k": (qn, kn, vn), "v": (qn, kn, vn)}[name]
            a_p = [xp if n == name else a for n, a in zip("qkv", args)]
            a_m = [xm if n == name else a for n, a in zip("qkv", args)]
            num[idx] = (loss(*a_p) - loss(*a_m)) / (2 * eps)
        np.testing.assert_allclose(grad, num, rtol=0, atol=2e-7, err_msg=name)


def test_softmax_jacobian_invariants():
    """Every row of dS sums to zero, so dK sums to zero over the keys of a head;
    with all keys equal the scores are constant and dQ vanishes."""
    q, k, v, d = qkvd(4, 2, 40, 16, 77)
    for causal in (True, False):
        dq, dk, dv = oracle.attention_backward(q, k, v, d, causal)
        assert np.abs(dk.sum(axis=2)).max() < 1e-12 * max(1.0, np.abs(dk).max())
    k_eq = k[:, :, :1].expand(k.shape).contiguous()
    dq, dk, dv = oracle.attention_backward(q, k_eq, v, d, False)
    assert np.abs(dq).max() < 1e-13


def test_gqa_is_the_group_sum_of_the_expanded_problem():
    Hq, Hkv = 4, 2
    q, k, v, d = qkvd(Hq, Hkv, 24, 8, 99)
    dq, dk, dv = oracle.attention_backward(q, k, v, d, True)
    ke, ve = (t.repeat_interleave(Hq // Hkv, dim=1).contiguous() for t in (k, v))
    dq2, dk2, dv2 = oracle.attention_backward(q, ke, ve, d, True)
    np.testing.assert_allclose(dq, dq2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk, dk2.reshape(1, Hkv, Hq // Hkv, 24, 8).sum(axis=2), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv, dv2.reshape(1, Hkv, Hq // Hkv, 24, 8).sum(axis=2), rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [True, False])
def test_dq_rows_equal_the_whole_backward(causal):
    """The row-by-row dQ (used on problems too large to differentiate whole)
    gives the whole backward's dQ rows, in the same order of operations."""
    Hq, Hkv, S, D = 4, 2, 50, 16
    q, k, v, d = qkvd(Hq, Hkv, S, D, 5)
    dq, _, _ = oracle.attention_backward(q, k, v, d, causal)
    rows = np.stack([np.array([0, 7, 31, 49]) for _ in range(Hq)])
    got = oracle.attention_backward_dq_rows(q, k, v, d, causal, rows)
    for h in range(Hq):
        np.testing.assert_array_equal(got[h], dq[0, h, rows[h]])
    with pytest.raises(ValueError):
        oracle.attention_backward_dq_rows(q, k, v, d, causal, rows + 1)  # row 50 is out of range
