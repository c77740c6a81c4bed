"""The e4m3 forward's parity criteria (tests/parity.py fp8_bound and
fp8_slope_errors) against an emulation of the kernel's one approximation
beyond rounding on the CPU: P rounded to e4m3 (round to nearest even) before
P V, l summed from the unrounded P, O rounded to bf16. The emulated O must
pass the three criteria of the GPU test: every element within the bound (plus
the 2^-8 |O| + 1e-4 the GPU test adds), the mean error below a quarter of the
mean bound, and the least-squares slopes of O on the oracle's, per head and
per column, within 2^-7 of 1. Systematic errors must fail them: O uniformly
3 % or 10 % too large, a V scale off by 10 %, one column off by 5 %, or O
taken from the wrong head. The element bound alone lets a uniform error of
about 10 % through (it is a worst case of 2^-4 per P); the slopes do not."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import FP8_SLOPE_TOL, fp8_bound, fp8_slope_errors


def e4m3_grid(t: torch.Tensor, scale: float) -> torch.Tensor:
    """t / scale rounded to e4m3, times scale (exact in bf16 for power-of-two scales)."""
    return ((t.float() / scale).to(torch.float8_e4m3fn).float() * scale).to(torch.bfloat16)


def emulate(q, k, v, causal, scale):
    qn, kn, vn = (t.double().numpy() for t in (q, k, v))
    B, Hq, S, D = qn.shape
    g = Hq // kn.shape[1]
    out = np.empty((B, Hq, S, D))
    for b in range(B):
        for h in range(Hq):
            s = scale * qn[b, h] @ kn[b, h // g].T
            if causal:
                s = np.where(np.tril(np.ones((S, S), dtype=bool)), s, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True)).astype(np.float32)
            l = p.sum(axis=1, keepdims=True, dtype=np.float64)
            p8 = torch.from_numpy(p).to(torch.float8_e4m3fn).double().numpy()
            o = (p8 @ vn[b, h // g]) / l
            out[b, h] = torch.from_numpy(o).to(torch.bfloat16).double().numpy()
    return out


@pytest.mark.parametrize("causal", [True, False])
def test_emulated_e4m3_p_lies_within_the_bound(causal):
    w = workloads.Workload("fp8_tol", 1, 4, 2, 320, 128, causal, 1, 1011)
    q, k, v = workloads.make_qkv(w)
    qd, kd, vd = e4m3_grid(q, 0.25), e4m3_grid(k, 0.5), e4m3_grid(v, 0.25)
    o_ref, _ = oracle.attention(qd, kd, vd, causal)
    got = emulate(qd, kd, vd, causal, w.scale)
    tol = fp8_bound(qd, kd, vd, causal, w.scale) + 2.0 ** -8 * np.abs(o_ref) + 1e-4

    def passes(x):
        err = np.abs(x - o_ref)
        head_dev, col_dev = fp8_slope_errors(x, o_ref)
        return (bool((err <= tol).all()) and err.mean() <= 0.25 * tol.mean()
                and head_dev <= FP8_SLOPE_TOL and col_dev <= FP8_SLOPE_TOL)

    assert passes(got)
    # the emulated slopes sit well inside the limit
    assert max(fp8_slope_errors(got, o_ref)) <= 0.5 * FP8_SLOPE_TOL
    assert not passes(got * 1.03)
    assert not passes(got * 1.10)
    assert not passes(got * 1.25)
    # V's scale folded in wrong by 10 %: the attention of 1.1 V
    assert not passes(emulate(qd, kd, (vd.float() * 1.1).to(torch.bfloat16), causal, w.scale))
    one_col = got.copy()
    one_col[..., 7] *= 1.05
    assert not passes(one_col)
    assert not passes(np.roll(got, 1, axis=1))  # a neighbouring head's output
