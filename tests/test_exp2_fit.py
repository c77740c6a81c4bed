"""The softmax's FMA-pipe exponential (exp2_poly_x2 in csrc/attn_common.cuh)
evaluates 2^f on f in [-1/2, 1/2] as 1 + f (c1 + f (c2 + f c3)). Its
coefficients are the minimax fit for relative error, found as a linear
program on a uniform grid: minimise t subject to
|1 + c1 f + c2 f^2 + c3 f^3 - 2^f| <= t 2^f at 20,001 points. This test
re-runs that fit, rounds it to fp32 and requires the constants in the source
to be exactly those, and checks the committed polynomial's maximum relative
error on a finer grid against the fit's optimum. (The GPU side, the kernel's
routine against 2^x, is tests/test_gpu_exp2.py.)"""
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "sequence_attn_fwd_gb300", "csrc", "attn_common.cuh")


def committed_coefficients() -> np.ndarray:
    text = open(SRC).read()
    vals = []
    for i in (1, 2, 3):
        m = re.search(rf"kExp2C{i}\s*=\s*(0x[0-9a-fA-F.]+p[-+]?\d+)f", text)
        assert m, f"kExp2C{i} not found"
        vals.append(float.fromhex(m.group(1)))
    return np.array(vals, dtype=np.float32)


def minimax_fit(n: int = 20001):
    linprog = pytest.importorskip("scipy.optimize").linprog
    f = np.linspace(-0.5, 0.5, n)
    e = 2.0 ** f
    a = np.stack([f / e, f * f / e, f ** 3 / e], axis=1)  # relative error = a c - (e - 1) / e
    b = (e - 1.0) / e
    ones = np.ones((n, 1))
    a_ub = np.vstack([np.hstack([a, -ones]), np.hstack([-a, -ones])])
    b_ub = np.concatenate([b, -b])
    res = linprog([0, 0, 0, 1], A_ub=a_ub, b_ub=b_ub, bounds=[(None, None)] * 4, method="highs")
    assert res.success, res.message
    return res.x[:3], res.x[3]


def test_exp2_polynomial_coefficients_are_the_minimax_fit():
    fit, t_opt = minimax_fit()
    c = committed_coefficients()
    assert np.array_equal(fit.astype(np.float32).view(np.int32), c.view(np.int32)), (fit, c)
    f = np.linspace(-0.5, 0.5, 400001)
    c64 = c.astype(np.float64)
    p = 1.0 + f * (c64[0] + f * (c64[1] + f * c64[2]))
    rel = np.abs(p / 2.0 ** f - 1.0).max()
    assert 1.0e-4 < t_opt < 1.02e-4
    assert rel <= 1.001 * t_opt, (rel, t_opt)
