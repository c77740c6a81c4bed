"""Tolerance checks shared by the GPU parity tests.

Bounds: |O_gpu - O_oracle| <= 1e-2 for bf16 (and fp32 partial) outputs and
|lse_gpu - lse_oracle| <= 1e-3 for fp32 lse, element by element; -inf must
match -inf exactly. One refinement for bf16 outputs: where |O_oracle| >= 4
the bf16 spacing alone is 2^-5, so a correctly rounded result can be up to
2^-6 > 1e-2 away from the exact value; there the GPU value is compared with
the oracle value rounded to bf16 (round-to-nearest-even) instead.
"""
import math

import numpy as np
import torch

O_TOL = 1e-2
LSE_TOL = 1e-3


def bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def check_o(o_gpu, o_ref: np.ndarray, tol: float = O_TOL, bf16_out: bool = True) -> float:
    """Returns max |O_gpu - O_oracle| over the elements under the plain bound."""
    g = o_gpu.detach().to(torch.float64).cpu().numpy() if isinstance(o_gpu, torch.Tensor) else np.asarray(o_gpu)
    assert g.shape == o_ref.shape, (g.shape, o_ref.shape)
    assert np.isfinite(g).all(), "non-finite output"
    err = np.abs(g - o_ref)
    if bf16_out:
        big = np.abs(o_ref) >= 4.0
        err_big = np.abs(g - bf16_round(o_ref))[big]
        assert err_big.size == 0 or err_big.max() <= tol, f"max |O - bf16(O_ref)| where |O_ref|>=4: {err_big.max()}"
        err = np.where(big, 0.0, err)
    m = float(err.max()) if err.size else 0.0
    assert m <= tol, f"max |dO| = {m} > {tol} at {np.unravel_index(err.argmax(), err.shape)}"
    return m


def check_lse(lse_gpu, lse_ref: np.ndarray, tol: float = LSE_TOL) -> float:
    g = lse_gpu.detach().to(torch.float64).cpu().numpy() if isinstance(lse_gpu, torch.Tensor) else np.asarray(lse_gpu)
    assert g.shape == lse_ref.shape
    ninf_ref = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(g), ninf_ref), "-inf pattern differs"
    fin = ~ninf_ref
    assert np.isfinite(g[fin]).all()
    err = np.abs(g[fin] - lse_ref[fin])
    m = float(err.max()) if err.size else 0.0
    assert m <= tol, f"max |dlse| = {m} > {tol}"
    return m


def gather_rows(t: torch.Tensor, rows: np.ndarray) -> torch.Tensor:
    """t [B,H,S,...] on any device, rows [B*H, R] -> [B,H,R,...] on the CPU."""
    B, H = t.shape[0], t.shape[1]
    idx = torch.from_numpy(rows).to(t.device).view(B, H, -1)
    if t.dim() == 4:
        idx = idx.unsqueeze(-1).expand(-1, -1, -1, t.shape[3])
    return torch.gather(t, 2, idx).cpu()


def _np(t) -> np.ndarray:
    return t.detach().double().cpu().numpy() if isinstance(t, torch.Tensor) else np.asarray(t, dtype=np.float64)


# Relative error of the bf16 rounding of P and dS in the backward kernels.
BF16_REL = 2.0 ** -9
# Largest relative error of the softmax's MUFU 2^x, as bounded on the device
# by tests/test_gpu_exp2.py.
EX2_REL = 4e-6
# Unit of the fp32 score accumulation inside the tensor core: the rounding
# mode of its internal adds is not documented, so one ulp per add (2^-23,
# truncation) instead of half an ulp (rounding to nearest).
ACC_U = 2.0 ** -23


def p_rel_error(s_scaled, lse_exact, lse_in, abs_qk, scale, D):
    """Relative error of P = 2^(s scale log2(e) - lse log2(e)) as the backward
    kernels form it, per element, from its sources:
      * the score s: D products accumulated in fp32, |ds| <= D ACC_U sum_d |q_d k_d|
        (the classical bound for a sum of D terms), which moves P by scale |ds|;
      * the argument x = s c - lse2 (c = scale log2 e and lse2 = lse log2 e each
        rounded to fp32, the product and the difference rounded): at most four
        fp32 roundings of magnitude <= |s c| + |lse2|, so |dx| <= 2^-22 (|s c| +
        |lse2|), which moves P by ln 2 |dx|;
      * the lse the kernel is given: P moves by |lse_in - lse|;
      * the MUFU exponential, EX2_REL; and P's bf16 rounding, BF16_REL.
    s_scaled = scale s (natural-log units); lse_exact, lse_in broadcast
    against it."""
    log2e = 1.0 / math.log(2.0)
    arg = np.abs(s_scaled) * log2e + np.abs(lse_exact) * log2e
    return (BF16_REL + EX2_REL + np.abs(lse_in - lse_exact) + math.log(2.0) * 2.0 ** -22 * arg
            + scale * D * ACC_U * abs_qk)


def bwd_bound(q, k, v, dout, causal, scale, o_in, lse_in=None):
    """Per-element bounds on the backward's error (numpy fp64, small shapes).
    The kernel's approximations: P formed in fp32 from the fp32 scores and
    the given lse, then rounded to bf16 (relative error p_rel_error, per
    element); dP = dO V^T in fp32 (error <= 2^-16 sum_d |dO_id v_jd|); delta
    formed in fp32 from the O it is given (o_in), off from the exact delta_i by
    at most dd_i = |<dO_i, o_in_i - O_i>| + 2^-16 sum_d |dO_id o_in_id|; dS
    rounded to bf16 (2^-9); the bf16 rounding of the results (added by
    bwd_ratio). So |d dS_ij| <= (p_rel_ij + 2^-9) |dS_ij| + P_ij (dd_i +
    2^-16 sum_d |dO_id v_jd|), |d P_ij| <= p_rel_ij P_ij, and each gradient's
    error is the sum of its terms' errors. lse_in is the lse the kernel is
    given ([B,Hq,S], natural log); by default the exact lse rounded to fp32."""
    qn, kn, vn, dn, on = (_np(t) for t in (q, k, v, dout, o_in))
    B, Hq, S, D = qn.shape
    g = Hq // kn.shape[1]
    bq = np.zeros_like(qn)
    bk = np.zeros_like(kn)
    bv = np.zeros_like(vn)
    mask = np.tril(np.ones((S, S), dtype=bool)) if causal else np.ones((S, S), dtype=bool)
    for b in range(B):
        for h in range(Hq):
            hk = h // g
            sc = scale * qn[b, h] @ kn[b, hk].T
            s = np.where(mask, sc, -np.inf)
            mx = s.max(axis=1, keepdims=True)
            p = np.exp(s - mx)
            tot = p.sum(axis=1, keepdims=True)
            p /= tot
            lse = mx + np.log(tot)
            lin = lse.astype(np.float32).astype(np.float64) if lse_in is None else _np(lse_in[b, h])[:, None]
            pr = np.where(mask, p_rel_error(sc, lse, lin, np.abs(qn[b, h]) @ np.abs(kn[b, hk]).T, scale, D), 0.0)
            o_ex = p @ vn[b, hk]
            dp = dn[b, h] @ vn[b, hk].T
            delta = (dn[b, h] * o_ex).sum(axis=1, keepdims=True)
            ds = p * (dp - delta)
            dd = (np.abs((dn[b, h] * (on[b, h] - o_ex)).sum(axis=1, keepdims=True))
                  + 2.0 ** -16 * np.abs(dn[b, h] * on[b, h]).sum(axis=1, keepdims=True))
            e_dp = 2.0 ** -16 * np.abs(dn[b, h]) @ np.abs(vn[b, hk]).T
            e_ds = (pr + BF16_REL) * np.abs(ds) + p * (dd + e_dp)
            bv[b, hk] += (pr * p).T @ np.abs(dn[b, h])
            bk[b, hk] += scale * e_ds.T @ np.abs(qn[b, h])
            bq[b, h] = scale * e_ds @ np.abs(kn[b, hk])
    return bq, bk, bv


def bwd_dq_rows_bound(q, k, v, dout, causal, scale, rows: np.ndarray, o_rows_in, lse_rows_in=None) -> np.ndarray:
    """bwd_bound's dQ bound for the query rows rows[b*Hq + h] only ([B*Hq, n, D]),
    row by row, for problems too large to bound whole; o_rows_in [B*Hq, n, D]
    and lse_rows_in [B*Hq, n] hold the O rows and lse values the kernel was
    given (lse by default the exact one rounded to fp32)."""
    B, Hq, S, D = q.shape
    g = Hq // k.shape[1]
    o_in = _np(o_rows_in)
    out = np.empty((B * Hq, rows.shape[1], D))
    for bh in range(B * Hq):
        b, h = divmod(bh, Hq)
        kn = k[b, h // g].double().numpy()
        vn = v[b, h // g].double().numpy()
        for r, i in enumerate(rows[bh]):
            n = int(i) + 1 if causal else S
            qi = q[b, h, i].double().numpy()
            di = dout[b, h, i].double().numpy()
            sc = scale * (kn[:n] @ qi)
            mx = sc.max()
            p = np.exp(sc - mx)
            tot = p.sum()
            p /= tot
            lse = mx + math.log(tot)
            lin = float(np.float32(lse)) if lse_rows_in is None else float(_np(lse_rows_in)[bh, r])
            pr = p_rel_error(sc, lse, lin, np.abs(kn[:n]) @ np.abs(qi), scale, D)
            o_ex = p @ vn[:n]
            ds = p * (vn[:n] @ di - di @ o_ex)
            dd = abs(float(di @ (o_in[bh, r] - o_ex))) + 2.0 ** -16 * float(np.abs(di * o_in[bh, r]).sum())
            e_dp = 2.0 ** -16 * (np.abs(vn[:n]) @ np.abs(di))
            out[bh, r] = scale * ((pr + BF16_REL) * np.abs(ds) + p * (dd + e_dp)) @ np.abs(kn[:n])
    return out


def bwd_ratio(got: torch.Tensor, ref: np.ndarray, bound: np.ndarray) -> float:
    """Largest |got - ref| / (bound + 2^-8 |ref| + 1e-4) over the elements (inf if any is not finite)."""
    g = got.double().cpu().numpy()
    if not np.isfinite(g).all():
        return float("inf")
    return float((np.abs(g - ref) / (bound + 2.0 ** -8 * np.abs(ref) + 1e-4)).max())


def fp8_bound(qd, kd, vd, causal, scale):
    """Per-element bound on |O_fp8 - O_exact| for inputs already on the e4m3
    grid (numpy fp64, small shapes): P is rounded to e4m3 in the kernel, so
    |dP| <= 2^-4 P (normal range) or 2^-10 (below 2^-6) in units where the row
    maximum is >= 1 (the kernel's reference maximum never exceeds the true one),
    and |dO_d| <= (2^-4 sum_j P_j |v_jd| + 2^-10 sum_{P_j < 2^-6} |v_jd|) / l;
    plus the bf16 rounding of O."""
    q, k, v = (t.double().numpy() for t in (qd, kd, vd))
    B, Hq, S, D = q.shape
    g = Hq // k.shape[1]
    bound = np.empty((B, Hq, S, D))
    for b in range(B):
        for h in range(Hq):
            s = scale * q[b, h] @ k[b, h // g].T
            if causal:
                s = np.where(np.tril(np.ones((S, S), dtype=bool)), s, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            l = p.sum(axis=1, keepdims=True)
            av = np.abs(v[b, h // g])
            bound[b, h] = (2.0 ** -4 * (p @ av) + 2.0 ** -10 * ((p < 2.0 ** -6) @ av)) / l
    return bound


# Largest allowed |alpha - 1| for the least-squares slopes of fp8_slope_errors.
FP8_SLOPE_TOL = 2.0 ** -7


def fp8_slope_errors(o_gpu, o_ref: np.ndarray):
    """Systematic-error check for the e4m3 forward: the least-squares slope
    alpha = sum(g r) / sum(r r) of the GPU output g on the oracle's r, per
    (batch, head) over its rows and columns, and per column d over every
    (batch, head, row). The e4m3 roundings of P are round-to-nearest-even and
    so nearly unbiased: their errors average out and leave alpha within a few
    1e-3 of 1 (an emulation of them on the CPU reaches 0.0035), whereas a
    mis-folded scale or a biased 1/l moves every element of a head, or every
    row of a column, by the same factor. Returns (max over heads, max over
    columns) of |alpha - 1|."""
    g = _np(o_gpu)
    r = np.asarray(o_ref, dtype=np.float64)
    a_head = (g * r).sum(axis=(2, 3)) / (r * r).sum(axis=(2, 3))
    a_col = (g * r).sum(axis=(0, 1, 2)) / (r * r).sum(axis=(0, 1, 2))
    return float(np.abs(a_head - 1.0).max()), float(np.abs(a_col - 1.0).max())
