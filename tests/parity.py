"""Tolerance checks shared by the GPU parity tests.

Bounds: |O_gpu - O_oracle| <= 1e-2 for bf16 (and fp32 partial) outputs and
|lse_gpu - lse_oracle| <= 1e-3 for fp32 lse, element by element; -inf must
match -inf exactly. One refinement for bf16 outputs: where |O_oracle| >= 4
the bf16 spacing alone is 2^-5, so a correctly rounded result can be up to
2^-6 > 1e-2 away from the exact value; there the GPU value is compared with
the oracle value rounded to bf16 (round-to-nearest-even) instead.
"""
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


def bwd_bound(q, k, v, dout, o_used, causal, scale):
    """Per-element bounds on the backward's error (numpy fp64, small shapes).
    The kernel's approximations beyond fp32 accumulation: P and dS rounded to
    bf16 before their products (2^-9 relative each), delta computed from the O
    it is given (the bf16 forward output, whose exact difference from the exact
    O is known here), and the bf16 rounding of the results. With dd_i = |<dO_i,
    O_used_i - O_i>| (plus its bf16 share): |d dS_ij| <= 2^-9 |dS_ij| + P_ij dd_i,
    and each gradient's error is the sum of its terms' errors, + 2^-8 |result|."""
    qn, kn, vn, dn, on = (t.double().numpy() for t in (q, k, v, dout, o_used))
    B, Hq, S, D = qn.shape
    g = Hq // kn.shape[1]
    bq = np.zeros_like(qn)
    bk = np.zeros_like(kn)
    bv = np.zeros_like(vn)
    mask = np.tril(np.ones((S, S), dtype=bool)) if causal else np.ones((S, S), dtype=bool)
    for b in range(B):
        for h in range(Hq):
            hk = h // g
            s = np.where(mask, scale * qn[b, h] @ kn[b, hk].T, -np.inf)
            p = np.exp(s - s.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            o_ex = p @ vn[b, hk]
            dp = dn[b, h] @ vn[b, hk].T
            delta = (dn[b, h] * o_ex).sum(axis=1, keepdims=True)
            ds = p * (dp - delta)
            dd = np.abs((dn[b, h] * (on[b, h] - o_ex)).sum(axis=1, keepdims=True))
            dd += 2.0 ** -8 * (np.abs(dn[b, h]) * np.abs(on[b, h])).sum(axis=1, keepdims=True)
            e_ds = 2.0 ** -9 * np.abs(ds) + p * dd
            bv[b, hk] += 2.0 ** -9 * p.T @ np.abs(dn[b, h])
            bk[b, hk] += scale * e_ds.T @ np.abs(qn[b, h])
            bq[b, h] = scale * e_ds @ np.abs(kn[b, hk])
    return bq, bk, bv


def bwd_ratio(got: torch.Tensor, ref: np.ndarray, bound: np.ndarray) -> float:
    """Largest |got - ref| / (bound + 2^-8 |ref| + 1e-4) over the elements (inf if any is not finite)."""
    g = got.double().cpu().numpy()
    if not np.isfinite(g).all():
        return float("inf")
    return float((np.abs(g - ref) / (bound + 2.0 ** -8 * np.abs(ref) + 1e-4)).max())
