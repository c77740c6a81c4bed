"""Pins for the fp64 oracle: results fixed by the mathematics, not by the oracle.

Each test targets a mistake the oracle could plausibly contain:
  * closed forms (equal keys -> mean of V and lse = s + ln n; causal row 0 ->
    V[0] and lse = scale * q0.k0) catch a missing 1/l, a dropped max in lse,
    a wrong scale, an off-by-one or reversed causal mask;
  * V = identity turns O into the weight matrix itself, compared with
    scipy.special.softmax / logsumexp (library routines) and checked to sum
    to one;
  * an mpmath brute force at 40 digits on tiny inputs catches a transposed
    operand or wrong index;
  * invariants: chunked partials merged by log-sum-exp equal the single pass
    for every split (the equivalence stated on page
    "Ulysses与Ring-Attention序列并行技术详解", Ring-Attention part), causal rows
    ignore later keys, offsets shift the mask, scaling q equals scaling the
    scale, and GQA uses contiguous head groups.
"""
import math

import mpmath
import numpy as np
import pytest
import scipy.special
import torch

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def rand_bf16(rng, *shape, scale=1.0):
    return torch.from_numpy((scale * rng.standard_normal(shape)).astype(np.float32)).to(torch.bfloat16)


def f64(t):
    return t.to(torch.float64).numpy()


@pytest.mark.parametrize("causal", [False, True])
def test_equal_keys_give_mean_of_visible_values(causal):
    rng = np.random.default_rng(1)
    B, Hq, Hkv, S, D = 2, 4, 2, 37, 16
    q = rand_bf16(rng, B, Hq, S, D)
    krow = rand_bf16(rng, D)
    k = krow.expand(B, Hkv, S, D).contiguous()
    v = rand_bf16(rng, B, Hkv, S, D)
    o, lse = oracle.attention(q, k, v, causal)
    scale = 1 / math.sqrt(D)
    for b in range(B):
        for h in range(Hq):
            hk = h // (Hq // Hkv)
            for r in range(S):
                n = r + 1 if causal else S
                s = scale * math.fsum(float(a) * float(c) for a, c in zip(f64(q[b, h, r]), f64(krow)))
                np.testing.assert_allclose(o[b, h, r], f64(v[b, hk, :n]).mean(axis=0), rtol=0, atol=1e-13)
                assert abs(lse[b, h, r] - (s + math.log(n))) < 1e-12


def test_causal_row_zero_is_first_value_row():
    rng = np.random.default_rng(2)
    q = rand_bf16(rng, 1, 3, 20, 8)
    k = rand_bf16(rng, 1, 3, 20, 8)
    v = rand_bf16(rng, 1, 3, 20, 8)
    o, lse = oracle.attention(q, k, v, causal=True)
    for h in range(3):
        assert np.array_equal(o[0, h, 0], f64(v[0, h, 0]))
        s00 = math.fsum(float(a) * float(c) for a, c in zip(f64(q[0, h, 0]), f64(k[0, h, 0])))
        assert abs(lse[0, h, 0] - s00 / math.sqrt(8)) < 1e-13


def test_causal_rows_ignore_later_keys_and_see_their_own():
    rng = np.random.default_rng(3)
    q, k, v = (rand_bf16(rng, 1, 2, 24, 8) for _ in range(3))
    o, lse = oracle.attention(q, k, v, causal=True)
    r = 11
    k2, v2 = k.clone(), v.clone()
    k2[:, :, r + 1:] = rand_bf16(rng, 1, 2, 24 - r - 1, 8)
    v2[:, :, r + 1:] = rand_bf16(rng, 1, 2, 24 - r - 1, 8)
    o2, lse2 = oracle.attention(q, k2, v2, causal=True)
    assert np.array_equal(o[:, :, : r + 1], o2[:, :, : r + 1])
    assert np.array_equal(lse[:, :, : r + 1], lse2[:, :, : r + 1])
    assert not np.array_equal(o[:, :, r + 1:], o2[:, :, r + 1:])
    # the key at the row's own position is visible: changing it changes the row
    v3 = v.clone()
    v3[:, :, r] += 1
    o3, _ = oracle.attention(q, k, v3, causal=True)
    assert not np.array_equal(o[:, :, r], o3[:, :, r])
    assert np.array_equal(o[:, :, :r], o3[:, :, :r])


def test_identity_values_expose_softmax_weights():
    """With D = Skv and V = I, O is the weight matrix; compare with scipy's softmax."""
    rng = np.random.default_rng(4)
    B, H, S = 1, 2, 32
    D = S
    q = rand_bf16(rng, B, H, S, D, scale=2.0)
    k = rand_bf16(rng, B, H, S, D)
    v = torch.eye(S, dtype=torch.bfloat16).expand(B, H, S, S).contiguous()
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, causal)
        scores = np.einsum("bhqd,bhkd->bhqk", f64(q), f64(k)) / math.sqrt(D)
        if causal:
            scores = np.where(np.tril(np.ones((S, S), bool)), scores, -np.inf)
        np.testing.assert_allclose(o, scipy.special.softmax(scores, axis=-1), rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse, scipy.special.logsumexp(scores, axis=-1), rtol=0, atol=1e-12)
        np.testing.assert_allclose(o.sum(-1), 1.0, rtol=0, atol=1e-13)
        assert (o >= 0).all()


@pytest.mark.parametrize("causal", [False, True])
def test_mpmath_brute_force_tiny(causal):
    mpmath.mp.dps = 40
    rng = np.random.default_rng(5)
    B, Hq, Hkv, S, D = 1, 2, 1, 5, 3
    q, k, v = rand_bf16(rng, B, Hq, S, D), rand_bf16(rng, B, Hkv, S, D), rand_bf16(rng, B, Hkv, S, D)
    o, lse = oracle.attention(q, k, v, causal)
    Q, K, V = f64(q), f64(k), f64(v)
    sc = mpmath.mpf(1) / mpmath.sqrt(D)
    for h in range(Hq):
        for r in range(S):
            n = r + 1 if causal else S
            s = [sc * mpmath.fsum(mpmath.mpf(Q[0, h, r, d]) * mpmath.mpf(K[0, 0, t, d]) for d in range(D))
                 for t in range(n)]
            z = mpmath.fsum(mpmath.e ** x for x in s)
            for d in range(D):
                want = mpmath.fsum(mpmath.e ** s[t] * mpmath.mpf(V[0, 0, t, d]) for t in range(n)) / z
                assert abs(o[0, h, r, d] - float(want)) < 1e-14
            assert abs(lse[0, h, r] - float(mpmath.log(z))) < 1e-13


def test_dominant_key_and_no_overflow():
    """Scores near 1e3 overflow exp() unless the row max is subtracted first."""
    rng = np.random.default_rng(6)
    S, D = 16, 8
    q = torch.full((1, 1, S, D), 16.0, dtype=torch.bfloat16)
    k = rand_bf16(rng, 1, 1, S, D, scale=0.1)
    k[0, 0, 7] = 32.0  # s_7 = 16*32*8/sqrt(8) ~ 1448, far above every other score
    v = rand_bf16(rng, 1, 1, S, D)
    o, lse = oracle.attention(q, k, v, causal=False)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(f64(v[0, 0, 7]), (S, D)), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], 16.0 * 32.0 * D / math.sqrt(D), rtol=1e-15)


def test_scale_equals_scaled_queries():
    rng = np.random.default_rng(7)
    q, k, v = (rand_bf16(rng, 1, 2, 19, 16) for _ in range(3))
    o1, l1 = oracle.attention(q, k, v, True, scale=2.0 / 4.0)
    o2, l2 = oracle.attention((q.float() * 2).to(torch.bfloat16), k, v, True)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def test_gqa_uses_contiguous_head_groups():
    rng = np.random.default_rng(8)
    B, Hq, Hkv, S, D = 1, 6, 2, 12, 8
    q = rand_bf16(rng, B, Hq, S, D)
    k = rand_bf16(rng, B, Hkv, S, D)
    v = rand_bf16(rng, B, Hkv, S, D)
    o, lse = oracle.attention(q, k, v, causal=False)
    for h in range(Hq):
        hk = h // 3  # heads 0,1,2 -> KV head 0; 3,4,5 -> KV head 1
        scores = f64(q[0, h]) @ f64(k[0, hk]).T / math.sqrt(D)
        np.testing.assert_allclose(o[0, h], scipy.special.softmax(scores, -1) @ f64(v[0, hk]), atol=1e-13)
        np.testing.assert_allclose(lse[0, h], scipy.special.logsumexp(scores, -1), atol=1e-12)


def _chunked(q, k, v, causal, bounds, q_off=0):
    parts_o, parts_l = [], []
    for a, b in zip(bounds[:-1], bounds[1:]):
        o, l = oracle.attention(q, k[:, :, a:b].contiguous(), v[:, :, a:b].contiguous(), causal,
                                q_off=q_off, kv_off=a)
        parts_o.append(o)
        parts_l.append(l)
    return oracle.lse_merge(np.stack(parts_o), np.stack(parts_l))


@pytest.mark.parametrize("causal", [False, True])
def test_chunked_merge_equals_single_pass_for_every_split(causal):
    rng = np.random.default_rng(9)
    B, Hq, Hkv, S, D = 2, 4, 2, 48, 8
    q, k, v = rand_bf16(rng, B, Hq, S, D), rand_bf16(rng, B, Hkv, S, D), rand_bf16(rng, B, Hkv, S, D)
    o_full, l_full = oracle.attention(q, k, v, causal)
    splits = [[0, S]] + [list(range(0, S + 1, S // P)) for P in (2, 3, 4, 6, 8, 12, 16, 24, 48)]
    splits += [[0, 5, 6, 29, 47, 48], [0, 1, 48]]
    for bounds in splits:
        o, l = _chunked(q, k, v, causal, bounds)
        np.testing.assert_allclose(o, o_full, rtol=0, atol=1e-13)
        np.testing.assert_allclose(l, l_full, rtol=0, atol=1e-12)


def test_query_offset_selects_rows_of_the_full_causal_problem():
    rng = np.random.default_rng(10)
    S, D = 40, 8
    q, k, v = (rand_bf16(rng, 1, 2, S, D) for _ in range(3))
    o_full, l_full = oracle.attention(q, k, v, True)
    a, b = 13, 31
    o, l = oracle.attention(q[:, :, a:b].contiguous(), k, v, True, q_off=a)
    assert np.array_equal(o, o_full[:, :, a:b]) and np.array_equal(l, l_full[:, :, a:b])
    # a block of rows against a later chunk of keys: rows before the chunk see nothing
    o2, l2 = oracle.attention(q, k[:, :, 20:].contiguous(), v[:, :, 20:].contiguous(), True, kv_off=20)
    assert (o2[:, :, :20] == 0).all() and np.isneginf(l2[:, :, :20]).all()
    assert np.isfinite(l2[:, :, 20:]).all()


def test_row_subset_matches_full_rows():
    rng = np.random.default_rng(11)
    q, k, v = (rand_bf16(rng, 1, 3, 33, 8) for _ in range(3))
    o_full, l_full = oracle.attention(q, k, v, True)
    rows = np.array([[0, 5, 32], [1, 2, 3], [31, 30, 7]], dtype=np.int64)
    o, l = oracle.attention(q, k, v, True, rows=rows)
    for h in range(3):
        assert np.array_equal(o[0, h], o_full[0, h, rows[h]])
        assert np.array_equal(l[0, h], l_full[0, h, rows[h]])


def test_merge_closed_forms():
    rng = np.random.default_rng(12)
    o1 = rng.standard_normal((5, 4))
    o2 = rng.standard_normal((5, 4))
    # identical partials: same O, lse + ln 2
    o, l = oracle.lse_merge(np.stack([o1, o1]), np.full((2, 5), 3.0))
    np.testing.assert_allclose(o, o1, rtol=0, atol=1e-15)
    np.testing.assert_allclose(l, 3.0 + math.log(2), rtol=0, atol=1e-15)
    # masses 1 and 3: weights 1/4 and 3/4, lse = ln 4
    o, l = oracle.lse_merge(np.stack([o1, o2]), np.stack([np.zeros(5), np.full(5, math.log(3))]))
    np.testing.assert_allclose(o, 0.25 * o1 + 0.75 * o2, rtol=0, atol=1e-15)
    np.testing.assert_allclose(l, math.log(4), rtol=0, atol=1e-15)
    # P = 1 is the identity
    o, l = oracle.lse_merge(o1[None], np.full((1, 5), -2.5))
    assert np.array_equal(o, o1) and (l == -2.5).all()
    # empty partials carry no weight; all-empty rows give O = 0, lse = -inf
    lse = np.stack([np.array([-np.inf, 1.0, -np.inf, 0, 0]), np.array([2.0, -np.inf, -np.inf, 0, 0])])
    o, l = oracle.lse_merge(np.stack([o1, o2]), lse)
    np.testing.assert_allclose(o[0], o2[0], atol=1e-15)
    np.testing.assert_allclose(o[1], o1[1], atol=1e-15)
    assert (o[2] == 0).all() and l[2] == -np.inf
    assert l[0] == 2.0 and l[1] == 1.0


def test_merge_lse_matches_scipy_logsumexp():
    rng = np.random.default_rng(13)
    lse = 10 * rng.standard_normal((7, 50))
    o_parts = rng.standard_normal((7, 50, 3))
    o, l = oracle.lse_merge(o_parts, lse)
    np.testing.assert_allclose(l, scipy.special.logsumexp(lse, axis=0), rtol=0, atol=1e-12)
    w = scipy.special.softmax(lse, axis=0)
    np.testing.assert_allclose(o, np.einsum("pr,prd->rd", w, o_parts), rtol=0, atol=1e-13)


def test_rejects_bad_arguments():
    q = torch.zeros(1, 3, 4, 8, dtype=torch.bfloat16)
    k = torch.zeros(1, 2, 4, 8, dtype=torch.bfloat16)
    with pytest.raises(AssertionError):
        oracle.attention(q, k, k, False)
    with pytest.raises(ValueError):
        oracle.attention(q[:, :2].contiguous(), k, k, False, rows=np.array([[0], [9]]))
