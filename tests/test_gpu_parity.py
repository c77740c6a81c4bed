"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Small cases span several 128-row tiles and a ragged tail and are checked in
full; the five named workloads run at full size in the launch configuration
the benchmark times and are checked on sampled query rows.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.parity import (FP8_SLOPE_TOL, LSE_TOL, O_TOL, bwd_bound, bwd_dq_rows_bound, bwd_ratio, check_lse, check_o,
                          fp8_bound, fp8_slope_errors, gather_rows)

pytestmark = pytest.mark.gpu

W = workloads.WORKLOADS


@pytest.fixture(scope="module")
def sa(cuda_dev):
    import sequence_attn_fwd_gb300 as sa

    yield sa
    sa.query_device_error()  # no kernel may have recorded a timed-out wait


def adhoc(B, Hq, Hkv, S, D, causal, seed=77):
    return workloads.Workload("adhoc", B, Hq, Hkv, S, D, causal, 1, seed)


def to_dev(*ts):
    return [t.cuda() for t in ts]


@pytest.mark.parametrize("causal", [False, True])
def test_tiny_workload_full(sa, causal):
    w = W["tiny_b1h2s256d64"]
    q, k, v = workloads.make_qkv(w)
    o_ref, lse_ref = oracle.attention(q, k, v, causal)
    o, lse = sa.attn_fwd(*to_dev(q, k, v), causal=causal)
    check_o(o, o_ref)
    check_lse(lse, lse_ref)


def test_tiny_workload_matches_stored_golden_rows(sa):
    from tests.test_golden import load_golden

    g, cases = load_golden()
    w = W[g["workload"]]
    q, k, v = workloads.make_qkv(w)
    for name, (o_ref, lse_ref) in cases.items():
        o, lse = sa.attn_fwd(*to_dev(q, k, v), causal=(name == "causal"))
        check_o(o[0, :, g["rows"]], o_ref)
        check_lse(lse[0, :, g["rows"]], lse_ref)


SHAPES = [
    # B, Hq, Hkv, S, D, causal
    (2, 4, 2, 1000, 128, True),
    (2, 4, 2, 1000, 128, False),
    (1, 3, 1, 777, 64, True),
    (1, 6, 3, 640, 64, False),
    (1, 2, 1, 129, 128, True),
    (1, 2, 2, 127, 64, False),
    (1, 1, 1, 1, 128, True),
    (1, 1, 1, 1, 64, False),
    (3, 2, 2, 384, 128, True),
    (1, 8, 1, 520, 128, True),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b{}hq{}hkv{}s{}d{}{}".format(*s[:5], "c" if s[5] else ""))
def test_attn_fwd_against_oracle(sa, shape):
    B, Hq, Hkv, S, D, causal = shape
    q, k, v = workloads.make_qkv(adhoc(B, Hq, Hkv, S, D, causal))
    o_ref, lse_ref = oracle.attention(q, k, v, causal)
    o, lse = sa.attn_fwd(*to_dev(q, k, v), causal=causal)
    check_o(o, o_ref)
    check_lse(lse, lse_ref)


def test_attn_fwd_custom_scale_and_large_scores(sa):
    """Scores of a few hundred: exponentials stay finite only with the max subtracted."""
    q, k, v = workloads.make_qkv(adhoc(1, 2, 2, 300, 128, True, seed=5))
    q = (q.float() * 8).to(torch.bfloat16)
    o_ref, lse_ref = oracle.attention(q, k, v, True, scale=0.5)
    o, lse = sa.attn_fwd(*to_dev(q, k, v), causal=True, scale=0.5)
    check_o(o, o_ref)
    check_lse(lse, lse_ref)


def test_outputs_leave_neighbouring_memory_untouched(sa):
    """Guard regions around every output (compute-sanitizer stands in for nothing here)."""
    B, Hq, S, D = 1, 3, 333, 128
    q, k, v = to_dev(*workloads.make_qkv(adhoc(B, Hq, Hq, S, D, True)))
    n_o, n_l, g = B * Hq * S * D, B * Hq * S, 4096
    o_buf = torch.full((n_o + 2 * g,), 7.0, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((n_l + 2 * g,), 7.0, dtype=torch.float32, device="cuda")
    o = o_buf[g:g + n_o].view(B, Hq, S, D)
    lse = l_buf[g:g + n_l].view(B, Hq, S)
    sa.attn_fwd(q, k, v, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert (o_buf[:g] == 7).all() and (o_buf[g + n_o:] == 7).all()
    assert (l_buf[:g] == 7).all() and (l_buf[g + n_l:] == 7).all()
    po = torch.full((n_o + 2 * g,), 7.0, dtype=torch.float32, device="cuda")
    sa.attn_partial(q, k[:, :, 100:200], v[:, :, 100:200], 0, 100, True,
                    out=po[g:g + n_o].view(B, Hq, S, D), lse=l_buf[g:g + n_l].view(B, Hq, S))
    torch.cuda.synchronize()
    assert (po[:g] == 7).all() and (po[g + n_o:] == 7).all()
    assert (l_buf[:g] == 7).all() and (l_buf[g + n_l:] == 7).all()


@pytest.mark.parametrize("q_off,a,b", [(0, 0, 256), (0, 256, 700), (0, 700, 1000), (300, 128, 512), (0, 999, 1000)])
def test_attn_partial_offsets_against_oracle(sa, q_off, a, b):
    B, Hq, Hkv, S, D = 1, 4, 2, 1000, 128
    q, k, v = workloads.make_qkv(adhoc(B, Hq, Hkv, S, D, True, seed=9))
    qb = q[:, :, q_off:].contiguous()
    o_ref, lse_ref = oracle.attention(qb, k[:, :, a:b].contiguous(), v[:, :, a:b].contiguous(), True,
                                      q_off=q_off, kv_off=a)
    qd, kd, vd = to_dev(qb, k, v)
    o, lse = sa.attn_partial(qd, kd[:, :, a:b], vd[:, :, a:b], q_off, a, True)
    check_o(o, o_ref, bf16_out=False)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("D", [64, 128])
def test_attn_partial_long_blocks_against_oracle(sa, D):
    """fp32 partials of blocks longer than 2048 keys take every exponential on
    the MUFU (shorter ones put a share on the FMA-pipe polynomial): a 2500-key
    chunk as a single problem, and as one block of a table beside a short one,
    checked in full against the oracle."""
    B, Hq, Hkv, S = 1, 4, 2, 2900
    a = 400  # the long chunk is keys [400, 2900): 2500 keys
    q, k, v = workloads.make_qkv(adhoc(B, Hq, Hkv, S, D, True, seed=17))
    qd, kd, vd = to_dev(q, k, v)
    o_ref, lse_ref = oracle.attention(q, k[:, :, a:].contiguous(), v[:, :, a:].contiguous(), True, kv_off=a)
    o, lse = sa.attn_partial(qd, kd[:, :, a:], vd[:, :, a:], 0, a, True)
    check_o(o, o_ref, bf16_out=False)
    check_lse(lse, lse_ref)
    # the same chunk in a block table with the short chunk [0, 400) beside it (part 1)
    o2, l2 = sa.attn_partial_blocks(qd, kd, vd, [(0, a, 0, 0, a, S, S - a, 0), (0, 0, 0, 0, 0, S, a, 1)],
                                    n_parts=2, causal=True)
    check_o(o2[0], o_ref, bf16_out=False)
    check_lse(l2[0], lse_ref)
    o_ref1, lse_ref1 = oracle.attention(q, k[:, :, :a].contiguous(), v[:, :, :a].contiguous(), True)
    check_o(o2[1], o_ref1, bf16_out=False)
    check_lse(l2[1], lse_ref1)


def test_attn_partial_chunk_invisible_to_every_row(sa):
    q, k, v = to_dev(*workloads.make_qkv(adhoc(1, 2, 2, 512, 64, True)))
    o, lse = sa.attn_partial(q[:, :, :256].contiguous(), k[:, :, 256:], v[:, :, 256:], 0, 256, True)
    torch.cuda.synchronize()
    assert (o == 0).all() and torch.isneginf(lse).all()


@pytest.mark.parametrize("D", [64, 128])
def test_attn_partial_skip_empty_leaves_invisible_rows_untouched(sa, D):
    """Chunk [600, 900) of 1000 keys under causal masking: query rows < 600 see none
    of it (whole 256-row blocks and part of one tile). With skip_empty their O rows
    keep their previous contents and their lse is -inf; all other rows match."""
    B, Hq, Hkv, S = 1, 4, 2, 1000
    a, b = 600, 900
    q, k, v = workloads.make_qkv(adhoc(B, Hq, Hkv, S, D, True, seed=13))
    o_ref, lse_ref = oracle.attention(q, k[:, :, a:b].contiguous(), v[:, :, a:b].contiguous(), True, kv_off=a)
    qd, kd, vd = to_dev(q, k, v)
    out = torch.full((B, Hq, S, D), 7.0, dtype=torch.float32, device="cuda")
    o, lse = sa.attn_partial(qd, kd[:, :, a:b], vd[:, :, a:b], 0, a, True, out=out, skip_empty=True)
    torch.cuda.synchronize()
    check_lse(lse, lse_ref)
    empty = torch.isneginf(lse)
    assert empty[:, :, :a].all() and not empty[:, :, a:].any()
    assert (o[:, :, :a] == 7.0).all()
    check_o(o[:, :, a:], o_ref[:, :, a:], bf16_out=False)


def test_ring_reduced_size_against_oracle_and_single_pass(sa):
    w = W["ring8_b2h32s4096d128_causal"]
    S = 1024
    q, k, v = workloads.make_qkv(w, S=S)
    q, k, v = q[:, :4].contiguous(), k[:, :4].contiguous(), v[:, :4].contiguous()
    o_ref, lse_ref = oracle.attention(q, k, v, True)
    qd, kd, vd = to_dev(q, k, v)
    o_ring, lse_ring = sa.ring_attn_fwd(qd, kd, vd, P=8, causal=True)
    check_o(o_ring, o_ref)
    check_lse(lse_ring, lse_ref)
    o_one, lse_one = sa.attn_fwd(qd, kd, vd, causal=True)
    assert (o_ring.float() - o_one.float()).abs().max().item() <= O_TOL
    assert (lse_ring - lse_one).abs().max().item() <= LSE_TOL


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal_pattern", [True, False])
def test_lse_merge_on_synthetic_partials(sa, D, causal_pattern):
    P, B, H, S = 16, 2, 3, 512
    o_parts, lse_parts = workloads.make_partials(P, B, H, S, D, seed=31, causal=causal_pattern)
    if not causal_pattern:  # scattered empty partials and one fully empty row
        lse_parts[3, 0, 1, :100] = -np.inf
        lse_parts[:, 1, 2, 7] = -np.inf
    o_ref, lse_ref = oracle.lse_merge(o_parts, lse_parts)
    op, lp = to_dev(o_parts, lse_parts)
    o32, l32 = sa.lse_merge(op, lp, out_dtype=torch.float32)
    check_o(o32, o_ref, tol=1e-5, bf16_out=False)
    check_lse(l32, lse_ref, tol=1e-5)
    o16, l16 = sa.lse_merge(op, lp, out_dtype=torch.bfloat16)
    check_o(o16, o_ref, tol=O_TOL)
    # in place: the merged result written over part 0
    sa.lse_merge(op, lp, out_dtype=torch.float32, out=op[0], lse=lp[0])
    check_o(op[0], o_ref, tol=1e-5, bf16_out=False)
    check_lse(lp[0], lse_ref, tol=1e-5)


@pytest.mark.parametrize("P,D", [(1, 128), (2, 128), (5, 128), (32, 128), (33, 128), (3, 64), (32, 64),
                                 (64, 64)])
def test_lse_merge_part_counts(sa, P, D):
    """Both merge paths (bulk copies up to 32 parts, rows of 130 not a multiple of
    the row group; the row kernel beyond)."""
    o_parts, lse_parts = workloads.make_partials(P, 1, 2, 130, D, seed=40 + P, causal=False)
    o_ref, lse_ref = oracle.lse_merge(o_parts, lse_parts)
    o, l = sa.lse_merge(*to_dev(o_parts, lse_parts), out_dtype=torch.float32)
    check_o(o, o_ref, tol=1e-5, bf16_out=False)
    check_lse(l, lse_ref, tol=1e-5)


@pytest.mark.parametrize("fused", [True, False], ids=["fused", "per_block"])
@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
@pytest.mark.parametrize("shape", [(1, 4, 2, 2048, 128, 4), (2, 3, 1, 1536, 64, 3), (1, 2, 2, 1200, 128, 3)],
                         ids=["gqa_s2048_p4", "d64_s1536_p3", "ragged_chunks_s1200_p3"])
def test_emulated_ring_layouts_against_oracle(sa, layout, shape, fused):
    """P emulated ring devices, each computing the blocks the schedule gives it
    hop by hop (one grouped launch per device and hop, or one attn_partial per
    block) and merging per query chunk: the assembled output is the
    single-pass causal attention."""
    B, Hq, Hkv, S, D, P = shape
    q, k, v = workloads.make_qkv(adhoc(B, Hq, Hkv, S, D, True, seed=55))
    o_ref, lse_ref = oracle.attention(q, k, v, True)
    ring = sa.EmulatedRing(*to_dev(q, k, v), P=P, layout=layout, causal=True, fused=fused)
    hop_ms, merge_ms = ring.run(timing=True)
    assert len(hop_ms) == P and all(len(r) == P for r in hop_ms) and len(merge_ms) == P
    o, lse = ring.output()
    check_o(o, o_ref)
    check_lse(lse, lse_ref)


def packed(Hq, Hkv, total_q, total_k, D, seed):
    """Packed [H, total, D] bf16 tensors from the seeded generator."""
    q, _, _ = workloads.make_qkv(adhoc(1, Hq, Hq, max(total_q, 1), D, False, seed=seed))
    _, k, v = workloads.make_qkv(adhoc(1, Hkv, Hkv, max(total_k, 1), D, False, seed=seed + 1))
    return q[0, :, :total_q].contiguous(), k[0, :, :total_k].contiguous(), v[0, :, :total_k].contiguous()


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D,Hq,Hkv", [(128, 4, 2), (64, 3, 3)])
def test_attn_fwd_varlen_against_oracle(sa, causal, D, Hq, Hkv):
    """Packed sequences of lengths 1 .. 517 (one empty), each compared with the
    oracle on its own rows; a sequence's last tile ends inside the next one's."""
    lens = [1, 127, 128, 0, 129, 300, 517, 64]
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    q, k, v = packed(Hq, Hkv, cu[-1], cu[-1], D, seed=91)
    o, lse = sa.attn_fwd_varlen(*to_dev(q, k, v), cu, cu, causal=causal)
    torch.cuda.synchronize()
    for s_, (a, b) in enumerate(zip(cu[:-1], cu[1:])):
        if b == a:
            continue
        o_ref, lse_ref = oracle.attention(q[None, :, a:b].contiguous(), k[None, :, a:b].contiguous(),
                                          v[None, :, a:b].contiguous(), causal)
        check_o(o[None, :, a:b], o_ref)
        check_lse(lse[None, :, a:b], lse_ref)


def test_attn_fwd_varlen_bottom_right_causal(sa):
    """Fewer query rows than keys: the mask is aligned at the bottom right
    (query i sees keys j <= i + Skv - Sq); more query rows than keys: the first
    rows see nothing (O = 0, lse = -inf)."""
    cq, ck = [0, 100, 150, 350], [0, 300, 350, 450]
    Hq, Hkv, D = 2, 1, 128
    q, k, v = packed(Hq, Hkv, cq[-1], ck[-1], D, seed=93)
    o, lse = sa.attn_fwd_varlen(*to_dev(q, k, v), cq, ck, causal=True)
    torch.cuda.synchronize()
    for (qa, qb), (ka, kb) in zip(zip(cq[:-1], cq[1:]), zip(ck[:-1], ck[1:])):
        sq, sk = qb - qa, kb - ka
        o_ref, lse_ref = oracle.attention(q[None, :, qa:qb].contiguous(), k[None, :, ka:kb].contiguous(),
                                          v[None, :, ka:kb].contiguous(), True, q_off=sk - sq, kv_off=0)
        check_o(o[None, :, qa:qb], o_ref)
        check_lse(lse[None, :, qa:qb], lse_ref)
    assert torch.isneginf(lse[:, 150:250]).all()  # the 3rd sequence: rows i < Sq - Skv = 100 see no key


def test_attn_partial_blocks_against_oracle(sa):
    """Ragged blocks at arbitrary rows and positions, overlapping query ranges,
    two output parts; every block's rows compared with the oracle."""
    B, Hq, Hkv, D = 2, 4, 2, 128
    q_rows, kv_rows, o_rows = 700, 900, 640
    q, k, v = workloads.make_qkv(adhoc(B, Hq, Hkv, max(q_rows, kv_rows), D, False, seed=97))
    q, k, v = q[:, :, :q_rows].contiguous(), k[:, :, :kv_rows].contiguous(), v[:, :, :kv_rows].contiguous()
    blocks = [(0, 0, 0, 0, 0, 300, 400, 0),
              (300, 400, 300, 300, 400, 340, 500, 0),
              (0, 100, 0, 50, 100, 257, 333, 1),
              (450, 0, 300, 1000, 0, 129, 900, 1),
              (600, 777, 500, 5, 900, 100, 123, 1)]
    for causal in (True, False):
        out = torch.full((2, B, Hq, o_rows, D), 7.0, dtype=torch.float32, device="cuda")
        lse = torch.full((2, B, Hq, o_rows), 7.0, dtype=torch.float32, device="cuda")
        sa.attn_partial_blocks(*to_dev(q, k, v), blocks, n_parts=2, o_rows=o_rows, causal=causal, out=out, lse=lse)
        torch.cuda.synchronize()
        written = torch.zeros((2, o_rows), dtype=torch.bool)
        for qr, kr, orow, qp, kp, sq, sk, part in blocks:
            o_ref, lse_ref = oracle.attention(q[:, :, qr:qr + sq].contiguous(), k[:, :, kr:kr + sk].contiguous(),
                                              v[:, :, kr:kr + sk].contiguous(), causal, q_off=qp, kv_off=kp)
            check_o(out[part, :, :, orow:orow + sq], o_ref, bf16_out=False)
            check_lse(lse[part, :, :, orow:orow + sq], lse_ref)
            written[part, orow:orow + sq] = True
        # rows no block writes keep their contents
        for part in range(2):
            free = (~written[part]).nonzero().flatten().tolist()
            if free:
                assert (out[part, :, :, free] == 7.0).all() and (lse[part, :, :, free] == 7.0).all()


def test_ring_grouped_launch_is_bitwise_the_per_chunk_launches(sa):
    q, k, v = to_dev(*workloads.make_qkv(adhoc(1, 4, 4, 2048, 128, True, seed=99)))
    o1, l1 = sa.ring_attn_fwd(q, k, v, P=4, causal=True)
    o2, l2 = sa.ring_attn_fwd(q, k, v, P=4, causal=True, grouped=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("D,Hq,Hkv", [(128, 8, 4), (64, 16, 8)])
def test_single_problem_head_chunks_cover_every_row(sa, D, Hq, Hkv):
    """At S = 32768 a single problem's items come in chunks of whole GQA groups
    whose K and V fit in 32 MB of L2 (two chunks in both cases), every chunk
    but the last padded with empty items to whole rounds of the grid. The same
    attention through the block-table launch (one block, items not chunked)
    must give bitwise the same fp32 partials and lse on every row; both
    outputs start as NaN, so a row that no item wrote fails. A few rows per
    head are also checked against the oracle."""
    S = 32768
    w = adhoc(1, Hq, Hkv, S, D, True, seed=91)
    q, k, v = workloads.make_qkv(w)
    qd, kd, vd = to_dev(q, k, v)
    nan = float("nan")
    o1 = torch.full((1, Hq, S, D), nan, device="cuda")
    l1 = torch.full((1, Hq, S), nan, device="cuda")
    sa.attn_partial(qd, kd, vd, 0, 0, True, out=o1, lse=l1)
    o2 = torch.full((1, 1, Hq, S, D), nan, device="cuda")
    l2 = torch.full((1, 1, Hq, S), nan, device="cuda")
    sa.attn_partial_blocks(qd, kd, vd, [(0, 0, 0, 0, 0, S, S, 0)], n_parts=1, causal=True, out=o2, lse=l2)
    torch.cuda.synchronize()
    sa.query_device_error()
    assert torch.equal(o1, o2[0]) and torch.equal(l1, l2[0])
    rows = workloads.sample_query_rows(w, n=4)
    o_ref, lse_ref = oracle.attention(q, k, v, True, rows=rows)
    check_o(gather_rows(o1, rows), o_ref, bf16_out=False)
    check_lse(gather_rows(l1, rows), lse_ref)


@pytest.mark.parametrize("D,Hq,Hkv,S,P,causal,skip_empty",
                         [(128, 8, 4, 16384, 8, True, False), (64, 6, 2, 13200, 66, True, False),
                          (128, 8, 4, 16384, 8, True, True), (128, 8, 4, 8192, 4, False, False)],
                         ids=["d128_8x2048", "d64_66x200", "d128_8x2048_skip", "d128_4x2048_noncausal"])
def test_shared_query_segments_match_block_table(sa, D, Hq, Hkv, S, P, causal, skip_empty):
    """Short key chunks that share all their query rows (one ring pass's
    blocks of a query chunk) run as the segments of each work item, Q loaded
    once (here chunks of 2048 keys, and 66 ragged chunks of 200 keys, split
    into launches of 64 and 2 segments). Each chunk's fp32 partial and lse must
    be bitwise those of the same block launched alone (the block-table
    kernel); all outputs start as NaN (as 7.0 with skip_empty, whose rows
    before a chunk's first key keep that value), so a row that no segment
    wrote fails. A few rows of the first and last chunks are also checked
    against the oracle."""
    C = S // P
    w = adhoc(1, Hq, Hkv, S, D, causal, seed=93)
    q, k, v = workloads.make_qkv(w)
    qd, kd, vd = to_dev(q, k, v)
    fill = 7.0 if skip_empty else float("nan")
    blocks = [(0, j * C, 0, 0, j * C, S, C, j) for j in range(P)]
    o1 = torch.full((P, 1, Hq, S, D), fill, device="cuda")
    l1 = torch.full((P, 1, Hq, S), fill, device="cuda")
    sa.attn_partial_blocks(qd, kd, vd, blocks, n_parts=P, causal=causal, out=o1, lse=l1, skip_empty=skip_empty)
    o2 = torch.full((P, 1, Hq, S, D), fill, device="cuda")
    l2 = torch.full((P, 1, Hq, S), fill, device="cuda")
    for b in blocks:
        sa.attn_partial_blocks(qd, kd, vd, [b], n_parts=P, causal=causal, out=o2, lse=l2, skip_empty=skip_empty)
    torch.cuda.synchronize()
    sa.query_device_error()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    if skip_empty:  # rows before each chunk's first key: O untouched, lse -inf
        for j in range(1, P):
            assert (o1[j, :, :, :j * C] == fill).all() and torch.isneginf(l1[j, :, :, :j * C]).all()
    del o2, l2
    rows = workloads.sample_query_rows(w, n=3)
    for j in (0, P - 1):
        o_ref, lse_ref = oracle.attention(q, k[:, :, j * C:(j + 1) * C].contiguous(),
                                          v[:, :, j * C:(j + 1) * C].contiguous(), causal, kv_off=j * C, rows=rows)
        check_lse(gather_rows(l1[j], rows), lse_ref)
        fin = ~np.isneginf(lse_ref)
        check_o(gather_rows(o1[j], rows).numpy()[fin], o_ref[fin], bf16_out=False)


@pytest.mark.parametrize("shape", [(1, 2, 2, 512, True), (1, 4, 2, 1008, True), (2, 2, 1, 384, False)],
                         ids=["s512c", "gqa_s1008c", "b2_s384"])
def test_attn_fwd_fp8_against_oracle(sa, shape):
    """e4m3 Q, K, V with power-of-two scales (so the dequantised inputs are exact
    bf16 and the oracle computes the exact attention of the quantised data);
    the kernel's only error beyond rounding is P in e4m3, held to the bound
    derived in fp8_bound plus 2^-8 |O| + 1e-4."""
    B, Hq, Hkv, S, causal = shape
    D = 128
    q, k, v = workloads.make_qkv(adhoc(B, Hq, Hkv, S, D, causal, seed=61))
    qs, ks, vs = 0.25, 0.5, 0.25
    q8, k8, v8 = (sa.quantize_e4m3(t, sc) for t, sc in ((q, qs), (k, ks), (v, vs)))
    qd, kd, vd = ((t.float() * sc).to(torch.bfloat16) for t, sc in ((q8, qs), (k8, ks), (v8, vs)))
    assert torch.equal(qd.float(), q8.float() * qs)  # exact: the dequantised inputs are bf16 values
    o_ref, lse_ref = oracle.attention(qd, kd, vd, causal)
    vt8 = v8.transpose(2, 3).contiguous()
    o, lse = sa.attn_fwd_fp8(q8.cuda(), k8.cuda(), vt8.cuda(), qs, ks, vs, causal=causal)
    torch.cuda.synchronize()
    check_lse(lse, lse_ref)
    err = np.abs(o.double().cpu().numpy() - o_ref)
    bound = fp8_bound(qd, kd, vd, causal, 1.0 / math.sqrt(D)) + 2.0 ** -8 * np.abs(o_ref) + 1e-4
    assert np.isfinite(o.float().cpu().numpy()).all()
    worst = float((err / bound).max())
    assert worst <= 1.0, f"fp8 error exceeds its bound by {worst:.2f}x"
    # rounding errors of many P elements partly cancel: the mean error sits well
    # below the mean of the worst-case bound (a layout or scale mistake would not)
    assert float(err.mean()) <= 0.25 * float(bound.mean())
    # and they are nearly unbiased: the least-squares slope of O on the oracle's,
    # per head and per column, stays within 2^-7 of 1, which a mis-folded scale
    # or a biased 1/l of a few percent would not
    head_dev, col_dev = fp8_slope_errors(o, o_ref)
    assert head_dev <= FP8_SLOPE_TOL and col_dev <= FP8_SLOPE_TOL, (head_dev, col_dev)


@pytest.mark.parametrize("shape", [(1, 2, 2, 256, True, 128), (1, 4, 2, 300, True, 128), (2, 2, 1, 200, False, 128),
                                   (1, 2, 2, 256, True, 64), (1, 4, 2, 300, True, 64), (2, 2, 1, 200, False, 64)],
                         ids=["s256c", "gqa_s300c", "b2_s200", "d64_s256c", "d64_gqa_s300c", "d64_b2_s200"])
def test_attn_bwd_against_oracle(sa, shape):
    """dQ, dK, dV (from the oracle's O and lse as the backward's inputs) against
    the oracle's exact gradients, each element within the bound derived in
    bwd_bound; head dims 128 and 64."""
    B, Hq, Hkv, S, causal, D = shape
    q, k, v = workloads.make_qkv(adhoc(B, Hq, Hkv, S, D, causal, seed=71))
    dout, _, _ = workloads.make_qkv(adhoc(B, Hq, Hq, S, D, causal, seed=72))
    qd, kd, vd, dod = to_dev(q, k, v, dout)
    # the forward's O and lse as the backward's inputs, from the oracle (O rounded to bf16)
    o_ref, lse_ref = oracle.attention(q, k, v, causal=causal)
    o_in = torch.from_numpy(o_ref).to(torch.bfloat16)
    o, lse = to_dev(o_in, torch.from_numpy(lse_ref).float())
    dq, dk, dv = sa.attn_bwd(qd, kd, vd, o, lse, dod, causal=causal)
    torch.cuda.synchronize()
    rq, rk, rv = oracle.attention_backward(q, k, v, dout, causal)
    bq, bk, bv = bwd_bound(q, k, v, dout, causal, 1.0 / math.sqrt(D), o_in)
    for name, got, ref, bnd in (("dq", dq, rq, bq), ("dk", dk, rk, bk), ("dv", dv, rv, bv)):
        worst = bwd_ratio(got, ref, bnd)
        assert worst <= 1.0, f"{name}: error exceeds its bound by {worst:.2f}x"


@pytest.mark.parametrize("P", [1, 4])
def test_ring_host_matches_device_ring(sa, P):
    """attn_ring_fwd_host (host buffers in and out) gives bitwise the device-side
    ring (one attn_partial per chunk, then lse_merge; P = 1: attn_fwd) and the
    oracle's values within the tolerance, from pinned or pageable inputs, and
    the same again from four calls queued on two alternating (stream,
    workspace) sets without waiting in between."""
    B, Hq, Hkv, S, D = 1, 4, 2, 512, 128
    q, k, v = workloads.make_qkv(adhoc(B, Hq, Hkv, S, D, True, seed=81))
    qp, kp, vp = (t.pin_memory() for t in (q, k, v))
    o_h, lse_h = sa.ring_attn_fwd_host(qp, kp, vp, P, causal=True)
    qd, kd, vd = to_dev(q, k, v)
    if P == 1:
        o_d, lse_d = sa.attn_fwd(qd, kd, vd, causal=True)
    else:
        o_d, lse_d = sa.ring_attn_fwd(qd, kd, vd, P=P, causal=True, grouped=False)
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(lse_h, lse_d.cpu())
    o_ref, lse_ref = oracle.attention(q, k, v, causal=True)
    check_o(o_h, o_ref)
    check_lse(lse_h, lse_ref)
    o2, l2 = sa.ring_attn_fwd_host(q, k, v, P, causal=True)  # pageable
    assert torch.equal(o2, o_h) and torch.equal(l2, lse_h)
    need = sa.ring_host_workspace_bytes(B, Hq, Hkv, S, D, P)
    sets = [(torch.cuda.Stream(), torch.empty(need, dtype=torch.uint8, device="cuda")) for _ in range(2)]
    outs = []
    for i in range(4):
        stream, ws = sets[i % 2]
        with torch.cuda.stream(stream):
            outs.append(sa.ring_attn_fwd_host(qp, kp, vp, P, causal=True, workspace=ws, synchronize=False))
    torch.cuda.synchronize()
    for o_i, l_i in outs:
        assert torch.equal(o_i, o_h) and torch.equal(l_i, lse_h)
    sa.query_device_error()


def test_ring_host_full_size_ring8(sa):
    """The host-buffer ring at the bench's default size: bitwise the device-side
    grouped ring (the partials of one launch per chunk and of one grouped launch
    are bitwise equal), and empty inputs return empty outputs."""
    w = workloads.WORKLOADS["ring8_b2h32s4096d128_causal"]
    q, k, v = workloads.make_qkv(w)
    o_h, lse_h = sa.ring_attn_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), w.P, causal=True)
    o_d, lse_d = sa.ring_attn_fwd(*to_dev(q, k, v), P=w.P, causal=True, grouped=True)
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(lse_h, lse_d.cpu())
    e = torch.empty((1, 2, 0, 128), dtype=torch.bfloat16)
    o_e, lse_e = sa.ring_attn_fwd_host(e, e, e, 4, causal=True)
    assert o_e.shape == (1, 2, 0, 128) and lse_e.shape == (1, 2, 0)
    sa.query_device_error()


def test_ring8_full_size_equals_single_pass(sa):
    """The ring-chunked workload at full size (B 2, H 32, S 4096, P 8 chunks of
    512), in the launch configuration the benchmark times (the 8 partials in
    one grouped launch, then lse_merge), against the single-pass attn_fwd on
    every element of every row: |dO| <= 1e-2, |dlse| <= 1e-3, no -inf. The
    oracle's side of the same workload is test_full_size_workload_sampled_rows."""
    w = workloads.WORKLOADS["ring8_b2h32s4096d128_causal"]
    qd, kd, vd = to_dev(*workloads.make_qkv(w))
    o_ring, lse_ring = sa.ring_attn_fwd(qd, kd, vd, P=w.P, causal=w.causal, grouped=True)
    o_one, lse_one = sa.attn_fwd(qd, kd, vd, causal=w.causal)
    torch.cuda.synchronize()
    sa.query_device_error()
    assert bool(torch.isfinite(lse_ring).all()) and bool(torch.isfinite(lse_one).all())
    assert bool(torch.isfinite(o_ring.float()).all())
    d_o = (o_ring.float() - o_one.float()).abs().max().item()
    d_l = (lse_ring - lse_one).abs().max().item()
    assert d_o <= O_TOL, d_o
    assert d_l <= LSE_TOL, d_l


def test_attn_bwd_full_size_gqa(sa):
    """The backward at the full size of the GQA workload, in the configuration
    bench.py --backward times (the GPU forward's O and lse as its inputs): on 8
    seeded query rows per head, the forward's O rows within the forward
    tolerance of the oracle's and dQ against the oracle's row-by-row dQ within
    the derived bound (delta's offset taken from those checked O rows, P's
    from the forward's lse on those rows); dV
    against the exact identity sum_j dV_j = sum over the group's query heads of
    sum_i dO_i (the rows of P sum to 1), within 2^-8 of the summed magnitudes;
    every gradient finite."""
    w = workloads.WORKLOADS["gqa_b1hq28hkv4s32768d128_causal"]
    q, k, v = workloads.make_qkv(w)
    dout = workloads.make_dout(w)
    qd, kd, vd, dod = to_dev(q, k, v, dout)
    o, lse = sa.attn_fwd(qd, kd, vd, causal=w.causal)
    dq, dk, dv = sa.attn_bwd(qd, kd, vd, o, lse, dod, causal=w.causal)
    torch.cuda.synchronize()
    sa.query_device_error()
    for t in (dq, dk, dv):
        assert bool(torch.isfinite(t).all())
    rows = workloads.sample_query_rows(w, n=8)
    pick = lambda t: torch.stack([t[b, h, torch.from_numpy(rows[b * w.Hq + h]).to(t.device)]
                                  for b in range(w.B) for h in range(w.Hq)])
    o_rows = pick(o).cpu()
    lse_rows = pick(lse).cpu()
    o_ref, lse_ref = oracle.attention(q, k, v, w.causal, rows=rows)
    check_o(o_rows.reshape(o_ref.shape), o_ref)
    check_lse(lse_rows.reshape(lse_ref.shape), lse_ref)
    ref = oracle.attention_backward_dq_rows(q, k, v, dout, w.causal, rows)
    bnd = bwd_dq_rows_bound(q, k, v, dout, w.causal, w.scale, rows, o_rows, lse_rows)
    got = pick(dq)
    worst = bwd_ratio(got, ref, bnd)
    assert worst <= 1.0, f"dQ rows: error exceeds the bound by {worst:.2f}x"
    g = w.Hq // w.Hkv
    dv_sum = dv.double().sum(dim=2).cpu().numpy()                                       # [B, Hkv, D]
    do_sum = dout.double().reshape(w.B, w.Hkv, g * w.S, w.D).sum(dim=2).numpy()
    tol = 2.0 ** -8 * (dout.double().abs().reshape(w.B, w.Hkv, g * w.S, w.D).sum(dim=2).numpy()
                       + dv.double().abs().sum(dim=2).cpu().numpy())
    assert (np.abs(dv_sum - do_sum) <= tol).all(), float((np.abs(dv_sum - do_sum) / tol).max())


# ----------------------------------------------------------------- full-size workloads

def run_workload(sa, w, q, k, v):
    """The launch configuration the benchmark times for this workload."""
    if w.varlen:
        cu = workloads.cu_seqlens(w)
        o, lse = sa.attn_fwd_varlen(q[0], k[0], v[0], cu, cu, causal=w.causal)
        return o[None], lse[None]
    if w.P == 1:
        return sa.attn_fwd(q, k, v, causal=w.causal)
    return sa.ring_attn_fwd(q, k, v, P=w.P, causal=w.causal, grouped=True)


@pytest.mark.parametrize("name", list(W))
def test_full_size_workload_sampled_rows(sa, name):
    w = W[name]
    q, k, v = workloads.make_qkv(w)
    if w.varlen:
        return check_varlen_workload(sa, w, q, k, v)
    rows = workloads.sample_query_rows(w, n=w.sample_rows or 32)
    # chunk boundaries and the last row are checked too
    extra = np.array(sorted({0, w.chunk - 1, w.chunk, w.S - 1} & set(range(w.S))), dtype=np.int64)
    rows = np.sort(np.concatenate([rows, np.tile(extra, (rows.shape[0], 1))], axis=1), axis=1)
    o_ref, lse_ref = oracle.attention(q, k, v, w.causal, rows=rows)
    qd, kd, vd = to_dev(q, k, v)
    del q, k, v
    o, lse = run_workload(sa, w, qd, kd, vd)
    check_o(gather_rows(o, rows), o_ref)
    check_lse(gather_rows(lse, rows), lse_ref)
    del o, lse, qd, kd, vd
    torch.cuda.empty_cache()


def check_varlen_workload(sa, w, q, k, v):
    """Sampled rows of a packed workload (the same for every head: 32 seeded
    rows plus each sequence's first and last row), each checked against the
    oracle on its own sequence."""
    cu = workloads.cu_seqlens(w)
    rng = np.random.default_rng(w.seed)
    rows = set(rng.choice(w.S, size=32, replace=False).tolist())
    rows |= {a for a in cu[:-1]} | {b - 1 for b in cu[1:]}
    rows = np.array(sorted(rows), dtype=np.int64)
    qd, kd, vd = to_dev(q, k, v)
    o, lse = run_workload(sa, w, qd, kd, vd)
    torch.cuda.synchronize()
    seq = np.searchsorted(np.array(cu), rows, side="right") - 1
    for s in np.unique(seq):
        a, b = cu[s], cu[s + 1]
        local = rows[seq == s] - a
        o_ref, lse_ref = oracle.attention(q[:, :, a:b].contiguous(), k[:, :, a:b].contiguous(),
                                          v[:, :, a:b].contiguous(), w.causal,
                                          rows=np.tile(local, (w.Hq, 1)))
        idx = torch.as_tensor(a + local, device=o.device)
        check_o(o[:, :, idx], o_ref)
        check_lse(lse[:, :, idx], lse_ref)
    del o, lse, qd, kd, vd
    torch.cuda.empty_cache()
