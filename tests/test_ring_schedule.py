"""Host logic of the emulated ring (no GPU): which blocks each device computes
at each hop, for the pages' contiguous layout and the load-balanced zigzag one.
The schedule is pinned to the oracle: chunk attention and merges following the
schedule reproduce the oracle's single-pass attention."""
import importlib.util
import os
import sys

import numpy as np
import pytest

import oracle
import workloads

_spec = importlib.util.spec_from_file_location(
    "ring_schedule", os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                                  "sequence_attn_fwd_gb300", "ring_schedule.py"))
rs = importlib.util.module_from_spec(_spec)
sys.modules[_spec.name] = rs  # dataclasses resolve annotations through the module table
_spec.loader.exec_module(rs)


@pytest.mark.parametrize("layout", rs.LAYOUTS)
@pytest.mark.parametrize("causal", [True, False])
def test_every_visible_block_exactly_once(layout, causal):
    for P in range(1, 10):
        nc = rs.n_chunks(P, layout)
        seen = [b for hop in rs.hop_blocks(P, layout, causal) for blocks in hop for b in blocks]
        want = {(q, k) for q in range(nc) for k in range(nc) if not causal or k <= q}
        assert sorted((b.q_chunk, b.kv_chunk) for b in seen) == sorted(want)


@pytest.mark.parametrize("layout", rs.LAYOUTS)
def test_devices_own_their_query_chunks_and_receive_kv_around_the_ring(layout):
    for P in range(1, 10):
        chunks = rs.device_chunks(P, layout)
        assert sorted(c for dc in chunks for c in dc) == list(range(rs.n_chunks(P, layout)))
        for t, hop in enumerate(rs.hop_blocks(P, layout, causal=False)):
            for d, blocks in enumerate(hop):
                assert {b.q_chunk for b in blocks} == set(chunks[d])
                assert {b.kv_chunk for b in blocks} == set(chunks[(d - t) % P])


def test_zigzag_balances_causal_work_and_contiguous_does_not():
    for P in range(2, 10):
        zz = rs.hop_work(P, "zigzag")
        assert all(w == 2.0 for hop in zz for w in hop)  # two chunk pairs per device per hop
        ct = rs.hop_work(P, "contiguous")
        assert ct[0] == [0.5] * P
        for t in range(1, P):
            assert ct[t] == [1.0 if d >= t else 0.0 for d in range(P)]
        # ring time in full contiguous-chunk pairs: P - 1/2 against the balanced P / 2
        assert rs.ring_time_units(P, "contiguous") == P - 0.5
        assert rs.ring_time_units(P, "zigzag") == P / 2
        total = sum(b.work for hop in rs.hop_blocks(P, "contiguous") for bl in hop for b in bl)
        assert total == P * P / 2  # the causal triangle, in contiguous chunk pairs


def test_bad_arguments():
    with pytest.raises(ValueError):
        rs.n_chunks(4, "striped")
    with pytest.raises(ValueError):
        rs.n_chunks(0, "zigzag")


@pytest.mark.parametrize("layout", rs.LAYOUTS)
def test_schedule_with_oracle_blocks_equals_single_pass(layout):
    """Follow the schedule with the oracle: per block the oracle's chunk
    attention at global offsets, per query chunk the oracle's merge of its
    blocks in hop order; the result is the single-pass attention."""
    P, B, Hq, Hkv, S, D = 3, 1, 4, 2, 96, 32
    w = workloads.Workload("sched", B, Hq, Hkv, S, D, True, 1, 4242)
    q, k, v = workloads.make_qkv(w)
    o_ref, lse_ref = oracle.attention(q, k, v, True)
    C = S // rs.n_chunks(P, layout)
    parts = {}
    for hop in rs.hop_blocks(P, layout):
        for blocks in hop:
            for b in blocks:
                qs, ks = slice(b.q_chunk * C, (b.q_chunk + 1) * C), slice(b.kv_chunk * C, (b.kv_chunk + 1) * C)
                o, l = oracle.attention(q[:, :, qs].contiguous(), k[:, :, ks].contiguous(),
                                        v[:, :, ks].contiguous(), True, q_off=b.q_chunk * C,
                                        kv_off=b.kv_chunk * C)
                parts.setdefault(b.q_chunk, []).append((o, l))
    for qc, pl in parts.items():
        o, l = oracle.lse_merge(np.stack([p[0] for p in pl]), np.stack([p[1] for p in pl]))
        np.testing.assert_allclose(o, o_ref[:, :, qc * C:(qc + 1) * C], rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, lse_ref[:, :, qc * C:(qc + 1) * C], rtol=0, atol=1e-12)
