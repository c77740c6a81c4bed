"""Host logic of bench.py, on the CPU: the replica path's max-over-ranks timing
with two gloo ranks, the algorithmic counts the roofline uses, the clock summary
and the peak-file loader."""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads


def _rank_main(rank, world, port, values, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(values[rank])
        with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
            json.dump(got, f)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks(tmp_path):
    import random

    port = 29500 + random.randint(0, 2000)
    values = [3.5, 7.25]
    mp.start_processes(_rank_main, args=(2, port, values, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        assert json.load(open(tmp_path / f"r{r}.json")) == 7.25


def test_max_over_ranks_single_process_is_identity():
    assert bench.max_over_ranks(1.5) == 1.5


def test_visible_pairs_matches_brute_force():
    for S_q, q_off, kv_len, kv_off, causal in [(37, 0, 37, 0, True), (50, 10, 20, 25, True), (9, 0, 13, 0, False),
                                               (64, 0, 16, 48, True), (16, 0, 16, 40, True)]:
        brute = sum(1 for r in range(S_q) for j in range(kv_len)
                    if not causal or kv_off + j <= q_off + r)
        assert bench.visible_pairs(S_q, q_off, kv_len, kv_off, causal) == brute


def test_causal_flops_count_equals_chunked_visible_pairs():
    """F = 4 B Hq S^2 D / 2 is the convention; the exact visible pairs add the diagonal."""
    w = workloads.WORKLOADS["ring8_b2h32s4096d128_causal"]
    pairs = sum(bench.visible_pairs(w.S, 0, w.chunk, j * w.chunk, True) for j in range(w.P))
    assert pairs == w.S * (w.S + 1) // 2
    assert math.isclose(w.attention_flops(), 4.0 * w.B * w.Hq * w.D * w.S * w.S / 2)


def test_merge_algorithmic_bytes_ring8():
    w = workloads.WORKLOADS["ring8_b2h32s4096d128_causal"]
    rows = w.B * w.Hq * w.S
    finite_rows = sum(w.B * w.Hq * (w.S - c * w.chunk) for c in range(w.P))
    assert finite_rows * 64 == w.P * rows * 36  # 36/64 of the P dense partials' rows are finite
    expected = w.P * rows * 4 + finite_rows * w.D * 4 + rows * w.D * 2 + rows * 4
    assert bench.merge_algorithmic_bytes(w) == expected
    assert abs(expected - 0.6805e9) < 1e6


def test_summarise_clocks():
    lines = ["0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active",
             "0, 1980, 2070, 1390.0, 0x4, Not Active, Not Active, Not Active, Active",
             "0, 2070, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active",
             "garbage line"]
    s = bench.summarise_clocks(lines)
    assert s == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    assert bench.summarise_clocks([])["samples"] == 0


def test_load_peaks(tmp_path):
    peaks, src = bench.load_peaks(str(tmp_path / "missing.json"))
    assert src == "fallback" and peaks["bf16_tflops"] == 1900.0 and peaks["hbm_gbs"] == 6800.0
    p = tmp_path / "peaks.json"
    p.write_text(json.dumps({"hbm_gbs": 7000.5, "bf16_tflops": {"value": 2000.0}}))
    peaks, src = bench.load_peaks(str(p))
    assert src == "measured" and peaks == {"hbm_gbs": 7000.5, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 2000.0}


def test_workload_sizes_match_the_stated_configurations():
    W = workloads.WORKLOADS
    assert [(w.B, w.Hq, w.Hkv, w.S, w.D, w.causal, w.P) for w in W.values()] == [
        (1, 2, 2, 256, 64, False, 1), (2, 32, 32, 4096, 128, True, 8), (1, 28, 4, 32768, 128, True, 1),
        (2, 32, 32, 8192, 128, True, 16), (1, 32, 8, 131072, 128, True, 16), (1, 32, 8, 65536, 128, True, 1),
        (1, 32, 8, 32768, 128, True, 4), (1, 32, 8, 32768, 128, True, 16)]
    # the reduced forms of the 131K ring keep its heads and, respectively, its
    # key-chunk length and its part count
    big = W["ring16_b1hq32hkv8s131072d128_causal"]
    assert W["ring4_b1hq32hkv8s32768d128_causal"].chunk == big.chunk
    assert W["ring16_b1hq32hkv8s32768d128_causal"].P == big.P
    v = W["varlen_hq32hkv8t65536d128_causal"]
    lens = workloads.seq_lens(v)
    assert lens.sum() == v.S and lens.min() >= 1 and lens[:-1].min() >= 128 and lens.max() <= 8192
    assert len(lens) > 20 and np.array_equal(lens, workloads.seq_lens(v))  # seeded
    cu = workloads.cu_seqlens(v)
    assert cu[0] == 0 and cu[-1] == v.S and len(cu) == len(lens) + 1
    assert math.isclose(v.attention_flops(), 2.0 * 32 * 128 * float((lens.astype(float) ** 2).sum()))
    w = W["gqa_b1hq28hkv4s32768d128_causal"]
    pos = workloads.boost_positions(w)
    assert len(pos) == 327 and len(np.unique(pos)) == 327
    rows = workloads.sample_query_rows(W["ring16_b1hq32hkv8s131072d128_causal"])
    assert rows.shape == (32, 64) and all(len(np.unique(r)) == 64 for r in rows)


def test_measured_traffic_follows_the_kernel_sources(tmp_path):
    digest = bench.sources_digest("lse_merge")
    (tmp_path / "x.md").write_text(
        "text\n```\ntraffic lse_merge wl bytes_per_launch=123 sources=%s\n"
        "traffic lse_merge other bytes_per_launch=9 sources=0000000000000000\n```\n" % digest)
    assert bench.measured_traffic("lse_merge", "wl", str(tmp_path)) == 123
    assert bench.measured_traffic("lse_merge", "other", str(tmp_path)) is None  # stale capture
    assert bench.measured_traffic("attn_partial", "wl", str(tmp_path)) is None


def test_code_text_ignores_comments_only():
    a = "int x = 1; // one\n/* block\n comment */ int y =  2;\n"
    b = "int x = 1;\n int y = 2; // two\n"
    assert bench.code_text(a) == bench.code_text(b) == "int x = 1; int y = 2;"
    assert bench.code_text("int x = 1;") != bench.code_text("int x = 2;")


def test_ring_time_from_hops():
    r = bench.ring_time_from_hops([[1.0, 3.0], [2.0, 2.0]])
    assert r["ring_ms"] == 5.0 and r["device_ms_total"] == 8.0
    assert r["hop_spread_max_over_mean"] == [1.5, 1.0]
    assert r["balance"] == 0.8


def test_dout_is_seeded_and_independent_of_qkv():
    w = workloads.WORKLOADS["gqa_b1hq28hkv4s32768d128_causal"]
    d1 = workloads.make_dout(w, S=64)
    d2 = workloads.make_dout(w, S=64)
    q, _, _ = workloads.make_qkv(w, S=64)
    assert d1.shape == (w.B, w.Hq, 64, w.D) and d1.dtype == torch.bfloat16
    assert torch.equal(d1, d2) and not torch.equal(d1, q)
    assert abs(float(d1.float().std()) - 1.0) < 0.05


def test_backward_sample_counts_two_and_a_half_forward_flops():
    """The oracle backward sample's FLOPs: 2.5 x 4 D per visible pair of the prefix."""
    w = workloads.WORKLOADS["gqa_b1hq28hkv4s32768d128_causal"]
    rate, secs, calls, _ = bench.oracle_backward_sample(w, 0.0, prefix=32)
    assert calls == 1
    assert rate * 1e12 * secs == pytest.approx(2.5 * 4 * w.D * 32 * 33 / 2, rel=1e-9)


def test_seq_len_override_is_backward_only():
    """--seq-len (a small case of a workload's backward for profiling) is refused
    for the forward and for ring workloads."""
    for argv in (["--seq-len", "4096"],
                 ["--seq-len", "4096", "--backward", "--workload", "ring8_b2h32s4096d128_causal"],
                 ["--seq-len", "0", "--backward", "--workload", "gqa_b1hq28hkv4s32768d128_causal"]):
        with pytest.raises(SystemExit):
            bench.main(argv)
