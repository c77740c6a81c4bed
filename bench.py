"""Benchmark: blockwise attention forward + log-sum-exp merge on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole path over one batch of the workload: for a
ring-chunked workload, the P key chunks' partials (by default one
attn_partial_blocks launch over all P chunks, --partials per-chunk for one
attn_partial launch per chunk; zero-copy views either way) and one lse_merge;
for a single-pass workload, one attn_fwd. The
default workload is the largest one that fits one GPU: ring-chunked causal
attention at 131,072 tokens, B=1, Hq=32, Hkv=8, D=128, with P=16 key chunks
of 8192 (about 37 GB of inputs, partials and outputs on the device). The
other workloads are reachable with --workload.

metric: causal-adjusted attention TFLOP/s, F = 4*B*Hq*S^2*D (halved when
causal), over the step time; the JSON line also carries the dominant
kernel's roofline, the merge's GB/s, an end-to-end figure through the C ABI
with host buffers, and the fp64 oracle timed on the host cores.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (there is no other implementation of this path to run).

Under torchrun (N > 1) every rank runs an independent replica (the path
needs no exchange when chunks are emulated on one GPU); value = total FLOPs
of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "attention fwd TFLOP/s (causal-adjusted) & % BF16 peak; lse_merge GB/s & % HBM"
METRIC_BWD = "attention bwd TFLOP/s (causal-adjusted, 2.5x the forward's FLOPs) & % BF16 peak"
DEFAULT_WORKLOAD = "ring16_b1hq32hkv8s131072d128_causal"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# A step this long keeps the GPU at its power cap the way the sustained GEMM
# loop of the peaks does: its kernels are held to the sustained peak.
LONG_STEP_MS = 50.0
L2_BYTES = 129e6


# ----------------------------------------------------------------- helpers (host logic, unit-tested on CPU)

def load_peaks(path: str = os.path.join(ROOT, "MEASURED_PEAKS.json")):
    """(peaks, source) from the measured file when present, else the fallback figures."""
    try:
        with open(path) as f:
            raw = json.load(f)
        peaks = {}
        for key in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
            val = raw.get(key)
            if isinstance(val, dict):
                val = val.get("value")
            if isinstance(val, (int, float)) and val > 0:
                peaks[key] = float(val)
        if "hbm_gbs" in peaks and "bf16_tflops" in peaks:
            peaks.setdefault("bf16_tflops_sustained", peaks["bf16_tflops"])
            return peaks, "measured"
    except (OSError, ValueError):
        pass
    return dict(FALLBACK_PEAKS), "fallback"


def measure_e4m3_gemm_tflops(n: int = 8192, iters: int = 20):
    """Dense e4m3 GEMM throughput of the vendor library (cuBLASLt through
    torch._scaled_mm: e4m3 operands, unit per-tensor scales, bf16 output),
    n x n x n, timed as a burst of back-to-back products after a warm-up, like
    the measured bf16 peak. The e4m3 forward's roofline denominator; None if
    the GEMM is unavailable (the caller then takes the measured bf16 peak times
    the nominal e4m3 / bf16 ratio)."""
    try:
        a = torch.randn(n, n, device="cuda").to(torch.float8_e4m3fn)
        b = torch.randn(n, n, device="cuda").to(torch.float8_e4m3fn).t()  # column-major operand
        one = torch.ones((), device="cuda", dtype=torch.float32)

        def gemm():
            return torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

        for _ in range(5):
            gemm()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(iters):
            gemm()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / iters
        return 2.0 * n ** 3 / (ms * 1e-3) / 1e12
    except Exception:  # no e4m3 GEMM in this build: the nominal ratio stands in
        return None


def visible_pairs(S_q: int, q_off: int, kv_len: int, kv_off: int, causal: bool) -> int:
    """Number of (query, key) pairs a chunk's attention visits exactly."""
    if not causal:
        return S_q * kv_len
    total = 0
    # row r sees keys j < kv_len with kv_off + j <= q_off + r
    r = np.arange(S_q, dtype=np.int64)
    n = np.clip(q_off + r - kv_off + 1, 0, kv_len)
    total = int(n.sum())
    return total


def merge_algorithmic_bytes(w: workloads.Workload, out_bytes: int = 2) -> int:
    """Bytes the merge must move: every lse_i, the O_i rows with finite lse_i,
    the merged O and lse."""
    rows = w.B * w.Hq * w.S
    finite_rows = 0
    C = w.chunk
    for c in range(w.P):
        finite_rows += w.B * w.Hq * (w.S - c * C if w.causal else w.S)
    return w.P * rows * 4 + finite_rows * w.D * 4 + rows * w.D * out_bytes + rows * 4


# The kernels' sources and the C-ABI layer that sets up their launches (the
# tables, item order and grid decide the traffic as much as the kernel code).
_FWD_SOURCES = ["attn_kernel.cu", "attn_common.cuh", "ptx.cuh", "kernels.h", "api.cu"]
KERNEL_SOURCES = {
    "attn_bwd": ["attn_kernel.cu", "attn_bwd.cuh", "ptx.cuh", "kernels.h", "api.cu"],
    "attn_partial": _FWD_SOURCES,
    "attn_partial_blocks": _FWD_SOURCES,
    "attn_fwd_varlen": _FWD_SOURCES,
    "attn_fwd_fp8": _FWD_SOURCES,
    "attn_fwd": _FWD_SOURCES,
    "lse_merge": ["lse_merge.cu", "kernels.h", "api.cu"],
}


def code_text(source: str) -> str:
    """C/CUDA source without comments and with runs of whitespace collapsed,
    so that an edit to comments alone leaves a kernel's digest unchanged (the
    sources hold no string literal with comment markers in it)."""
    import re

    source = re.sub(r"/\*.*?\*/", " ", source, flags=re.S)
    source = re.sub(r"//[^\n]*", " ", source)
    return " ".join(source.split())


def sources_digest(kernel: str) -> str:
    """SHA-256 prefix of the code (comments left out) of the sources a kernel
    is built from."""
    import hashlib

    m = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "sequence_attn_fwd_gb300", "csrc", f), encoding="utf-8") as fh:
            m.update(code_text(fh.read()).encode("utf-8"))
    return m.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str, profiles_dir: str = os.path.join(ROOT, "profiles")):
    """DRAM bytes per launch from a committed ncu summary (a line
    `traffic <kernel> <workload> bytes_per_launch=<n> sources=<digest>`), or None
    when there is none or the kernel's sources changed since it was captured."""
    import glob
    import re

    digest = sources_digest(kernel)
    pat = re.compile(r"^traffic (\S+) (\S+) bytes_per_launch=(\d+) sources=([0-9a-f]+)\s*$")
    for path in sorted(glob.glob(os.path.join(profiles_dir, "*.md"))):
        with open(path) as f:
            for line in f:
                m = pat.match(line.strip())
                if m and m.group(1) == kernel and m.group(2) == workload and m.group(4) == digest:
                    return int(m.group(3))
    return None


def ring_time_from_hops(hop_ms) -> dict:
    """Emulated ring timing from per-(hop, device) times hop_ms[t][d]: a hop
    lasts as long as its slowest device; spread = slowest / mean device."""
    ring = sum(max(row) for row in hop_ms)
    busy = sum(sum(row) for row in hop_ms)
    spread = [max(row) / (sum(row) / len(row)) if sum(row) > 0 else 1.0 for row in hop_ms]
    return {"ring_ms": ring, "device_ms_total": busy, "hop_spread_max_over_mean": spread,
            "balance": busy / (len(hop_ms[0]) * ring) if ring > 0 else 1.0}


def max_over_ranks(value: float) -> float:
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        t = torch.tensor([value], dtype=torch.float64,
                         device="cuda" if dist.get_backend() == "nccl" else "cpu")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return value


def summarise_clocks(lines):
    """Median SM clock, max clock and the throttle reasons seen in nvidia-smi CSV lines."""
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            mx.append(float(parts[2]))
        except ValueError:
            continue
        for name, flag in zip(names, parts[5:9]):
            if flag.lower() == "active":
                reasons.add(name)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
            "samples": len(sm)}


class ClockSampler:
    """nvidia-smi polled every 200 ms while the GPU works; read-only."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-i", str(index), "-lms", "200"], stdout=self.file,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        lines = self.file.read().splitlines()
        self.file.close()
        os.unlink(self.file.name)
        return summarise_clocks(lines)


# ----------------------------------------------------------------- the GPU arm

def run_ours(args, w: workloads.Workload, rank: int, world: int):
    import sequence_attn_fwd_gb300 as sa

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    q_h, k_h, v_h = workloads.make_qkv(w)
    inputs = (q_h, k_h, v_h)  # the bf16 inputs, kept for the oracle's timed sample
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    B, Hq, S, D, P, C = w.B, w.Hq, w.S, w.D, w.P, w.chunk
    o = torch.empty((B, Hq, S, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=dev)
    o_parts = lse_parts = None
    if P > 1:
        o_parts = torch.empty((P, B, Hq, S, D), dtype=torch.float32, device=dev)
        lse_parts = torch.empty((P, B, Hq, S), dtype=torch.float32, device=dev)
    fp8 = args.dtype == "e4m3"
    if fp8:  # inputs on the e4m3 grid with power-of-two per-tensor scales (untimed preparation)
        if w.varlen or P > 1 or D != 128:
            raise SystemExit("--dtype e4m3 runs single-pass head-dim-128 workloads")
        sc = [2.0 ** math.ceil(math.log2(float(t.abs().max()) / 448.0)) for t in (q_h, k_h, v_h)]
        # the step's inputs become the e4m3 tensors (V transposed), on the device and the host
        q, k, v = (sa.quantize_e4m3(q, sc[0]), sa.quantize_e4m3(k, sc[1]),
                   sa.quantize_e4m3(v, sc[2]).transpose(2, 3).contiguous())
        q_h, k_h, v_h = q.cpu(), k.cpu(), v.cpu()
    grouped = P > 1 and args.partials == "grouped"
    cu = workloads.cu_seqlens(w) if w.varlen else None
    launches_per_step = (2 if grouped else P + 1) if P > 1 else 1
    chunk_blocks = [(0, j * C, 0, 0, j * C, S, C, j) for j in range(P)]

    def step(qq, kk, vv, ev=None, oo=None, ll=None):
        oo = o if oo is None else oo
        ll = lse if ll is None else ll
        if fp8:  # qq, kk, vv: e4m3 Q, K and V^T
            if ev:
                ev[0].record(stream)
            sa.attn_fwd_fp8(qq, kk, vv, sc[0], sc[1], sc[2], causal=w.causal, out=oo, lse=ll)
            if ev:
                ev[1].record(stream)
            return
        if w.varlen:  # packed sequences: [Hq, total, D] views of the B = 1 tensors
            if ev:
                ev[0].record(stream)
            sa.attn_fwd_varlen(qq[0], kk[0], vv[0], cu, cu, causal=w.causal, out=oo[0], lse=ll[0])
            if ev:
                ev[1].record(stream)
            return
        if P == 1:
            if ev:
                ev[0].record(stream)
            sa.attn_fwd(qq, kk, vv, causal=w.causal, out=oo, lse=ll)
            if ev:
                ev[1].record(stream)
            return
        if ev:
            ev[0].record(stream)
        if grouped:  # the P chunks' partials in one persistent launch
            sa.attn_partial_blocks(qq, kk, vv, chunk_blocks, n_parts=P, causal=w.causal, out=o_parts,
                                   lse=lse_parts, skip_empty=True)
        else:
            for j in range(P):
                sa.attn_partial(qq, kk[:, :, j * C:(j + 1) * C], vv[:, :, j * C:(j + 1) * C], 0, j * C,
                                w.causal, out=o_parts[j], lse=lse_parts[j], skip_empty=True)
        if ev:
            ev[1].record(stream)
        sa.lse_merge(o_parts, lse_parts, torch.bfloat16, out=o, lse=lse)
        if ev:
            ev[2].record(stream)

    F = w.attention_flops()
    sampler = ClockSampler(dev.index) if rank == 0 else None
    # warm-up: at least W steps and --warmup-seconds of work so clocks settle
    t_end = time.time() + args.warmup_seconds
    n = 0
    while n < args.warmup or time.time() < t_end:
        step(q, k, v)
        n += 1
        if n % 8 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        step(q, k, v, evs[i])
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    sa.query_device_error(dev)
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1))
    ms_per_step = elapsed_ms / args.steps
    attn_ms = [e[0].elapsed_time(e[1]) for e in evs]
    merge_ms = [e[1].elapsed_time(e[2]) for e in evs] if P > 1 else []
    value = world * F * args.steps / (elapsed_ms * 1e-3) / 1e12

    # end to end through the public API: pinned host inputs in, host result out
    e2e = None
    if rank == 0 and not args.no_e2e and not fp8 and not w.varlen:
        e2e = e2e_host_ring(sa, w, dev, stream, q_h, k_h, v_h, F, args.steps)
    elif rank == 0 and not args.no_e2e:  # fp8 and varlen: torch copies around the device step
        q_p, k_p, v_p = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
        sets = [{"stream": torch.cuda.Stream(dev), "in": [torch.empty_like(t) for t in (q, k, v)],
                 "out": [torch.empty_like(o), torch.empty_like(lse)],
                 "host": [torch.empty(o.shape, dtype=o.dtype).pin_memory(),
                          torch.empty(lse.shape, dtype=lse.dtype).pin_memory()]} for _ in range(2)]

        def e2e_step(st_):
            with torch.cuda.stream(st_["stream"]):
                for d_, h_ in zip(st_["in"], (q_p, k_p, v_p)):
                    d_.copy_(h_, non_blocking=True)
                step(*st_["in"], oo=st_["out"][0], ll=st_["out"][1])
                for h_, d_ in zip(st_["host"], st_["out"]):
                    h_.copy_(d_, non_blocking=True)

        e2e_ms = overlapped_steps_ms(dev, stream, sets, e2e_step, args.steps)
        h2d = sum(t.numel() * t.element_size() for t in (q_h, k_h, v_h))
        d2h = o.numel() * o.element_size() + lse.numel() * lse.element_size()
        e2e = {"value": F / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "path": ("torch copies of the inputs and outputs around the device-side step; two (stream, "
                        "buffers) sets alternate across steps")}
        del sets

    peaks, peak_src = load_peaks()
    n_attn = P if P > 1 and not grouped else 1  # attention launches per step
    attn_avg_ms = statistics.mean(attn_ms) / n_attn  # per launch
    flops_per_launch = F / n_attn
    achieved = flops_per_launch / (attn_avg_ms * 1e-3) / 1e12
    entry = "attn_partial_blocks" if grouped else ("attn_partial" if P > 1 else
                                                   ("attn_fwd_varlen" if w.varlen else
                                                    ("attn_fwd_fp8" if fp8 else "attn_fwd")))
    what = {"attn_partial_blocks": f"<f32 out> (attn_partial_blocks: the {P} key chunks in one launch)",
            "attn_partial": "<f32 out> (attn_partial)", "attn_fwd": "<bf16 out>",
            "attn_fwd_varlen": f"<bf16 out> (attn_fwd_varlen: {len(cu) - 1 if cu else 0} packed sequences)",
            "attn_fwd_fp8": "<bf16 out, e4m3 Q/K/V/P> (attn_fwd_fp8)"}[entry]
    # The burst peak for a kernel timed alone; the sustained one (a seconds-long
    # GEMM loop under the power cap) for a kernel inside a long step, here the
    # partials launch of a step of LONG_STEP_MS or more, which runs as long as
    # that loop does. e4m3 MMAs: an e4m3 GEMM burst measured here, else the
    # measured bf16 peak times the nominal e4m3 / bf16 ratio (4.5 / 2.25).
    sustained = ms_per_step >= LONG_STEP_MS
    bf16_peak = peaks["bf16_tflops_sustained"] if sustained else peaks["bf16_tflops"]
    peak = bf16_peak * (2.0 if fp8 else 1.0)
    source = (f"{peak_src} bf16 sustained (a {ms_per_step:.0f} ms step)" if sustained
              else f"{peak_src} bf16 burst") + (" x 2 (nominal e4m3 / bf16 ratio)" if fp8 else "")
    nominal_fp8_peak = peak
    e4m3_gemm = measure_e4m3_gemm_tflops() if fp8 else None
    if e4m3_gemm is not None:
        peak = e4m3_gemm
        source = "measured here: e4m3 GEMM burst (cuBLASLt through torch._scaled_mm, 8192^3, bf16 out)"
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "traffic": measured_traffic(entry, w.name),
                "kernel": f"attn_fwd_kernel<{D}>" + what,
                "peak_source": source,
                "frac_of_burst": achieved / (peaks["bf16_tflops"] * (2.0 if fp8 else 1.0)),
                "launch_ms": attn_avg_ms}
    if fp8:
        roofline["frac_of_nominal_e4m3"] = achieved / nominal_fp8_peak
    merge = None
    if merge_ms:
        mb = merge_algorithmic_bytes(w)
        mms = statistics.mean(merge_ms)
        gbs = mb / (mms * 1e-3) / 1e9
        merge = {"achieved": gbs, "unit": "GB/s", "peak": peaks["hbm_gbs"], "frac": gbs / peaks["hbm_gbs"],
                 "launch_ms": mms, "algorithmic_bytes": mb, "peak_source": f"{peak_src} copy",
                 "traffic": measured_traffic("lse_merge", w.name)}
    return {
        "value": value, "ms_per_step": ms_per_step, "e2e": e2e, "roofline": roofline, "merge": merge,
        "gpu_launches": args.steps * launches_per_step, "clocks": clocks,
        "attn_ms_per_step": statistics.mean(attn_ms), "inputs": inputs,
    }


def overlapped_steps_ms(dev, stream, sets, run, steps: int) -> float:
    """Milliseconds per end-to-end step with two sets of buffers, each with its
    own stream (set["stream"]), used alternately so that one step's copies
    overlap its neighbours' compute: run(set) queues a whole step (uploads,
    compute, downloads) on set["stream"]. Timed from an event before the first
    step to one after both streams' last step."""
    for i in range(4):
        run(sets[i % 2])
    torch.cuda.synchronize(dev)
    n = max(4, min(steps, 20))
    a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for s_ in sets:
        s_["stream"].wait_stream(stream)
    for i in range(n):
        run(sets[i % 2])
    for s_ in sets:
        stream.wait_stream(s_["stream"])
    b_.record(stream)
    torch.cuda.synchronize(dev)
    return a.elapsed_time(b_) / n


def e2e_host_ring(sa, w: workloads.Workload, dev, stream, q_h, k_h, v_h, F: float, steps: int) -> dict:
    """The step end to end through the C ABI's host-buffer entry point
    (attn_ring_fwd_host): pinned host Q, K, V in, host O and lse out, every
    step. Two (stream, workspace, output) sets alternate, so one step's uploads
    overlap the previous step's compute and downloads; the timed region runs
    from an event before the first step to one after every stream's last."""
    qp, kp, vp = (t.pin_memory() for t in (q_h, k_h, v_h))
    B, Hq, S, D, P = w.B, w.Hq, w.S, w.D, w.P
    need = sa.ring_host_workspace_bytes(B, Hq, w.Hkv, S, D, P)
    sets = [{"stream": torch.cuda.Stream(dev), "ws": torch.empty(need, dtype=torch.uint8, device=dev),
             "o": torch.empty(q_h.shape, dtype=torch.bfloat16).pin_memory(),
             "lse": torch.empty((B, Hq, S), dtype=torch.float32).pin_memory()} for _ in range(2)]

    def host_step(st_):
        with torch.cuda.stream(st_["stream"]):
            sa.ring_attn_fwd_host(qp, kp, vp, P, causal=w.causal, out=st_["o"], lse=st_["lse"],
                                  workspace=st_["ws"], device=dev, synchronize=False)

    ms = overlapped_steps_ms(dev, stream, sets, host_step, steps)
    return {"value": F / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": ms,
            "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in (q_h, k_h, v_h)),
            "d2h_bytes_per_step": sets[0]["o"].numel() * 2 + sets[0]["lse"].numel() * 4,
            "path": ("attn_ring_fwd_host (C ABI, host buffers): Q and each K/V chunk uploaded on the library's "
                     "copy stream while earlier chunks' partials run (one attn_partial per chunk), merge, O and "
                     "lse downloaded; two (stream, workspace) sets alternate across steps")}


def run_ours_backward(args, w: workloads.Workload, rank: int, world: int):
    """The backward step: one attn_bwd call (delta pre-pass, dK/dV kernel, dQ
    kernel) from the forward's O and lse, for a seeded dO. FLOPs counted as
    2.5x the forward's (the five products of the backward: S, dP, dV, dK, dQ;
    the kernels recompute S and dP once more for dQ, which is not counted)."""
    import sequence_attn_fwd_gb300 as sa

    if w.P > 1 or w.varlen or w.D != 128 or args.dtype != "bf16":
        raise SystemExit("--backward runs single-pass head-dim-128 bf16 workloads")
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    q_h, k_h, v_h = workloads.make_qkv(w)
    do_h = workloads.make_dout(w)
    q, k, v, do = q_h.to(dev), k_h.to(dev), v_h.to(dev), do_h.to(dev)
    o, lse = sa.attn_fwd(q, k, v, causal=w.causal)  # untimed: the backward's inputs
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    delta = torch.empty_like(lse)

    def step(qq, kk, vv, oo, ll, dd, grads=None):
        g_ = grads or (dq, dk, dv, delta)
        sa.attn_bwd(qq, kk, vv, oo, ll, dd, causal=w.causal, dq=g_[0], dk=g_[1], dv=g_[2], delta=g_[3])

    F = 2.5 * w.attention_flops()
    sampler = ClockSampler(dev.index) if rank == 0 else None
    t_end = time.time() + args.warmup_seconds
    n = 0
    while n < args.warmup or time.time() < t_end:
        step(q, k, v, o, lse, do)
        n += 1
        if n % 8 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        evs[i][0].record(stream)
        step(q, k, v, o, lse, do)
        evs[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop() if sampler else None
    sa.query_device_error(dev)
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1))
    call_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    value = world * F * args.steps / (elapsed_ms * 1e-3) / 1e12

    e2e = None
    if rank == 0 and not args.no_e2e:  # pinned host Q, K, V, O, lse, dO in; dQ, dK, dV out
        ins_h = [t.pin_memory() for t in (q_h, k_h, v_h, o.cpu(), lse.cpu(), do_h)]
        sets = [{"stream": torch.cuda.Stream(dev), "in": [torch.empty_like(t, device=dev) for t in ins_h],
                 "grads": [torch.empty_like(t) for t in (dq, dk, dv, delta)],
                 "host": [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (dq, dk, dv)]}
                for _ in range(2)]

        def e2e_step(st_):
            with torch.cuda.stream(st_["stream"]):
                for d_, h_ in zip(st_["in"], ins_h):
                    d_.copy_(h_, non_blocking=True)
                step(*st_["in"], grads=st_["grads"])
                for h_, d_ in zip(st_["host"], st_["grads"][:3]):
                    h_.copy_(d_, non_blocking=True)

        e2e_ms = overlapped_steps_ms(dev, stream, sets, e2e_step, args.steps)
        e2e = {"value": F / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in ins_h),
               "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in sets[0]["host"]),
               "path": ("torch copies around attn_bwd; two (stream, buffers) sets alternate across steps")}
        del sets

    peaks, peak_src = load_peaks()
    achieved = F / (call_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"], "traffic": measured_traffic("attn_bwd", w.name),
                "kernel": "attn_bwd (one call: delta_kernel, attn_bwd_kernel<dK/dV>, attn_bwd_kernel<dQ>)",
                "peak_source": f"{peak_src} bf16 burst", "launch_ms": call_ms}
    return {"value": value, "ms_per_step": elapsed_ms / args.steps, "e2e": e2e, "roofline": roofline,
            "merge": None, "gpu_launches": 3 * args.steps, "clocks": clocks}


def oracle_backward_sample(w: workloads.Workload, budget_s: float, prefix: int = 1024):
    """Times the fp64 oracle's backward on the first `prefix` positions of one
    (batch, query head) and its KV head per call, heads in turn, until about
    budget_s seconds of CPU work are done; FLOPs 2.5x the forward's on the
    prefix. Returns (TFLOP/s, seconds, calls, threads)."""
    import oracle

    q, k, v = workloads.make_qkv(w, S=prefix)
    do = workloads.make_dout(w, S=prefix)
    threads = oracle.default_threads()
    g = w.Hq // w.Hkv
    pairs = prefix * (prefix + 1) / 2 if w.causal else prefix * prefix
    flops, calls = 0.0, 0
    t0 = time.perf_counter()
    while True:
        b, h = divmod(calls % (w.B * w.Hq), w.Hq)
        oracle.attention_backward(q[b:b + 1, h:h + 1], k[b:b + 1, h // g:h // g + 1],
                                  v[b:b + 1, h // g:h // g + 1], do[b:b + 1, h:h + 1], w.causal,
                                  threads=threads)
        flops += 2.5 * 4.0 * w.D * pairs
        calls += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    secs = time.perf_counter() - t0
    return flops / secs / 1e12, secs, calls, threads


# ----------------------------------------------------------------- the CPU oracle arm

def oracle_sample(w: workloads.Workload, budget_s: float, q=None, k=None, v=None, max_calls: int | None = None):
    """Times the fp64 oracle on sampled query rows of the workload: 256 seeded
    rows of one (batch, head) per call, heads in turn, until about budget_s
    seconds of CPU work are done (at least one call). FLOPs are counted
    exactly, 4*D per visible (query, key) pair.
    Returns (TFLOP/s, seconds, rows done, threads)."""
    import oracle

    if q is None:
        q, k, v = workloads.make_qkv(w)
    threads = oracle.default_threads()
    g = w.Hq // w.Hkv
    flops = 0.0
    done = 0
    calls = 0
    t0 = time.perf_counter()
    if w.varlen:  # one head of one sequence per call, up to 256 seeded rows of it, sequences in turn
        cu = workloads.cu_seqlens(w)
        rng = np.random.Generator(np.random.PCG64(w.seed))
        while True:
            s, h = divmod(calls, w.Hq)
            s %= len(cu) - 1
            a, b = cu[s], cu[s + 1]
            r = np.sort(rng.choice(b - a, size=min(256, b - a), replace=False)).astype(np.int64)[None]
            oracle.attention(q[:, h:h + 1, a:b], k[:, h // g:h // g + 1, a:b], v[:, h // g:h // g + 1, a:b],
                             w.causal, rows=r, threads=threads)
            nvis = r[0] + 1 if w.causal else np.full(r.shape[1], b - a)
            flops += 4.0 * w.D * float(nvis.sum())
            done += r.shape[1]
            calls += 1
            if time.perf_counter() - t0 >= budget_s or (max_calls and calls >= max_calls):
                break
        secs = time.perf_counter() - t0
        return flops / secs / 1e12, secs, done, threads
    rows = workloads.sample_query_rows(w, n=min(w.S, 256))
    while True:
        bh = calls % (w.B * w.Hq)
        b, h = divmod(bh, w.Hq)
        r = rows[bh:bh + 1]
        oracle.attention(q[b:b + 1, h:h + 1], k[b:b + 1, h // g:h // g + 1], v[b:b + 1, h // g:h // g + 1],
                         w.causal, rows=r, threads=threads)
        nvis = np.minimum(r[0] + 1, w.S) if w.causal else np.full(r.shape[1], w.S)
        flops += 4.0 * w.D * float(nvis.sum())
        done += r.shape[1]
        calls += 1
        if time.perf_counter() - t0 >= budget_s or (max_calls and calls >= max_calls):
            break
    secs = time.perf_counter() - t0
    return flops / secs / 1e12, secs, done, threads


def run_reference(args, w):
    q, k, v = workloads.make_qkv(w)
    for _ in range(args.warmup):
        oracle_sample(w, 0.0, q, k, v, max_calls=1)
    rates, secs_all, heads = [], 0.0, 0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        r, s, n, threads = oracle_sample(w, args.reference_budget, q, k, v)
        rates.append(r)
        secs_all += s
        heads += n
    elapsed = time.perf_counter() - t0
    value = sum(rates) / len(rates)
    unit = "(sequence, head), sequences and heads" if w.varlen else "(batch, head), heads"
    sample = (f"{heads} seeded query rows (up to 256 per {unit} in turn) over {args.steps} steps "
              f"(about {args.reference_budget:.0f} s of CPU work per step); fp64 definition")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(w, args.partials),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_ring_schedules(args, w: workloads.Workload) -> dict:
    """Causal ring pass emulated device by device (each device's launches of a
    hop timed alone: on a real ring every device is a whole GPU), for the
    pages' contiguous layout and the zigzag one; per (hop, device) the median
    over the timed passes."""
    import sequence_attn_fwd_gb300 as sa
    from sequence_attn_fwd_gb300 import ring_schedule as rs

    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    out = {}
    for layout in rs.LAYOUTS:
        ring = sa.EmulatedRing(q, k, v, P=w.P, layout=layout, causal=w.causal)
        for _ in range(args.warmup):
            ring.run()
        # a 20 ms GPU-side hold ahead of each timed pass: the pass's launches are
        # all enqueued before it ends, so the events time GPU work only
        runs = [ring.run(timing=True, hold_cycles=40_000_000) for _ in range(args.steps)]
        hop = [[statistics.median(r[0][t][d] for r in runs) for d in range(w.P)] for t in range(w.P)]
        merge = [statistics.median(r[1][d] for r in runs) for d in range(w.P)]
        res = ring_time_from_hops(hop)
        res.update({"merge_ms_max_device": max(merge), "ideal_units": rs.ring_time_units(w.P, layout, w.causal),
                    "hop_ms": [[round(x, 4) for x in row] for row in hop]})
        out[layout] = res
        del ring
        torch.cuda.empty_cache()
    return {"metric": "emulated causal ring pass: sum over hops of the slowest device's attention time",
            "unit": "ms", "higher_is_better": False, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "data": "synthetic", "config": workload_config(w), "layouts": out,
            "speedup_zigzag": out["contiguous"]["ring_ms"] / out["zigzag"]["ring_ms"]}


def workload_config(w: workloads.Workload, partials: str | None = None):
    c = {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "S": w.S, "D": w.D, "causal": w.causal,
         "P": w.P, "chunk": w.chunk, "scale": "1/sqrt(D)",
         "l2": "no flush: each step writes P fp32 partials and reads them back "
               "(>1 GB for ring workloads, inputs >129 MB L2 for single-pass ones)"}
    if w.P > 1 and partials:
        c["partials"] = ("one attn_partial_blocks launch computes the P key chunks' partials"
                         if partials == "grouped" else "one attn_partial launch per key chunk")
    return c


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--warmup-seconds", type=float, default=1.0)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--reference-budget", type=float, default=3.0, help="CPU seconds per reference step")
    ap.add_argument("--cpu-baseline-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "e4m3"],
                    help="e4m3: Q, K, V quantised to FP8 with per-tensor scales (attn_fwd_fp8)")
    ap.add_argument("--partials", default="grouped", choices=["grouped", "per-chunk"],
                    help="ring workloads: the P chunks' partials in one attn_partial_blocks launch "
                         "(default) or one attn_partial launch per chunk")
    ap.add_argument("--backward", action="store_true",
                    help="time the backward (attn_bwd: dQ, dK, dV) instead of the forward step "
                         "(single-pass workloads)")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="with --backward: a smaller sequence length of the same workload (profiling the "
                         "same kernels on a small case)")
    ap.add_argument("--ring-schedule", action="store_true",
                    help="instead of the step: per-hop device times of the emulated causal ring, "
                         "contiguous vs zigzag layout (ring workloads)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)
    w = workloads.WORKLOADS[args.workload]
    if args.seq_len is not None:
        if not args.backward or w.P > 1 or w.varlen or args.seq_len < 1:
            raise SystemExit("--seq-len applies to --backward on single-pass workloads")
        w = dataclasses.replace(w, S=args.seq_len, name=f"{w.name}@S{args.seq_len}")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        if args.impl == "reference":
            if rank != 0:
                return 0
        else:
            dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if args.impl == "reference":
        print(json.dumps(run_reference(args, w)), flush=True)
        return 0

    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    if args.ring_schedule:
        if rank != 0:
            return 0
        if w.P < 2:
            print(json.dumps({"error": "--ring-schedule needs a ring workload"}))
            return 1
        print(json.dumps(run_ring_schedules(args, w)), flush=True)
        return 0
    r = run_ours_backward(args, w, rank, world) if args.backward else run_ours(args, w, rank, world)
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline and args.backward:
            val, secs, calls, threads = oracle_backward_sample(w, args.cpu_baseline_budget)
            cpu = {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                   "sample": f"the oracle's backward on the first 1024 positions of {calls} "
                             f"(batch, query head) pairs in turn ({secs:.1f} s), fp64 chain rule"}
        elif world == 1 and not args.no_cpu_baseline:
            val, secs, heads, threads = oracle_sample(w, args.cpu_baseline_budget, *r.get("inputs", ()))
            unit = "(sequence, head), sequences and heads" if w.varlen else "(batch, head), heads"
            cpu = {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                   "sample": f"{heads} seeded query rows of the workload (up to 256 per {unit} "
                             f"in turn; {secs:.1f} s), fp64 definition"}
        metric = METRIC_BWD if args.backward else METRIC
        line = {"metric": metric, "value": r["value"], "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": args.dtype, "data": "synthetic",
                "config": workload_config(w, args.partials), "roofline": r["roofline"], "merge": r["merge"],
                "cpu_baseline": cpu, "e2e": r["e2e"], "gpu_launches": r["gpu_launches"], "clocks": r["clocks"]}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
