"""Seeded synthetic workloads for blockwise attention and the log-sum-exp merge.

This module holds shapes and random draws only. It contains none of the
attention or merge arithmetic, so both the fp64 oracle and the CUDA path can
take their inputs from here without sharing any of the method's code.

Shapes follow the [B, H, S, D] layout (D innermost) that the page
"Ulysses与Ring-Attention序列并行技术详解" uses in its Ulysses listing
(the "# [B, H, L, D]" comment on the gathered keys). Sizes are those of
7B-class attention heads (D = 128) at 4K-131K context, the workloads the
pages talk about; the pages name no dataset that this stands in for.

Recipe (every draw is reproducible from the integer seed):
  * SeedSequence(seed).spawn(4) gives the streams for Q, K, V and "extra".
  * Q, K and V each spawn one child stream per (batch, head); that head's
    [S, D] block is PCG64 standard_normal in float32, rounded to bf16 with
    round-to-nearest-even (torch's float32 -> bfloat16 cast).
  * "extra" spawns the stream for the key-boost positions (a distinct
    sample of floor(frac * S) sequence positions whose keys are multiplied
    by 2, exact in bf16, for every batch and KV head), the stream for the
    sampled query rows, the stream for synthetic merge partials, the stream
    for the sequence lengths of a packed (varlen) workload, and the stream
    of the output gradient dO for the backward (drawn like Q: one
    child stream per (batch, query head), N(0, 1) rounded to bf16).
  * A packed workload (B = 1, S = total tokens) draws sequence lengths
    round(exp(N(ln 1536, 0.8^2))) clipped to [128, 8192] until the total is
    reached, the last one cut to fit: a training-style length mix with many
    short and some long sequences. Q, K and V are drawn as for one sequence
    of S tokens; the sequences are consecutive row ranges of it.
"""
from __future__ import annotations

import dataclasses
import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, masking, ring chunking and its seed."""

    name: str
    B: int
    Hq: int
    Hkv: int
    S: int
    D: int
    causal: bool
    P: int  # number of KV chunks of the emulated ring (1 = single pass)
    seed: int
    k_boost_frac: float = 0.0  # fraction of positions whose keys are doubled
    sample_rows: int = 0  # query rows per (batch, head) checked against the oracle; 0 = all
    varlen: bool = False  # packed sequences of seeded lengths (B = 1, S = total tokens)

    @property
    def chunk(self) -> int:
        return self.S // self.P

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def attention_flops(self) -> float:
        """Causal-adjusted FLOPs 4*B*Hq*S^2*D (halved when causal); a packed
        workload sums this over its sequences."""
        if self.varlen:
            lens = seq_lens(self).astype(np.float64)
            f = 4.0 * self.Hq * self.D * float((lens * lens).sum())
        else:
            f = 4.0 * self.B * self.Hq * self.S * self.S * self.D
        return f * 0.5 if self.causal else f


# The workloads the attention path is checked and measured on.
WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_b1h2s256d64", 1, 2, 2, 256, 64, False, 1, 1001),
        Workload("ring8_b2h32s4096d128_causal", 2, 32, 32, 4096, 128, True, 8, 1002),
        Workload("gqa_b1hq28hkv4s32768d128_causal", 1, 28, 4, 32768, 128, True, 1, 1003,
                 k_boost_frac=0.01),
        Workload("merge16_b2h32s8192d128_causal", 2, 32, 32, 8192, 128, True, 16, 1004),
        Workload("ring16_b1hq32hkv8s131072d128_causal", 1, 32, 8, 131072, 128, True, 16, 1005,
                 sample_rows=64),
        Workload("varlen_hq32hkv8t65536d128_causal", 1, 32, 8, 65536, 128, True, 1, 1006,
                 varlen=True),
        # Reduced forms of the 131K ring for profiling under ncu (a few GB on the
        # device): the same heads and key-chunk length (8192) over a quarter of
        # the sequence, and the same 16-way merge over a quarter of the rows.
        Workload("ring4_b1hq32hkv8s32768d128_causal", 1, 32, 8, 32768, 128, True, 4, 1007,
                 sample_rows=64),
        Workload("ring16_b1hq32hkv8s32768d128_causal", 1, 32, 8, 32768, 128, True, 16, 1008,
                 sample_rows=64),
    ]
}


def _streams(seed: int):
    return np.random.SeedSequence(seed).spawn(4)


def _normal_heads(ss: np.random.SeedSequence, B: int, H: int, S: int, D: int,
                  threads: int = 8) -> torch.Tensor:
    """[B, H, S, D] bf16 (CPU): one child stream per head, N(0, 1) draws."""
    children = ss.spawn(B * H)
    out = np.empty((B * H, S, D), dtype=np.float32)

    def fill(i: int) -> None:
        np.random.Generator(np.random.PCG64(children[i])).standard_normal(
            (S, D), dtype=np.float32, out=out[i])

    with ThreadPoolExecutor(max_workers=max(1, min(threads, B * H))) as ex:
        list(ex.map(fill, range(B * H)))
    t = torch.from_numpy(out).view(B, H, S, D)
    return t.to(torch.bfloat16)


def make_qkv(w: Workload, S: int | None = None):
    """Seeded bf16 Q [B,Hq,S,D], K and V [B,Hkv,S,D] on the CPU.

    S overrides the sequence length (for reduced-size parity cases that
    keep every other property of the workload)."""
    S = w.S if S is None else S
    sq, sk, sv, sx = _streams(w.seed)
    q = _normal_heads(sq, w.B, w.Hq, S, w.D)
    k = _normal_heads(sk, w.B, w.Hkv, S, w.D)
    v = _normal_heads(sv, w.B, w.Hkv, S, w.D)
    if w.k_boost_frac > 0:
        pos = boost_positions(w, S)
        k[:, :, pos, :] = k[:, :, pos, :] * 2  # exact: a bf16 exponent bump
    return q, k, v


def make_dout(w: Workload, S: int | None = None) -> torch.Tensor:
    """Seeded bf16 output gradient dO [B,Hq,S,D] on the CPU (backward inputs)."""
    S = w.S if S is None else S
    return _normal_heads(_streams(w.seed)[3].spawn(5)[4], w.B, w.Hq, S, w.D)


def boost_positions(w: Workload, S: int | None = None) -> np.ndarray:
    S = w.S if S is None else S
    rng = np.random.Generator(np.random.PCG64(_streams(w.seed)[3].spawn(3)[0]))
    n = int(math.floor(w.k_boost_frac * S))
    return np.sort(rng.choice(S, size=n, replace=False))


def sample_query_rows(w: Workload, n: int | None = None, S: int | None = None) -> np.ndarray:
    """[B*Hq, n] distinct sorted query rows per (batch, head), uniform on [0, S)."""
    S = w.S if S is None else S
    n = w.sample_rows if n is None else n
    rng = np.random.Generator(np.random.PCG64(_streams(w.seed)[3].spawn(3)[1]))
    rows = np.stack([np.sort(rng.choice(S, size=n, replace=False)) for _ in range(w.B * w.Hq)])
    return rows.astype(np.int64)


def seq_lens(w: Workload) -> np.ndarray:
    """Sequence lengths of a packed workload (int64, summing to w.S); [S] otherwise."""
    if not w.varlen:
        return np.array([w.S], dtype=np.int64)
    rng = np.random.Generator(np.random.PCG64(_streams(w.seed)[3].spawn(4)[3]))
    lens, total = [], 0
    while total < w.S:
        n = int(min(max(round(math.exp(rng.normal(math.log(1536.0), 0.8))), 128), 8192))
        n = min(n, w.S - total)
        lens.append(n)
        total += n
    return np.array(lens, dtype=np.int64)


def cu_seqlens(w: Workload) -> list[int]:
    """[0, L0, L0 + L1, ..., S] for a packed workload."""
    return [0] + np.cumsum(seq_lens(w)).tolist()


def make_partials(P: int, B: int, H: int, S: int, D: int, seed: int, causal: bool = True):
    """Synthetic per-chunk partials for the merge alone.

    O_i ~ N(0, 1) float32 [P,B,H,S,D]; lse_i = 8 + 2 N(0, 1) float32 [P,B,H,S].
    With ``causal``, the keys are split into P equal chunks and chunk c is
    invisible to rows s < c*S/P, as in a causal ring: there lse_i = -inf and
    O_i = 0, the values an empty partial carries."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed).spawn(4)[3].spawn(3)[2]))
    o = rng.standard_normal((P, B, H, S, D), dtype=np.float32)
    lse = (8.0 + 2.0 * rng.standard_normal((P, B, H, S), dtype=np.float32)).astype(np.float32)
    if causal:
        C = S // P
        for c in range(1, P):
            lse[c, :, :, : c * C] = -np.inf
            o[c, :, :, : c * C, :] = 0.0
    return torch.from_numpy(o), torch.from_numpy(lse)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """The raw uint16 bit patterns of a contiguous bf16 CPU tensor."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)
