"""Which blocks of a causal Ring-Attention pass each device computes at each hop.

The pages' ring (page "Ulysses与Ring-Attention序列并行技术详解", Ring-Attention
part) gives every device one contiguous chunk of the sequence and passes the K/V
chunks around the ring, one device per hop. Under a causal mask that leaves the
devices with unequal work: at hop t device d attends to the chunk of device
(d - t) mod P, which is visible only when it lies at or before its own chunk,
so device 0 works in one hop and device P - 1 in all P, and every hop takes as
long as a full chunk pair.

The zigzag layout (a load-balanced schedule for the same ring, not on the pages)
cuts the sequence into 2P chunks and gives device d the chunks d and 2P - 1 - d,
one from each end. K/V still travel one device per hop. At every hop every
device then has exactly two chunk pairs' worth of visible work (the two diagonal
halves plus one full pair at hop 0, two full pairs at every later hop), so no
device waits for another.

Chunks are numbered along the sequence. A block (q_chunk, kv_chunk) is the
attention of that query chunk to that key chunk: all keys visible when
kv_chunk < q_chunk, the causal triangle when they are equal, nothing when
kv_chunk > q_chunk (never scheduled).
"""
from __future__ import annotations

from dataclasses import dataclass

LAYOUTS = ("contiguous", "zigzag")


@dataclass(frozen=True)
class Block:
    q_chunk: int
    kv_chunk: int

    @property
    def diagonal(self) -> bool:
        return self.q_chunk == self.kv_chunk

    @property
    def work(self) -> float:
        """Visible (query, key) pairs in units of one full chunk pair (the
        diagonal's own-position pairs are left out, as in the FLOP count)."""
        return 0.5 if self.diagonal else 1.0


def n_chunks(P: int, layout: str) -> int:
    if layout not in LAYOUTS:
        raise ValueError(f"layout must be one of {LAYOUTS}")
    if P < 1:
        raise ValueError("P must be >= 1")
    return P if layout == "contiguous" else 2 * P


def device_chunks(P: int, layout: str) -> list[list[int]]:
    """The sequence chunks (of Q, K and V) device d holds, in sequence order."""
    if n_chunks(P, layout) == P:
        return [[d] for d in range(P)]
    return [[d, 2 * P - 1 - d] for d in range(P)]


def hop_blocks(P: int, layout: str, causal: bool = True) -> list[list[list[Block]]]:
    """blocks[t][d]: the blocks device d computes at hop t, when it holds the
    K/V chunks of device (d - t) mod P."""
    chunks = device_chunks(P, layout)
    out = []
    for t in range(P):
        hop = []
        for d in range(P):
            src = (d - t) % P
            hop.append([Block(qc, kc) for qc in chunks[d] for kc in chunks[src]
                        if not causal or kc <= qc])
        out.append(hop)
    return out


def hop_work(P: int, layout: str, causal: bool = True) -> list[list[float]]:
    """work[t][d] in units of one full pair of this layout's chunks."""
    return [[sum(b.work for b in blocks) for blocks in hop] for hop in hop_blocks(P, layout, causal)]


def ring_time_units(P: int, layout: str, causal: bool = True) -> float:
    """Ring time if every hop lasts as long as its busiest device, in units of a
    full pair of contiguous (S/P) chunks; a zigzag chunk pair is a quarter of that."""
    scale = 1.0 if layout == "contiguous" else 0.25
    return scale * sum(max(w) for w in hop_work(P, layout, causal))
