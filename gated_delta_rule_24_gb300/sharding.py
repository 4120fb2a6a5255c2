"""Splitting one packed varlen prefill batch across ranks (one GPU each).

Sequences are independent in Gated Delta Rule prefill (each (sequence, head)
scan starts from its own state), so a batch shards by sequence with no
exchange at all: rank r takes a contiguous range of sequences, runs the
prefill on its rows, and writes its own state slots.  Ranges are chosen to
balance tokens; state slots keep their global numbering through explicit
state indices, so pools can be shared or replicated without renumbering.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Sequence


@dataclass
class Shard:
    rank: int
    seq_begin: int       # first sequence of this rank
    seq_end: int         # one past the last
    row_begin: int       # first packed token row
    row_end: int
    cu_local: List[int]  # cu_seqlens of the shard, starting at 0
    slots: List[int]     # state slot of each local sequence (global numbering)


def split_sequences(cu_seqlens: Sequence[int], world: int,
                    state_indices: Sequence[int] | None = None) -> List[Shard]:
    """Contiguous sequence ranges per rank with near-equal token counts.

    Every sequence lands on exactly one rank; a rank may get no sequence when
    there are fewer sequences than ranks.
    """
    cu = [int(x) for x in cu_seqlens]
    n = len(cu) - 1
    total = cu[-1] - cu[0]
    bounds = [0]
    for r in range(1, world):
        target = cu[0] + total * r / world
        # first sequence boundary at or past the target, never before the previous cut
        b = bounds[-1]
        while b < n and cu[b] < target:
            b += 1
        bounds.append(b)
    bounds.append(n)
    shards = []
    for r in range(world):
        a, b = bounds[r], bounds[r + 1]
        base = cu[a]
        slots = list(range(a, b)) if state_indices is None else [int(state_indices[i]) for i in range(a, b)]
        shards.append(Shard(rank=r, seq_begin=a, seq_end=b, row_begin=cu[a], row_end=cu[b],
                            cu_local=[c - base for c in cu[a:b + 1]] if b > a else [0], slots=slots))
    return shards


def shard_problem(p, world: int, rank: int):
    """Rank ``rank``'s part of problem ``p`` (a workloads.Problem) as a call of its own,
    in the library's argument contract: the shard's token rows of q/k/v/g/beta, its
    cu_seqlens starting at 0, and explicit state_indices holding the global slots of its
    sequences into the unchanged state pools (initial and output), so every rank writes
    only its own slots.  Returns (Shard, Problem)."""
    import dataclasses

    import torch

    idx = None if p.state_indices is None else p.state_indices.tolist()
    s = split_sequences(p.cu_seqlens.tolist(), world, idx)[rank]
    rows = slice(s.row_begin, s.row_end)
    pick = {name: (None if getattr(p, name) is None else getattr(p, name)[rows])
            for name in ("q", "k", "v", "g", "beta")}
    idx_dtype = torch.int32 if p.state_indices is None else p.state_indices.dtype
    sub = dataclasses.replace(
        p, **pick, name=f"{p.name}_shard{rank}of{world}",
        cu_seqlens=torch.tensor(s.cu_local, dtype=p.cu_seqlens.dtype, device=p.cu_seqlens.device),
        state_indices=torch.tensor(s.slots, dtype=idx_dtype, device=p.cu_seqlens.device))
    return s, sub
