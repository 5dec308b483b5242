"""The parameter list split over the ranks of a data-parallel job (a ZeRO-style partition), for a sharded step:
each rank holds a contiguous part of the list's parameters (with their gradients and moments), sums the squares of
its part's gradient (mica_grad_sumsq), the ranks exchange those sums (an all-gather of one double each), every rank
derives the same clip factor from them in rank order (mica_clip_factor_from_sumsq), and each rank updates its own
part (mica_adamw_steps). The joint norm is that of every gradient of every rank, as ClipGradNorms takes it.

The split is by element: the list's tensors laid end to end, rank r takes elements [P r / N, P (r + 1) / N), each
boundary moved down to the nearest multiple of 8 elements within its tensor, so that every piece starts at a whole
octet (a 32-byte float32 vector, a 16-byte binary16 one or 4 packed BF16 words) of its tensor: the pieces keep the
tensors' alignment and packed words are never split.
"""
from __future__ import annotations

from typing import Sequence

import torch

OCT = 8


def _boundary(sizes: Sequence[int], starts: Sequence[int], x: int) -> int:
    """The list position x moved down to a multiple of OCT within the tensor that holds it."""
    lo, hi = 0, len(sizes)
    while hi - lo > 1:  # the last tensor starting at or before x
        mid = (lo + hi) // 2
        if starts[mid] <= x:
            lo = mid
        else:
            hi = mid
    return starts[lo] + (x - starts[lo]) // OCT * OCT


def shard_pieces(sizes: Sequence[int], world: int, rank: int) -> list[tuple[int, int, int]]:
    """Rank `rank`'s part of a list of tensors of `sizes` elements split over `world` ranks: a list of (tensor,
    first element, end element) pieces, in list order. Over all ranks the pieces cover every element once."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of {world}")
    starts, total = [], 0
    for n in sizes:
        starts.append(total)
        total += int(n)
    if total == 0:
        return []
    lo = _boundary(sizes, starts, total * rank // world) if rank > 0 else 0
    hi = _boundary(sizes, starts, total * (rank + 1) // world) if rank < world - 1 else total
    pieces = []
    for k, (s, n) in enumerate(zip(starts, sizes)):
        a, b = max(lo, s), min(hi, s + int(n))
        if a < b:
            pieces.append((k, a - s, b - s))
    return pieces


def piece_views(tensors: Sequence[torch.Tensor], pieces, packed: bool = False) -> list[torch.Tensor]:
    """The views of `tensors` that `pieces` name: elements [a, b) of tensor k, or, for packed BF16 moments (one
    32-bit word per two elements), words [a / 2, ceil(b / 2))."""
    if packed:
        return [tensors[k][a // 2:(b + 1) // 2] for k, a, b in pieces]
    return [tensors[k][a:b] for k, a, b in pieces]
