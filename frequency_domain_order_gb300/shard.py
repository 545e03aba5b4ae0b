"""Cutting one input stream into shards that are filtered independently (one per GPU, or one
after another), with the same result as filtering the stream in one call.

Overlap-save blocks depend on the input only (step 3 of the claim in "一种基于GPU的高阶数字FIR
滤波器频域并行处理实现方法", zl.czvv.com/42398539.html: E_i = {D_{i-1}, B_i}), so a stream splits
into contiguous shards as long as each shard starts with the M-1 samples that precede it -- its
halo -- as the state S0 of its call: the halo of shard g is the tail of shard g-1 (of S0 for the
first shard).  Shards start on a multiple of L (2L for real data, whose blocks are filtered in
pairs), so every shard cuts the stream where one call's transforms begin and the sharded result
equals one call's bit for bit.  The final state S0' is the one the last shard returns.

Host logic only: these functions compute ranges and slice arrays (numpy or torch); no data moves
between devices here.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple


def shard_ranges(n: int, L: int, parts: int, real: bool = False) -> List[Tuple[int, int]]:
    """`parts` contiguous half-open ranges covering [0, n).  Every start is a multiple of the
    transform span (L, or 2L for real data); whole spans are dealt out as evenly as possible
    (earlier shards take the remainder), and the last shard also takes the partial span at the
    end.  Shards may be empty when there are fewer spans than parts."""
    if n < 0 or L < 1 or parts < 1:
        raise ValueError("need n >= 0, L >= 1, parts >= 1")
    span = L * (2 if real else 1)
    whole = n // span
    base, extra = divmod(whole, parts)
    out, start = [], 0
    for g in range(parts):
        stop = start + (base + (1 if g < extra else 0)) * span
        if g == parts - 1:
            stop = n
        out.append((start, stop))
        start = stop
    return out


def halo(x, s0, start: int, M: int):
    """The M-1 samples that precede x[start] in the stream concat(s0, x): the state S0 for a
    call that filters x[start:].  Returns an array of the same kind as x (concatenated with
    numpy or torch as needed) of length M-1."""
    h = M - 1
    if h == 0:
        return x[0:0]
    if start >= h:
        return x[start - h:start]
    head = s0[start:]  # the newest h - start samples of S0
    tail = x[:start]
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return torch.cat([head.to(x.device, x.dtype), tail])
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    import numpy as np
    return np.concatenate([np.asarray(head, dtype=x.dtype), tail])


def shard_states(x, s0, ranges: Sequence[Tuple[int, int]], M: int):
    """The state of each shard's call: halo(x, s0, start, M) for every range."""
    return [halo(x, s0, a, M) for a, _ in ranges]
