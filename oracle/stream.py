"""Time model of whole-layer double-buffered prefill streaming.

[Review] §2.2 "全层双缓冲": while the GPU computes layer l from buffer A, a
transfer stream fills buffer B with all of layer l+1; the buffers then swap.
The copy of layer l+1 can start before layer l's routing is known because the
whole layer is loaded.  Without the second buffer, copy and compute alternate.

For per-layer copy times c_l and compute times p_l (l = 0..L-1):
  double-buffered: c_0, then for each l the next copy c_{l+1} runs beside p_l;
                   the copy into a buffer also waits for the compute that last
                   read it (layer l-1), which the recurrence below encodes.
  serialized:      sum_l (c_l + p_l).
"""
from typing import Sequence


def serialized_time(copy: Sequence[float], compute: Sequence[float]) -> float:
    return float(sum(copy) + sum(compute))


def overlapped_time(copy: Sequence[float], compute: Sequence[float]) -> float:
    """Finish time of the last compute with two buffers and one transfer stream."""
    L = len(copy)
    copy_done = [0.0] * L
    comp_done = [0.0] * L
    t_copy = 0.0
    for l in range(L):
        start = t_copy
        if l >= 2:                       # buffer l % 2 is free once layer l-2 is computed
            start = max(start, comp_done[l - 2])
        copy_done[l] = start + copy[l]
        t_copy = copy_done[l]
        prev = comp_done[l - 1] if l else 0.0
        comp_done[l] = max(copy_done[l], prev) + compute[l]
    return comp_done[-1] if L else 0.0


def link_bound_time(pool_bytes: float, link_bytes_per_s: float) -> float:
    """Lower bound when compute is fully hidden: the whole pool crosses the link once."""
    return pool_bytes / link_bytes_per_s
