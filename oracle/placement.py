"""Expert-placement policies replayed on a routing trace -- [Review] §2.4.

The ablation on the page replays routing traces under three ways of deciding
which (layer, expert) pairs live in GPU memory, at equal capacity, and counts
the routed experts that are not resident ("misses"):

* global LRU (the engine's own policy): one residency set shared by all
  layers; a routed expert that is resident is refreshed, one that is not is
  loaded and the least recently used entry is evicted (§2.4, the shared LRU).
  The rules are the cache simulator's (``lru.LRUSim``) with every miss filled.
* prefill-time placement: the hot experts are picked when the prompt is
  processed and then frozen for decode (§2.4, the placement updated at prefill
  time).  Reading here: the ``capacity`` keys routed most often during the
  prefill, ties to the lower key, stay resident for the whole decode.
* static split: tensors assigned to devices when the model loads, whatever the
  routing (§2.4, the routing-agnostic static split).  Reading here: whole
  layers in order, i.e. the keys 0 .. capacity-1 of key = layer * E + expert.

A trace is a list of decode steps; each step lists, per layer, the experts its
tokens were routed to (duplicates allowed).  An access is one unique routed
expert of one layer step.
"""
from __future__ import annotations

from typing import Dict, Iterable, List, Sequence, Tuple

from .lru import LRUSim


def _unique(experts: Iterable[int]) -> List[int]:
    return sorted(set(int(e) for e in experts if int(e) >= 0))


def global_lru(trace: Sequence[Sequence[Sequence[int]]], n_layers: int, n_experts: int,
               capacity: int) -> Tuple[int, int]:
    """(accesses, misses) of the trace under the shared LRU, starting empty."""
    sim = LRUSim(capacity, n_experts)
    acc = miss = 0
    for step in trace:
        for layer in range(n_layers):
            U = _unique(step[layer])
            acc += len(U)
            events, _ = sim.step(layer, U, 1.0)
            miss += sum(1 for e in events if e[0] == "fill")
    return acc, miss


def prefill_hot_set(prefill_counts: Dict[int, int], capacity: int) -> set:
    """The ``capacity`` keys with the most prefill assignments (ties to the lower key)."""
    ranked = sorted((k for k, c in prefill_counts.items() if c > 0), key=lambda k: (-prefill_counts[k], k))
    return set(ranked[:capacity])


def static_set(n_layers: int, n_experts: int, capacity: int) -> set:
    """Keys 0 .. capacity-1: whole layers in order."""
    return set(range(min(capacity, n_layers * n_experts)))


def fixed_set(trace: Sequence[Sequence[Sequence[int]]], n_layers: int, n_experts: int,
              resident: set) -> Tuple[int, int]:
    """(accesses, misses) of the trace when exactly ``resident`` keys are on the GPU throughout."""
    acc = miss = 0
    for step in trace:
        for layer in range(n_layers):
            for e in _unique(step[layer]):
                acc += 1
                miss += (layer * n_experts + e) not in resident
    return acc, miss
