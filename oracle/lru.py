"""Simulator of the shared slot-pool expert cache, written from the pages' rules.

* One slot holds every tensor of one (layer, expert); residency, lookup and
  execution go by the logical key (layer, expert) ([Review] §2 opening).
* One cache is shared by all MoE layers; a hit refreshes recency, a miss
  loads the expert and evicts the least recently used one ([Review] §2.4).
* Per layer step the routed experts are de-duplicated, classified hit/miss
  against the residency table, q is taken from the bandwidth ratio, victims
  are chosen and each routed expert is rewritten to a slot or to an
  "evaluate elsewhere" marker ([Review] §2.6, "设备侧缓存控制").  Experts in C
  do not change residency ([Review] §2.5).  Victims are the least recently
  used slots found in one pass; the miss path uses the first q ([Review]
  §2.6, "一次遍历选受害者").
* The cache can be rebuilt for a new slot budget at a safe point without
  reloading the host pool ([Review] §2.7).
* Prefill takes two whole-layer buffers from the same slot pool, and entries
  that survive prefill warm the decode cache ([Review] §2.2).

Readings where the pages are silent (each one a choice, listed with the others
in the design notes):
  - routed experts are processed in ascending expert id;
  - the q filled misses are the first q misses in ascending expert id;
  - a step whose unique experts exceed the slot count runs in waves of at most
    N experts; each wave has its own recency stamp;
  - victims: empty slots first (ascending slot), then slots not touched by
    this wave ordered by (stamp, slot);
  - resize keeps the min(used, N') entries with the largest (stamp, -slot);
    kept entries below N' stay in place, kept entries at or above N' move, in
    ascending old slot order, into the lowest free slots below N';
  - streaming takes the last 2E slots (a resize to N - 2E), and at the end
    adopts the experts of the last two streamed layers (older layer first,
    one stamp per layer, experts in ascending id): a key already resident
    is refreshed and its buffer slot left empty.

Event codes: ("hit", e, slot), ("fill", e, slot, evicted_key or -1), ("ext", e).
"""
from __future__ import annotations

from typing import List, Optional, Sequence, Tuple

import numpy as np

from .qsplit import qsplit_ratio


class LRUSim:
    def __init__(self, n_slots: int, n_experts: int):
        self.E = int(n_experts)
        self.N = int(n_slots)
        self.key = [-1] * self.N          # key = layer * E + expert, -1 empty
        self.stamp = [0] * self.N         # 0 for empty slots
        self.clock = 0
        self.where = {}                   # key -> slot
        self.hits = self.fills = self.externals = 0

    # -- helpers -------------------------------------------------------
    def _victims(self, q: int, touched: set) -> List[int]:
        cand = [s for s in range(self.N) if s not in touched]
        cand.sort(key=lambda s: (0 if self.key[s] < 0 else 1, self.stamp[s], s))
        return cand[:q]

    def n_waves(self, n_unique: int) -> int:
        return 0 if n_unique == 0 else -(-n_unique // self.N)

    # -- one layer step ------------------------------------------------
    def step(self, layer: int, experts: Sequence[int], ratio: float = 1.0, wave: Optional[int] = None):
        """Process the routed experts of one layer step (any order, duplicates allowed).

        Returns (events, slot_of) where slot_of maps expert -> slot (>= 0),
        -2 (evaluated elsewhere) or -1 (not routed / not in this wave).  With
        ``wave`` None all waves run in order and ``slot_of`` is per wave list.
        """
        U = sorted(set(int(e) for e in experts))
        waves = [U[i:i + self.N] for i in range(0, len(U), self.N)]
        if wave is not None:
            waves = [waves[wave]] if wave < len(waves) else []
        all_events, all_slot_of = [], []
        for W in waves:
            ev, so = self._wave(layer, W, ratio)
            all_events.extend(ev)
            all_slot_of.append(so)
        return all_events, all_slot_of

    def _wave(self, layer: int, W: List[int], ratio: float):
        slot_of = [-1] * self.E
        if not W:
            return [], slot_of
        self.clock += 1
        c = self.clock
        touched = set()
        misses = []
        events = {}
        for e in W:
            key = layer * self.E + e
            s = self.where.get(key)
            if s is not None:
                self.stamp[s] = c
                touched.add(s)
                slot_of[e] = s
                events[e] = ("hit", e, s)
                self.hits += 1
            else:
                misses.append(e)
        q = qsplit_ratio(len(misses), ratio)
        victims = self._victims(q, touched)
        for e, s in zip(misses[:q], victims):
            old = self.key[s]
            if old >= 0:
                del self.where[old]
            key = layer * self.E + e
            self.key[s], self.stamp[s] = key, c
            self.where[key] = s
            slot_of[e] = s
            events[e] = ("fill", e, s, old)
            self.fills += 1
        for e in misses[q:]:
            slot_of[e] = -2
            events[e] = ("ext", e)
            self.externals += 1
        return [events[e] for e in W], slot_of

    # -- safe-point resize --------------------------------------------
    def resize(self, n_new: int) -> List[Tuple[int, int]]:
        """Rebuild for n_new slots; returns the (src, dst) slot moves, in order."""
        used = [s for s in range(self.N) if self.key[s] >= 0]
        used.sort(key=lambda s: (-self.stamp[s], s))
        kept = set(used[:n_new])
        movers = sorted(s for s in kept if s >= n_new)
        free = [s for s in range(min(self.N, n_new)) if s not in kept]
        moves = list(zip(movers, free))
        key = [-1] * n_new
        stamp = [0] * n_new
        for s in kept:
            if s < n_new:
                key[s], stamp[s] = self.key[s], self.stamp[s]
        for src, dst in moves:
            key[dst], stamp[dst] = self.key[src], self.stamp[src]
        self.N, self.key, self.stamp = n_new, key, stamp
        self.where = {k: s for s, k in enumerate(key) if k >= 0}
        return moves

    # -- prefill streaming --------------------------------------------
    def stream_begin(self) -> Tuple[int, List[Tuple[int, int]]]:
        """Carve two whole-layer buffers off the end of the pool; returns (buffer base, moves)."""
        if self.N < 2 * self.E:
            raise ValueError("fewer than two whole layers of slots: use the on-demand path")
        n_full = self.N
        moves = self.resize(n_full - 2 * self.E)
        self._n_full = n_full
        return n_full - 2 * self.E, moves

    def stream_end(self, layers: Sequence[Tuple[int, int]]):
        """Give the buffers back; ``layers`` = [(layer, buffer index)] streamed last, oldest first.

        Buffer b occupies slots base + b*E .. base + b*E + E - 1, expert e at base + b*E + e.
        """
        base = self.N
        n_full = self._n_full
        self.key += [-1] * (n_full - base)
        self.stamp += [0] * (n_full - base)
        self.N = n_full
        for layer, b in layers:
            self.clock += 1
            c = self.clock
            for e in range(self.E):
                key = layer * self.E + e
                s_buf = base + b * self.E + e
                s_old = self.where.get(key)
                if s_old is not None:
                    self.stamp[s_old] = c
                else:
                    self.key[s_buf], self.stamp[s_buf] = key, c
                    self.where[key] = s_buf

    def state(self):
        """(key_of_slot, stamp) as int arrays."""
        return np.array(self.key, dtype=np.int64), np.array(self.stamp, dtype=np.int64)
