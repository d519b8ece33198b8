"""ORACLE (test infrastructure only): admission / eviction policy of the
per-tensor HBM expert pools.

Sources (page titles and sections):
- Zapdev-labs/a6000-custom-kernels, the pointer-table paragraph: each expert
  tensor has its own table, pool and stamp array; cold reads are logged as
  (tensor_id << 12 | expert); a promotion pass between decode steps admits
  repeatedly-missed experts (2nd sighting) into free pool slots and evicts by
  stamp scan; pools are seeded from a routing-frequency table.
- neurall/llama.cpp, "How it works", Expert cache: a missed expert takes a
  slot only after repeated use within the last 64 tokens; the prompt pass
  borrows expert blocks and gives them back afterwards, refilled with hot
  experts.

State per tensor t: capacity, slot_of[e] (-1 = cold), owner[slot] (-1 =
free), stamp[slot], last_seen[e] (-1 = no sighting).  One clock for all.

Readings where the pages are silent:
- a step of n tokens advances the clock by n before anything else; hits of
  the step get stamp = clock; all tokens of a step share one sighting;
- sightings count misses only; a miss of e is admitted when
  last_seen[e] >= 0 and clock - last_seen[e] < window (both sightings within
  the last `window` tokens); otherwise last_seen[e] = clock;
- misses are handled in ascending key order; an admission takes the lowest
  free slot, else the slot with the smallest stamp among slots with
  stamp < clock (ties: lowest slot); with no such slot, or after
  max_swaps_per_step admissions (0 = no limit), the admission is skipped and
  last_seen is kept;
- the placed expert gets stamp = clock and last_seen = -1; an evicted
  expert's sighting history starts empty (last_seen = -1);
- seeding puts seed_order[0..n_seed) into slots 0..n_seed-1, stamps 0;
- borrow/return: global slot g of a pool with `slots_per_tensor` slots per
  tensor and n_tensors tensors is local slot g // n_tensors of tensor
  g % n_tensors; borrow(n) lends the n highest global slots (their experts
  are evicted and their tensors' capacities shrink); while slots are lent a
  step advances the clock, stamps hits and logs misses but admits nothing;
  give_back() returns them and refills each returned slot, in ascending
  global order, with its tensor's most frequent non-resident expert by seed
  order (stamp = clock).
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass
class _Tensor:
    capacity: int
    seed_order: list
    slot_of: list
    owner: list
    stamp: list
    last_seen: list
    lent: set = field(default_factory=set)  # local slots lent to a prefill pass


class PolicyOracle:
    def __init__(self, n_experts: int, window: int = 64, max_swaps_per_step: int = 0,
                 slots_per_tensor: int | None = None, n_tensors: int | None = None):
        self.E = n_experts
        self.window = window
        self.max_swaps = max_swaps_per_step
        self.clock = 0
        self.t: dict[int, _Tensor] = {}
        self.slots_per_tensor = slots_per_tensor
        self.n_tensors = n_tensors
        self.n_lent = 0
        self.stats = dict(hits=0, misses=0, admissions=0, evictions=0)

    # -- registration ------------------------------------------------------
    def add_tensor(self, tid: int, capacity: int, seed_order, n_seed: int | None = None):
        seed_order = [int(e) for e in seed_order]
        if n_seed is None:
            n_seed = min(capacity, len(seed_order))
        assert 0 <= n_seed <= capacity <= self.E
        assert len(set(seed_order)) == len(seed_order)
        t = _Tensor(capacity, seed_order, [-1] * self.E, [-1] * capacity, [0] * capacity, [-1] * self.E)
        for s in range(n_seed):
            e = seed_order[s]
            t.slot_of[e] = s
            t.owner[s] = e
        self.t[tid] = t

    # -- one step ------------------------------------------------------------
    def step(self, n_tokens: int, used: dict) -> list:
        """used: {tid: iterable of experts read this step}.  Returns the
        sorted unique miss keys (tid << 12 | e) of the step."""
        self.clock += n_tokens
        misses = []
        for tid in sorted(used):
            t = self.t[tid]
            for e in sorted(set(int(v) for v in used[tid])):
                s = t.slot_of[e]
                if s >= 0:
                    t.stamp[s] = self.clock
                    self.stats["hits"] += 1
                else:
                    misses.append((tid << 12) | e)
        misses.sort()
        self.stats["misses"] += len(misses)
        if self.n_lent == 0:
            self._admit(misses)
        return misses

    def _usable(self, t: _Tensor):
        return [s for s in range(t.capacity) if s not in t.lent]

    def _admit(self, misses):
        swaps = 0
        for key in misses:
            tid, e = key >> 12, key & 0xFFF
            t = self.t[tid]
            ls = t.last_seen[e]
            if not (ls >= 0 and self.clock - ls < self.window):
                t.last_seen[e] = self.clock
                continue
            if self.max_swaps and swaps >= self.max_swaps:
                continue
            slot = self._pick_slot(t)
            if slot is None:
                continue
            victim = t.owner[slot]
            if victim >= 0:
                t.slot_of[victim] = -1
                t.last_seen[victim] = -1
                self.stats["evictions"] += 1
            t.owner[slot] = e
            t.slot_of[e] = slot
            t.stamp[slot] = self.clock
            t.last_seen[e] = -1
            swaps += 1
            self.stats["admissions"] += 1

    def _pick_slot(self, t: _Tensor):
        usable = self._usable(t)
        for s in usable:
            if t.owner[s] < 0:
                return s
        best = None
        for s in usable:
            if t.stamp[s] < self.clock and (best is None or t.stamp[s] < t.stamp[best]):
                best = s
        return best

    # -- borrow / return around a prefill pass -------------------------------
    def _global_tail(self, n: int):
        nt, spt = self.n_tensors, self.slots_per_tensor
        assert nt is not None and spt is not None, "borrow needs the global slot layout"
        G = nt * spt
        assert 0 <= n <= G
        return [(g % nt, g // nt) for g in range(G - n, G)]

    def borrow(self, n: int):
        assert self.n_lent == 0
        for tid, local in self._global_tail(n):
            t = self.t.get(tid)
            if t is None or local >= t.capacity:
                continue
            e = t.owner[local]
            if e >= 0:
                t.slot_of[e] = -1
                t.last_seen[e] = -1
                t.owner[local] = -1
                self.stats["evictions"] += 1
            t.lent.add(local)
        self.n_lent = n

    def give_back(self):
        for tid, local in self._global_tail(self.n_lent):
            t = self.t.get(tid)
            if t is None or local >= t.capacity:
                continue
            t.lent.discard(local)
            for e in t.seed_order:
                if t.slot_of[e] < 0:
                    t.owner[local] = e
                    t.slot_of[e] = local
                    t.stamp[local] = self.clock
                    t.last_seen[e] = -1
                    break
        self.n_lent = 0

    # -- inspection --------------------------------------------------------------
    def snapshot(self, tid: int) -> dict:
        t = self.t[tid]
        return dict(slot_of=list(t.slot_of), owner=list(t.owner), stamp=list(t.stamp),
                    last_seen=list(t.last_seen), capacity=t.capacity - len(t.lent))

    def check_invariants(self):
        for tid, t in self.t.items():
            for s, e in enumerate(t.owner):
                if e >= 0:
                    assert t.slot_of[e] == s, (tid, s, e)
                    assert s not in t.lent
            for e, s in enumerate(t.slot_of):
                if s >= 0:
                    assert t.owner[s] == e, (tid, e, s)
                    assert t.last_seen[e] == -1
            assert sum(1 for e in t.owner if e >= 0) <= t.capacity - len(t.lent)
            assert all(st <= self.clock for st in t.stamp)
