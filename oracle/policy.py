"""ORACLE (test infrastructure only): admission / eviction policy of the
HBM expert pool, per tensor or global across layers.

Sources (page titles and sections):
- Zapdev-labs/a6000-custom-kernels, the pointer-table paragraph: each expert
  tensor has its own table, pool and stamp array; cold reads are logged as
  (tensor_id << 12 | expert); between decode steps a promotion pass moves an
  expert into a free pool slot on its second miss, choosing victims by a scan
  of the stamps; pools start from a routing-frequency table.
- neurall/llama.cpp, "How it works", Expert cache: an expert that missed is
  admitted only when it missed again inside a 64-token window; instead of a
  fixed number of blocks per layer, every layer draws on one shared pool;
  the prompt pass borrows expert blocks and gives them back afterwards,
  refilled with the model's globally hot experts and with experts that the
  prompt pass itself needed (prefill preheat); the features table measures
  both (global expert pool; prefill preheat).

State per tensor t: slot_of[e] (-1 = cold) and last_seen[e] (-1 = no
sighting).  Slots: per-tensor mode keeps owner[slot] (-1 = free) and
stamp[slot] per tensor with local slot ids; global mode keeps one
owner[g] = (t << 12 | e) and stamp[g] for every arena slot g, and slot_of[e]
holds g.  One clock for all.

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
- per-tensor mode searches the missing tensor's own slots (local order);
  global mode searches every slot of the pool in arena order g, whichever
  tensor holds it, so an admission may evict another layer's expert;
- the placed expert gets stamp = clock and last_seen = -1; an evicted
  expert's sighting history starts empty (last_seen = -1);
- arena layout: global slot g is local slot g // n_tensors of tensor
  g % n_tensors; a tensor registered with capacity C contributes its local
  slots 0..C-1 to the pool (global mode: the pool is the union of those);
- seeding puts seed_order[0..n_seed) into local slots 0..n_seed-1, stamps 0;
- borrow(n) lends the n highest global slots (their experts are evicted; in
  per-tensor mode their tensors' capacities shrink); while slots are lent a
  step advances the clock, stamps hits and logs misses but admits nothing;
- give_back() returns them and refills each returned pool slot, in ascending
  global order, with the best non-resident candidate: per-tensor mode takes
  the slot's own tensor's experts, global mode every registered tensor's;
  candidates rank by (use count in the prompt pass, descending; rank in the
  tensor's seed order, ascending; tensor id, ascending).  Use counts are the
  (token, expert) assignments of each layer routed while slots were lent,
  shared by the layer's gate, up and down tensors; without preheat they are
  all 0, which leaves the seed-order (global hotness) refill.  The refilled
  slot gets stamp = clock.
"""
from __future__ import annotations

from dataclasses import dataclass, field


@dataclass
class _Tensor:
    capacity: int
    seed_order: list
    rank: list
    slot_of: list
    owner: list
    stamp: list
    last_seen: list
    lent: set = field(default_factory=set)  # local slots lent to a prefill pass


class PolicyOracle:
    def __init__(self, n_experts: int, window: int = 64, max_swaps_per_step: int = 0,
                 slots_per_tensor: int | None = None, n_tensors: int | None = None,
                 global_pool: bool = False):
        self.E = n_experts
        self.window = window
        self.max_swaps = max_swaps_per_step
        self.clock = 0
        self.t: dict[int, _Tensor] = {}
        self.slots_per_tensor = slots_per_tensor
        self.n_tensors = n_tensors
        self.n_lent = 0
        self.global_pool = global_pool
        if global_pool:
            assert slots_per_tensor is not None and n_tensors is not None, "global pool needs the arena layout"
            G = slots_per_tensor * n_tensors
            self.g_owner = [-1] * G   # (t << 12 | e) or -1
            self.g_stamp = [0] * G
            self.g_pool = [False] * G
            self.g_lent = [False] * G
        self.stats = dict(hits=0, misses=0, admissions=0, evictions=0)

    def _g(self, tid: int, local: int) -> int:
        return local * self.n_tensors + tid

    # -- registration ------------------------------------------------------
    def add_tensor(self, tid: int, capacity: int, seed_order, n_seed: int | None = None):
        seed_order = [int(e) for e in seed_order]
        if n_seed is None:
            n_seed = min(capacity, len(seed_order))
        assert 0 <= n_seed <= capacity <= self.E
        assert len(set(seed_order)) == len(seed_order)
        rank = [self.E] * self.E
        for r, e in enumerate(seed_order):
            rank[e] = r
        t = _Tensor(capacity, seed_order, rank, [-1] * self.E, [-1] * capacity, [0] * capacity, [-1] * self.E)
        if self.global_pool:
            assert capacity <= self.slots_per_tensor and 0 <= tid < self.n_tensors
            for s in range(capacity):
                self.g_pool[self._g(tid, s)] = True
            for s in range(n_seed):
                g = self._g(tid, s)
                t.slot_of[seed_order[s]] = g
                self.g_owner[g] = (tid << 12) | seed_order[s]
        else:
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
                    if self.global_pool:
                        self.g_stamp[s] = self.clock
                    else:
                        t.stamp[s] = self.clock
                    self.stats["hits"] += 1
                else:
                    misses.append((tid << 12) | e)
        misses.sort()
        self.stats["misses"] += len(misses)
        if self.n_lent == 0:
            self._admit(misses)
        return misses

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
            if self.global_pool:
                g = self._pick_global()
                if g is None:
                    continue
                self._evict_global(g)
                self._place_global(g, tid, e)
            else:
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
        usable = [s for s in range(t.capacity) if s not in t.lent]
        for s in usable:
            if t.owner[s] < 0:
                return s
        best = None
        for s in usable:
            if t.stamp[s] < self.clock and (best is None or t.stamp[s] < t.stamp[best]):
                best = s
        return best

    def _pick_global(self):
        usable = [g for g in range(len(self.g_owner)) if self.g_pool[g] and not self.g_lent[g]]
        for g in usable:
            if self.g_owner[g] < 0:
                return g
        best = None
        for g in usable:
            if self.g_stamp[g] < self.clock and (best is None or self.g_stamp[g] < self.g_stamp[best]):
                best = g
        return best

    def _evict_global(self, g: int):
        key = self.g_owner[g]
        if key >= 0:
            vt = self.t[key >> 12]
            vt.slot_of[key & 0xFFF] = -1
            vt.last_seen[key & 0xFFF] = -1
            self.g_owner[g] = -1
            self.stats["evictions"] += 1

    def _place_global(self, g: int, tid: int, e: int):
        self.g_owner[g] = (tid << 12) | e
        self.t[tid].slot_of[e] = g
        self.t[tid].last_seen[e] = -1
        self.g_stamp[g] = self.clock

    # -- borrow / return around a prefill pass -------------------------------
    def _global_tail(self, n: int):
        nt, spt = self.n_tensors, self.slots_per_tensor
        assert nt is not None and spt is not None, "borrow needs the global slot layout"
        G = nt * spt
        assert 0 <= n <= G
        return list(range(G - n, G))

    def borrow(self, n: int):
        assert self.n_lent == 0
        for g in self._global_tail(n):
            if self.global_pool:
                self._evict_global(g)
                self.g_lent[g] = True
                continue
            tid, local = g % self.n_tensors, g // self.n_tensors
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

    def _rank_key(self, tid: int, e: int, use_counts):
        c = 0 if use_counts is None else int(use_counts[tid // 3][e])
        return (-c, self.t[tid].rank[e], tid)

    def give_back(self, use_counts=None):
        """use_counts: None (refill by seed order) or, per layer, the E
        assignment counts of the prompt pass (prefill preheat)."""
        tail = self._global_tail(self.n_lent)
        if self.global_pool:
            cands = sorted(((tid, e) for tid in self.t for e in range(self.E)),
                           key=lambda te: self._rank_key(te[0], te[1], use_counts))
            pos = 0
            for g in tail:
                self.g_lent[g] = False
                if not self.g_pool[g]:
                    continue
                while pos < len(cands) and self.t[cands[pos][0]].slot_of[cands[pos][1]] >= 0:
                    pos += 1
                if pos == len(cands):
                    continue
                tid, e = cands[pos]
                self._place_global(g, tid, e)
            self.n_lent = 0
            return
        for g in tail:
            tid, local = g % self.n_tensors, g // self.n_tensors
            t = self.t.get(tid)
            if t is None or local >= t.capacity:
                continue
            t.lent.discard(local)
            free = [e for e in range(self.E) if t.slot_of[e] < 0]
            if not free:
                continue
            e = min(free, key=lambda v: self._rank_key(tid, v, use_counts))
            t.owner[local] = e
            t.slot_of[e] = local
            t.stamp[local] = self.clock
            t.last_seen[e] = -1
        self.n_lent = 0

    # -- inspection --------------------------------------------------------------
    def snapshot(self, tid: int) -> dict:
        t = self.t[tid]
        if self.global_pool:
            return dict(slot_of=list(t.slot_of), last_seen=list(t.last_seen))
        return dict(slot_of=list(t.slot_of), owner=list(t.owner), stamp=list(t.stamp),
                    last_seen=list(t.last_seen), capacity=t.capacity - len(t.lent))

    def pool_snapshot(self) -> dict:
        """Global mode: owner key (or -1) and stamp of every arena slot."""
        assert self.global_pool
        return dict(owner=list(self.g_owner), stamp=list(self.g_stamp))

    def check_invariants(self):
        if self.global_pool:
            n_res = 0
            for g, key in enumerate(self.g_owner):
                if key >= 0:
                    n_res += 1
                    assert self.g_pool[g] and not self.g_lent[g], g
                    assert self.t[key >> 12].slot_of[key & 0xFFF] == g, (g, key)
            for tid, t in self.t.items():
                for e, g in enumerate(t.slot_of):
                    if g >= 0:
                        assert self.g_owner[g] == (tid << 12) | e, (tid, e, g)
                        assert t.last_seen[e] == -1
            assert n_res <= sum(1 for g in range(len(self.g_pool)) if self.g_pool[g] and not self.g_lent[g])
            assert all(st <= self.clock for st in self.g_stamp)
            return
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
