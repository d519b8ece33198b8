"""Pins of the policy oracle: hand-traced sequences (tests/golden), invariants
after every step of long random runs, and a brute-force re-derivation of the
miss sets from the routing and the resident sets."""
import numpy as np

import synth
from oracle import PolicyOracle


def _ints(s):
    return [] if s in ("-", "") else [int(v) for v in s.split(",")]


def test_hand_traced_sequence(golden):
    p = PolicyOracle(n_experts=8, window=4)
    p.add_tensor(0, capacity=2, seed_order=range(8), n_seed=2)
    for n, used, misses, owner, stamp, last_seen in golden("policy_trace.txt"):
        got = p.step(int(n), {0: _ints(used)})
        snap = p.snapshot(0)
        assert got == _ints(misses)
        assert snap["owner"] == _ints(owner)
        assert snap["stamp"] == _ints(stamp)
        assert snap["last_seen"] == _ints(last_seen)
        p.check_invariants()


def test_hand_traced_max_swaps():
    # same trace as the golden file up to step 10, then the last step with a
    # limit of one admission per step: e0 is admitted, e5 keeps its sighting
    rows = []
    import os
    from conftest import read_golden
    rows = read_golden("policy_trace.txt")
    p = PolicyOracle(n_experts=8, window=4, max_swaps_per_step=1)
    p.add_tensor(0, capacity=2, seed_order=range(8), n_seed=2)
    for n, used, *_ in rows[:-1]:
        p.step(int(n), {0: _ints(used)})
    p.step(1, {0: [0, 5]})
    s = p.snapshot(0)
    assert s["owner"] == [3, 0] and s["stamp"] == [9, 12]
    assert s["last_seen"][5] == 11 and s["last_seen"][0] == -1


def test_hand_traced_borrow_return(golden):
    rows = golden("policy_borrow_trace.txt")
    p = PolicyOracle(n_experts=6, window=4, slots_per_tensor=3, n_tensors=2)
    p.add_tensor(0, 3, [3, 1, 0, 2, 4, 5])
    p.add_tensor(1, 3, [5, 4, 0, 1, 2, 3])
    p.borrow(3)

    def owners(tid):
        s = p.snapshot(tid)
        lent = p.t[tid].lent
        return ["-" if (i in lent or e < 0) else str(e) for i, e in enumerate(s["owner"])]

    for tid, ob, *_ in rows:
        assert ",".join(owners(int(tid))) == ob
    misses = p.step(4, {0: [0, 3], 1: [4]})
    assert misses == [0, (1 << 12) | 4]
    for tid, _, oa, sa, *_ in rows:
        assert ",".join(owners(int(tid))) == oa
        assert p.snapshot(int(tid))["stamp"] == _ints(sa)
    p.give_back()
    for tid, _, _, _, orr, sr in rows:
        s = p.snapshot(int(tid))
        assert s["owner"] == _ints(orr) and s["stamp"] == _ints(sr)
    p.check_invariants()


def test_invariants_and_brute_force_misses_long_run():
    rng = np.random.default_rng(5)
    E, n_t = 64, 3
    p = PolicyOracle(n_experts=E, window=16)
    caps = [8, 16, 5]
    for t in range(n_t):
        p.add_tensor(t, caps[t], rng.permutation(E), n_seed=caps[t] - (t == 1))
    for step in range(400):
        n = int(rng.integers(1, 4))
        used = {t: rng.choice(E, size=int(rng.integers(1, 6)), replace=False,
                              p=synth.zipf_probs(E, 1.1)).tolist() for t in range(n_t)}
        resident = {t: {e for e in range(E) if p.t[t].slot_of[e] >= 0} for t in range(n_t)}
        expect = sorted((t << 12) | e for t in range(n_t) for e in set(used[t]) if e not in resident[t])
        assert p.step(n, used) == expect
        p.check_invariants()
        for t in range(n_t):
            for e in set(used[t]):
                s = p.t[t].slot_of[e]
                if s >= 0:
                    assert p.t[t].stamp[s] == p.clock or e not in resident[t]


def test_admission_needs_second_sighting_within_window():
    p = PolicyOracle(n_experts=4, window=64)
    p.add_tensor(0, 1, [0, 1, 2, 3])
    p.step(1, {0: [1]})
    assert p.t[0].slot_of[1] == -1
    for _ in range(62):
        p.step(1, {0: [0]})
    # second sighting 63 tokens after the first: inside the window
    p.step(1, {0: [1]})
    assert p.t[0].slot_of[1] == 0
    q = PolicyOracle(n_experts=4, window=64)
    q.add_tensor(0, 1, [0, 1, 2, 3])
    q.step(1, {0: [1]})
    for _ in range(63):
        q.step(1, {0: [0]})
    # 64 tokens apart: outside the window, becomes a new first sighting
    q.step(1, {0: [1]})
    assert q.t[0].slot_of[1] == -1 and q.t[0].last_seen[1] == q.clock
