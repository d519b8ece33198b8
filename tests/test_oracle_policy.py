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
    # slots are lent: nothing admitted and no sighting recorded
    assert p.snapshot(0)["last_seen"][0] == -1 and p.snapshot(1)["last_seen"][4] == -1
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


def _global_trace_oracle():
    p = PolicyOracle(n_experts=6, window=4, slots_per_tensor=2, n_tensors=2, global_pool=True)
    p.add_tensor(0, 2, [0, 1, 2, 3, 4, 5], n_seed=1)
    p.add_tensor(1, 1, [5, 4, 3, 2, 1, 0], n_seed=1)
    return p


def _owners(vals):
    return ["-" if v < 0 else str(v) for v in vals]


def test_hand_traced_global_pool(golden):
    rows = golden("policy_global_trace.txt")
    steps = [r for r in rows if len(r) == 8]
    cases = {r[0]: r[1:] for r in rows if len(r) == 5}
    assert len(steps) == 7 and set(cases) == {"preheat", "seed"}
    for case, (own_b, miss, own_r, stamp_r) in cases.items():
        p = _global_trace_oracle()
        for n, u0, u1, misses, owner, stamp, ls0, ls1 in steps:
            assert p.step(int(n), {0: _ints(u0), 1: _ints(u1)}) == _ints(misses)
            ps = p.pool_snapshot()
            assert ",".join(_owners(ps["owner"])) == owner
            assert ps["stamp"] == _ints(stamp)
            assert p.snapshot(0)["last_seen"] == _ints(ls0)
            assert p.snapshot(1)["last_seen"] == _ints(ls1)
            p.check_invariants()
        p.borrow(2)
        assert ",".join(_owners(p.pool_snapshot()["owner"])) == own_b
        assert p.step(2, {0: [1], 1: [2]}) == _ints(miss)
        # lent slots: nothing admitted, no sighting recorded
        assert p.snapshot(0)["last_seen"][1] == -1 and p.snapshot(1)["last_seen"][2] == -1
        p.check_invariants()
        counts = {0: [0, 3, 7, 0, 0, 0]} if case == "preheat" else None
        p.give_back(counts)
        ps = p.pool_snapshot()
        assert ",".join(_owners(ps["owner"])) == own_r and ps["stamp"] == _ints(stamp_r)
        p.check_invariants()


def test_hand_traced_preheat_per_tensor():
    # the borrow/return trace of policy_borrow_trace.txt, returned with the
    # prompt pass's layer-0 counts e1 = 2, e2 = 5 (others 0):
    # g3 -> t1 l1: t1 non-resident e0..e4, e2 (-5) first -> e2
    # g4 -> t0 l2: t0 non-resident e0, e2, e4, e5 -> e2
    # g5 -> t1 l2: t1 non-resident e0, e1, e3, e4 -> e1 (-2)
    p = PolicyOracle(n_experts=6, window=4, slots_per_tensor=3, n_tensors=2)
    p.add_tensor(0, 3, [3, 1, 0, 2, 4, 5])
    p.add_tensor(1, 3, [5, 4, 0, 1, 2, 3])
    p.borrow(3)
    p.step(4, {0: [0, 3], 1: [4]})
    p.give_back({0: [0, 2, 5, 0, 0, 0]})
    assert p.snapshot(0)["owner"] == [3, 1, 2] and p.snapshot(1)["owner"] == [5, 2, 1]
    assert p.snapshot(0)["stamp"] == [4, 0, 4] and p.snapshot(1)["stamp"] == [0, 4, 4]
    p.check_invariants()


def test_global_pool_of_one_tensor_is_the_per_tensor_policy():
    # with a single tensor the global arena order is the local slot order, so
    # both modes must agree step by step (the per-tensor mode is pinned by
    # the hand traces above)
    rng = np.random.default_rng(11)
    E, C = 40, 9
    seed = rng.permutation(E)
    a = PolicyOracle(n_experts=E, window=12, slots_per_tensor=C, n_tensors=1)
    b = PolicyOracle(n_experts=E, window=12, slots_per_tensor=C, n_tensors=1, global_pool=True)
    a.add_tensor(0, C, seed, n_seed=C - 2)
    b.add_tensor(0, C, seed, n_seed=C - 2)
    probs = synth.zipf_probs(E, 0.9)
    for step in range(300):
        n = int(rng.integers(1, 4))
        used = {0: rng.choice(E, size=int(rng.integers(1, 5)), replace=False, p=probs).tolist()}
        assert a.step(n, used) == b.step(n, used)
        if step in (100, 200):
            a.borrow(3), b.borrow(3)
            a.step(2, used), b.step(2, used)
            cnt = {0: rng.integers(0, 4, size=E).tolist()}
            a.give_back(cnt), b.give_back(cnt)
        sa, sb, pb = a.snapshot(0), b.snapshot(0), b.pool_snapshot()
        assert sa["slot_of"] == sb["slot_of"] and sa["last_seen"] == sb["last_seen"]
        assert [o if o >= 0 else -1 for o in sa["owner"]] == [k & 0xFFF if k >= 0 else -1 for k in pb["owner"]]
        assert sa["stamp"] == pb["stamp"]
        b.check_invariants()


def test_global_pool_invariants_and_misses_long_run():
    rng = np.random.default_rng(13)
    E, nt, spt = 32, 6, 6
    caps = [6, 3, 0, 5, 6, 2]
    p = PolicyOracle(n_experts=E, window=10, slots_per_tensor=spt, n_tensors=nt, global_pool=True)
    for t in range(nt):
        p.add_tensor(t, caps[t], rng.permutation(E), n_seed=max(0, caps[t] - 1))
    probs = synth.zipf_probs(E, 1.0)
    pool = sum(caps)
    cross = 0
    for step in range(500):
        n = int(rng.integers(1, 3))
        used = {t: rng.choice(E, size=int(rng.integers(1, 4)), replace=False, p=probs).tolist() for t in range(nt)}
        resident = {t: {e for e in range(E) if p.t[t].slot_of[e] >= 0} for t in range(nt)}
        before = list(p.g_owner)
        expect = sorted((t << 12) | e for t in range(nt) for e in set(used[t]) if e not in resident[t])
        assert p.step(n, used) == expect
        p.check_invariants()
        assert sum(1 for k in p.g_owner if k >= 0) <= pool
        # a slot changing hands between tensors is what the per-tensor pools cannot do
        cross += sum(1 for x, y in zip(before, p.g_owner) if x >= 0 and y >= 0 and (x >> 12) != (y >> 12))
        if step % 97 == 50:
            p.borrow(int(rng.integers(1, nt * spt)))
            p.step(1, used)
            p.check_invariants()
            p.give_back({0: rng.integers(0, 3, size=E).tolist(), 1: [0] * E})
            p.check_invariants()
    assert cross > 0
    # a tensor with no reserve of its own still gets pool slots
    assert any(g >= 0 for g in p.t[2].slot_of)
