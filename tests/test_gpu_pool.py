"""GPU parity of the shared expert pool (one arena of expert blocks for all
layers) and of prefill preheat (blocks lent to a prompt pass come back
holding the experts the pass used most), through the C ABI, against the
policy oracle: the whole pool (owner and stamp of every arena slot), every
tensor's table, slots and sightings after every promotion pass, and the
layer outputs on the way."""
import copy

import numpy as np
import pytest

import oracle
import quantized_expert_cache_gb300 as qec
import synth
from gpu_helpers import Model, check_layer_parity

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    qec.build.build()
    qec.load()


def _steps(m, n_steps, T_of, step0=0, lg_wl=None, check_every=0, counts=None):
    """Decode / prompt steps through the library and the oracle.  The experts
    each tensor reads (and the prompt-pass use counts) come from the oracle's
    own top-k; the library's indices must equal them."""
    for i in range(n_steps):
        step, T = step0 + i, T_of(i)
        used = {}
        for layer in range(m.L):
            x = m.wl.x(layer, step, T)
            lg = (lg_wl or m.wl).logits(layer, step, T)
            idx, w = m.route(lg)
            y = m.forward(layer, x, idx, w)
            idx_o, _ = oracle.topk(lg, m.k)
            idx_np = idx.cpu().numpy()
            assert np.array_equal(idx_np, idx_o)
            if counts is not None:
                counts[layer] = counts.get(layer, np.zeros(m.E, np.int64)) + np.bincount(idx_o.ravel(), minlength=m.E)
            for kind in range(3):
                used[layer * 3 + kind] = idx_o.ravel().tolist()
            if check_every and i % check_every == 0:
                torch.cuda.synchronize()
                check_layer_parity(m, layer, x, lg, y.cpu().numpy(), idx_np, w.cpu().numpy())
        qec.cache_step(m.ctx, T)
        m.policy.step(T, used)
        yield i


def _assert_state(m):
    G = 3 * m.L * m.spt
    ps = qec.moe_pool_snapshot(m.ctx, G)
    if m.global_pool:
        o = m.policy.pool_snapshot()
        assert ps["owner"].tolist() == o["owner"]
        assert ps["stamps"].tolist() == o["stamp"]
    for tid in range(3 * m.L):
        snap = qec.moe_cache_snapshot(m.ctx, tid, m.E, m.spt)
        o = m.policy.snapshot(tid)
        assert snap["slot_of"].tolist() == o["slot_of"], tid
        assert snap["last_seen"].tolist() == o["last_seen"], tid
        assert np.array_equal(snap["tbl"], m.expected_tbl(tid)), tid
        if not m.global_pool:
            lent = m.policy.t[tid].lent
            assert snap["owner"].tolist()[: len(o["owner"])] == [(-1 if s in lent else e)
                                                                   for s, e in enumerate(o["owner"])], tid
            # the arena view agrees with the per-tensor one
            for s, e in enumerate(o["owner"]):
                g = s * 3 * m.L + tid
                assert ps["owner"][g] == (-1 if (s in lent or e < 0) else (tid << 12) | e)
                assert ps["stamps"][g] == o["stamp"][s]


def _stats_match(m):
    st = qec.moe_stats(m.ctx)
    for k in ("admissions", "evictions", "misses", "hits"):
        assert st[k] == m.policy.stats[k], k
    return st


def _cross_layer_moves(before, after):
    return sum(1 for a, b in zip(before, after) if a >= 0 and b >= 0 and (a >> 12) != (b >> 12))


def test_global_pool_state_bit_exact_every_step():
    # three layers with unequal reserves (8, 2, 0 slots per tensor): the
    # shared pool lets the busy layers take blocks from the others
    m = Model(H=256, F=256, E=32, k=4, L=3, capacity=[8, 2, 0], max_tokens=4, window=8, zipf_s=1.1,
              slots_per_tensor=8, global_pool=True)
    try:
        G = 3 * m.L * m.spt
        moves = 0
        before = qec.moe_pool_snapshot(m.ctx, G)["owner"].tolist()
        for _ in _steps(m, 70, lambda s: 1 if s % 5 else 3, check_every=23):
            _assert_state(m)
            m.policy.check_invariants()
            after = qec.moe_pool_snapshot(m.ctx, G)["owner"].tolist()
            moves += _cross_layer_moves(before, after)
            before = after
        st = _stats_match(m)
        assert st["admissions"] > 0 and st["evictions"] > 0
        assert moves > 0, "no block changed layers"
        # layer 2 has no reserve of its own, yet holds experts
        assert any(s >= 0 for s in m.policy.snapshot(6)["slot_of"])
    finally:
        m.close()


def test_global_pool_max_swaps():
    m = Model(H=256, F=256, E=64, k=8, L=2, capacity=[10, 4], max_tokens=2, window=64, max_swaps=3,
              zipf_s=0.9, slots_per_tensor=10, global_pool=True)
    try:
        for _ in _steps(m, 30, lambda s: 2):
            _assert_state(m)
        _stats_match(m)
    finally:
        m.close()


@pytest.mark.parametrize("global_pool", [True, False])
def test_borrow_and_preheat_return_match_oracle(global_pool):
    m = Model(H=256, F=256, E=16, k=2, L=2, capacity=[6, 4], max_tokens=64, window=8, slots_per_tensor=6,
              global_pool=global_pool, preheat=True)
    # the prompt is routed by another popularity order than the seeding
    # table's, so the experts it uses most are not simply the seed-order ones
    prompt = synth.Workload("prompt", m.H, m.E, m.k, m.F, m.L, routing="zipf", zipf_s=1.1, seed=7)
    try:
        for _ in _steps(m, 6, lambda s: 1):
            pass
        qec.moe_pool_borrow(m.ctx, 13)
        m.policy.borrow(13)
        _assert_state(m)
        counts = {}
        # a prompt-sized step and a small one while slots are lent: misses
        # logged, nothing admitted, assignments counted
        for _ in _steps(m, 2, lambda s: (40, 3)[s], step0=100, lg_wl=prompt, check_every=1, counts=counts):
            _assert_state(m)
        seed_refill = copy.deepcopy(m.policy)
        seed_refill.give_back()
        qec.moe_pool_return(m.ctx)
        m.policy.give_back({l: c.tolist() for l, c in counts.items()})
        m.policy.check_invariants()
        _assert_state(m)
        if global_pool:
            assert m.policy.pool_snapshot()["owner"] != seed_refill.pool_snapshot()["owner"], \
                "preheat made no difference: the test does not exercise the use counts"
        else:
            assert any(m.policy.snapshot(t)["owner"] != seed_refill.snapshot(t)["owner"] for t in range(6))
        for _ in _steps(m, 8, lambda s: 1, step0=200, check_every=4):
            _assert_state(m)
        _stats_match(m)
        # counts were cleared by the return: a second borrow / return without
        # forwards refills by seed order
        qec.moe_pool_borrow(m.ctx, 5)
        m.policy.borrow(5)
        qec.moe_pool_return(m.ctx)
        m.policy.give_back()
        _assert_state(m)
    finally:
        m.close()


def test_pool_mode_errors():
    ctx = qec.moe_layer_init(256, 256, 8, 2, 1, 4, 4, stream=torch.cuda.current_stream().cuda_stream)
    try:
        wl = synth.Workload("t", 256, 8, 2, 256, 1, seed=3)
        qec.register_expert_tensor(ctx, 0, 0, wl.expert_tensor(0, 0), 256, 256, 4, None, 2)
        with pytest.raises(qec.MoeError) as ex:
            qec.moe_set_global_pool(ctx, True)
        assert ex.value.code == -7
        qec.moe_set_preheat(ctx, True)
        for kind in (1, 2):
            r, c = wl.tensor_shapes[kind]
            qec.register_expert_tensor(ctx, 0, kind, wl.expert_tensor(0, kind), r, c, 4, None, 2)
        qec.moe_pool_borrow(ctx, 2)
        with pytest.raises(qec.MoeError) as ex:
            qec.moe_set_preheat(ctx, False)
        assert ex.value.code == -7
        qec.moe_pool_return(ctx)
    finally:
        qec.moe_destroy(ctx)


def test_cache_reset_switches_pool_mode_and_restarts_from_seeding():
    m = Model(H=256, F=256, E=32, k=4, L=2, capacity=[8, 3], max_tokens=4, window=8, zipf_s=1.0,
              slots_per_tensor=8)
    try:
        for gp in (False, True, True, False):
            if gp or m.policy.clock:
                m.reset(gp)
            _assert_state(m)
            st = qec.moe_stats(m.ctx)
            assert st["hits"] == st["misses"] == st["admissions"] == st["steps"] == 0
            for _ in _steps(m, 25, lambda s: 1 if s % 4 else 2, check_every=12):
                _assert_state(m)
            _stats_match(m)
    finally:
        m.close()


@pytest.mark.parametrize("global_pool", [False, True])
def test_upload_overlap_same_state_and_outputs(global_pool):
    # per-layer upload events instead of one wait for the whole promotion
    # pass: the cache state after every step and the layer outputs are the
    # oracle's, as without the overlap
    m = Model(H=256, F=256, E=32, k=4, L=3, capacity=[8, 4, 6], max_tokens=4, window=8, zipf_s=1.0,
              slots_per_tensor=8, global_pool=global_pool)
    try:
        qec.moe_set_upload_overlap(m.ctx, True)
        for _ in _steps(m, 40, lambda s: 1 if s % 3 else 2, check_every=7):
            _assert_state(m)
        st = _stats_match(m)
        assert st["admissions"] > 0
        qec.moe_set_upload_overlap(m.ctx, False)
        for _ in _steps(m, 5, lambda s: 1, step0=100, check_every=2):
            _assert_state(m)
    finally:
        m.close()
