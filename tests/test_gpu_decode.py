"""GPU parity of the decode path against the oracle, through the C ABI:
router top-k, block dots, whole layers (hot and cold experts, ragged
shapes, several tiles, small and large batches), the miss log, stamps, and
the cache state after every promotion pass."""
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


def _ctx(E, k, H=256, F=256, L=1, spt=0, M=512):
    return qec.moe_layer_init(H, F, E, k, L, spt, M, stream=torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("E,k,T", [(8, 2, 4), (512, 8, 37), (128, 4, 300), (4096, 8, 5), (64, 32, 9), (1000, 3, 17)])
def test_route_topk_parity(E, k, T):
    ctx = _ctx(E, k, M=max(T, 1))
    try:
        lg = synth.normal(synth.key(11, 7, E, k, T), (T, E))
        lg[::2] = np.round(lg[::2] * 2) / 2  # ties
        lg[1, :3] = [0.0, -0.0, 0.0]
        d_lg = torch.from_numpy(lg).cuda()
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), dtype=torch.float32, device="cuda")
        qec.route_topk(ctx, d_lg, T, E, k, idx, w)
        torch.cuda.synchronize()
        idx_o, w_o = oracle.topk(lg, k)
        assert np.array_equal(idx.cpu().numpy(), idx_o)
        np.testing.assert_allclose(w.cpu().numpy(), w_o, rtol=1e-5, atol=1e-7)
    finally:
        qec.moe_destroy(ctx)


def test_block_dots_bit_exact_hot_and_cold():
    m = Model(H=256, F=512, E=8, k=2, L=1, capacity=4, max_tokens=4, routing="normal")
    try:
        rng = np.random.default_rng(3)
        for tid in (0, 1, 2):
            rows, cols = (512, 256) if tid < 2 else (256, 512)
            snap = qec.moe_cache_snapshot(m.ctx, tid, m.E, m.spt)
            hot = [e for e in range(8) if snap["slot_of"][e] >= 0]
            cold = [e for e in range(8) if snap["slot_of"][e] < 0]
            assert hot and cold
            for e in (hot[0], cold[-1]):
                qa = rng.integers(-127, 128, cols).astype(np.int8)
                d_qa = torch.from_numpy(qa).cuda()
                n_rows = 37
                out = torch.empty((n_rows, cols // 32), dtype=torch.int32, device="cuda")
                qec.moe_debug_block_dots(m.ctx, tid, e, 5, n_rows, d_qa, out)
                got = out.cpu().numpy()
                W = m.tensors[tid][e]
                ref = np.array([[oracle.block_dot(W[5 + r, b], qa[32 * b:32 * b + 32]) for b in range(cols // 32)]
                                for r in range(n_rows)])
                assert np.array_equal(got, ref)
    finally:
        m.close()


def test_tiny_layer_parity():
    """The tiny correctness workload: hidden 256, 8 experts, top-2, FFN 512,
    4 tokens, all experts resident, seed 0."""
    wl = synth.WORKLOADS["tiny"]
    m = Model(H=wl.hidden, F=wl.ffn, E=wl.n_experts, k=wl.top_k, L=1, capacity=wl.n_experts, max_tokens=4,
              routing="normal", seed=wl.seed)
    try:
        T = 4
        x, lg = wl.x(0, 0, T), wl.logits(0, 0, T)
        assert np.array_equal(x, m.wl.x(0, 0, T)) and np.array_equal(lg, m.wl.logits(0, 0, T))
        idx, w = m.route(lg)
        y = m.forward(0, x, idx, w)
        torch.cuda.synchronize()
        check_layer_parity(m, 0, x, lg, y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy())
        assert len(qec.miss_drain(m.ctx)) == 0
        for tid in range(3):
            snap = qec.moe_cache_snapshot(m.ctx, tid, m.E, m.spt)
            used = set(idx.cpu().numpy().ravel().tolist())
            for e in range(m.E):
                s = snap["slot_of"][e]
                assert snap["stamps"][s] == (T if e in used else 0)
    finally:
        m.close()


@pytest.mark.parametrize("H,F,E,k,T", [(512, 384, 64, 4, 1), (512, 384, 64, 4, 3), (512, 384, 64, 4, 8),
                                       (512, 384, 64, 4, 19), (512, 384, 64, 4, 33), (512, 384, 64, 4, 70),
                                       (640, 1440, 16, 3, 5), (640, 1440, 16, 3, 40), (2048, 1152, 64, 8, 1)])
def test_layer_parity_shapes_hot_and_cold(H, F, E, k, T):
    m = Model(H=H, F=F, E=E, k=k, L=2, capacity=E // 2, max_tokens=T, zipf_s=0.6)
    try:
        for layer in range(2):
            x, lg = m.wl.x(layer, 1, T), m.wl.logits(layer, 1, T)
            idx, w = m.route(lg)
            y = m.forward(layer, x, idx, w)
            torch.cuda.synchronize()
            idx_np = idx.cpu().numpy()
            check_layer_parity(m, layer, x, lg, y.cpu().numpy(), idx_np, w.cpu().numpy())
            # miss log: exactly the (tensor, expert) pairs read while cold
            used = sorted(set(idx_np.ravel().tolist()))
            expect = []
            for kind in range(3):
                tid = layer * 3 + kind
                slot_of = m.policy.snapshot(tid)["slot_of"]
                expect += [(tid << 12) | e for e in used if slot_of[e] < 0]
            got = qec.miss_drain(m.ctx)
            assert got.tolist() == sorted(expect)
            # stamps: resident used experts carry clock + T
            for kind in range(3):
                tid = layer * 3 + kind
                snap = qec.moe_cache_snapshot(m.ctx, tid, m.E, m.spt)
                for e in used:
                    s = snap["slot_of"][e]
                    if s >= 0:
                        assert snap["stamps"][s] == T
    finally:
        m.close()


def _run_steps(m, steps, T_of_step, check_every=0):
    n_alt = 0
    for step in range(steps):
        T = T_of_step(step)
        used = {}
        for layer in range(m.L):
            x, lg = m.wl.x(layer, step, T), m.wl.logits(layer, step, T)
            idx, w = m.route(lg)
            y = m.forward(layer, x, idx, w)
            idx_np = idx.cpu().numpy()
            for kind in range(3):
                used[layer * 3 + kind] = idx_np.ravel().tolist()
            if check_every and step % check_every == 0:
                torch.cuda.synchronize()
                n_alt += check_layer_parity(m, layer, x, lg, y.cpu().numpy(), idx_np, w.cpu().numpy())
        qec.cache_step(m.ctx, T)
        m.policy.step(T, used)
        yield step


def _assert_state(m):
    for tid in range(3 * m.L):
        snap = qec.moe_cache_snapshot(m.ctx, tid, m.E, m.spt)
        o = m.policy.snapshot(tid)
        assert snap["slot_of"].tolist() == o["slot_of"], tid
        assert snap["owner"].tolist()[: len(o["owner"])] == [(-1 if s in m.policy.t[tid].lent else e)
                                                               for s, e in enumerate(o["owner"])], tid
        assert snap["last_seen"].tolist() == o["last_seen"], tid
        assert snap["stamps"].tolist()[: len(o["stamp"])] == o["stamp"], tid
        assert np.array_equal(snap["tbl"], m.expected_tbl(tid)), tid


def test_cache_step_state_bit_exact_every_step():
    m = Model(H=256, F=256, E=32, k=4, L=2, capacity=8, max_tokens=4, window=8, zipf_s=1.1)
    try:
        for _ in _run_steps(m, 80, lambda s: 1 if s % 7 else 3, check_every=20):
            _assert_state(m)
            m.policy.check_invariants()
        st = qec.moe_stats(m.ctx)
        assert st["admissions"] == m.policy.stats["admissions"] > 0
        assert st["evictions"] == m.policy.stats["evictions"] > 0
        assert st["misses"] == m.policy.stats["misses"]
        assert st["hits"] == m.policy.stats["hits"]
    finally:
        m.close()


def test_cache_step_max_swaps_and_full_window():
    m = Model(H=256, F=256, E=64, k=8, L=1, capacity=16, max_tokens=2, window=64, max_swaps=2, zipf_s=0.9)
    try:
        for _ in _run_steps(m, 40, lambda s: 2):
            _assert_state(m)
    finally:
        m.close()


def test_borrow_and_return_match_oracle():
    m = Model(H=256, F=256, E=16, k=2, L=2, capacity=6, max_tokens=64, window=8, slots_per_tensor=6)
    try:
        for _ in _run_steps(m, 5, lambda s: 1):
            pass
        ws, nbytes = qec.moe_pool_borrow(m.ctx, 13)
        m.policy.borrow(13)
        lay = qec.moe_cache_layout(m.ctx, 0)
        assert ws == lay["pool_base"] + (6 * 6 - 13) * lay["slot_bytes"] and nbytes == 13 * lay["slot_bytes"]
        _assert_state(m)
        # a prefill-sized step while slots are lent: misses logged, nothing admitted
        for _ in _run_steps(m, 1, lambda s: 40, check_every=1):
            pass
        _assert_state(m)
        qec.moe_pool_return(m.ctx)
        m.policy.give_back()
        _assert_state(m)
        for _ in _run_steps(m, 6, lambda s: 1, check_every=3):
            _assert_state(m)
    finally:
        m.close()


def test_injected_upload_failure_rolls_back_consistently():
    m = Model(H=256, F=256, E=32, k=4, L=1, capacity=4, max_tokens=1, window=64)
    try:
        qec.moe_debug_fail_upload(m.ctx, 1)
        failed = False
        for step in range(40):
            x, lg = m.wl.x(0, step, 1), m.wl.logits(0, step, 1)
            idx, w = m.route(lg)
            m.forward(0, x, idx, w)
            try:
                qec.cache_step(m.ctx, 1)
            except qec.MoeError as ex:
                assert ex.code == -8 and not failed
                failed = True
            # whatever happened, the state is self-consistent
            for tid in range(3):
                snap = qec.moe_cache_snapshot(m.ctx, tid, m.E, m.spt)
                lay = qec.moe_cache_layout(m.ctx, tid)
                for e in range(m.E):
                    s = int(snap["slot_of"][e])
                    if s >= 0:
                        assert snap["owner"][s] == e
                        assert int(snap["tbl"][e]) == lay["pool_base"] + (s * 3 + tid) * lay["slot_bytes"]
                    else:
                        assert int(snap["tbl"][e]) == (lay["host_base"] + e * lay["slot_bytes"]) | 1
        assert failed
        # outputs after the fault still match the oracle
        x, lg = m.wl.x(0, 99, 1), m.wl.logits(0, 99, 1)
        idx, w = m.route(lg)
        y = m.forward(0, x, idx, w)
        torch.cuda.synchronize()
        check_layer_parity(m, 0, x, lg, y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy())
    finally:
        m.close()


def test_probe_host_read_and_not_pinned():
    buf = torch.empty(64 << 20, dtype=torch.uint8).pin_memory()
    gbs, cgbs = qec.moe_probe_host_read(buf.data_ptr(), buf.numel(), iters=3)
    assert gbs > 1.0 and cgbs > 1.0
    pageable = np.zeros(1 << 20, np.uint8)
    with pytest.raises(qec.MoeError) as ei:
        qec.moe_probe_host_read(pageable.ctypes.data, pageable.nbytes, iters=1)
    assert ei.value.code == -4


@pytest.mark.parametrize("H,F,E,k,T", [(2048, 1152, 512, 8, 1), (512, 384, 64, 4, 3), (640, 1440, 128, 4, 8),
                                       (512, 384, 128, 4, 32), (256, 512, 8, 2, 40)])
def test_routed_forward_matches_route_then_forward(H, F, E, k, T):
    m = Model(H=H, F=F, E=E, k=k, L=1, capacity=E // 2, max_tokens=T, zipf_s=0.8)
    try:
        x, lg = m.wl.x(0, 4, T), m.wl.logits(0, 4, T)
        lg[0, :4] = 1.5  # ties inside the top-k
        idx_ref, w_ref = m.route(lg)
        y_ref = m.forward(0, x, idx_ref, w_ref)
        torch.cuda.synchronize()
        y_ref = y_ref.cpu().numpy()
        qec.miss_drain(m.ctx)
        d_x, d_lg = m.dev(x), m.dev(lg)
        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, k), device="cuda")
        y = torch.empty((T, H), device="cuda")
        qec.moe_ffn_forward_routed(m.ctx, 0, d_x, d_lg, T, idx, w, y)
        torch.cuda.synchronize()
        assert torch.equal(idx, idx_ref)
        np.testing.assert_allclose(w.cpu().numpy(), w_ref.cpu().numpy(), rtol=1e-6, atol=1e-8)
        check_layer_parity(m, 0, x, lg, y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy())
        np.testing.assert_allclose(y.cpu().numpy(), y_ref, rtol=1e-5, atol=1e-6)
    finally:
        m.close()


def test_cache_step_poll_timeout_keeps_the_context_usable():
    """Failure detection without a fault: a bounded busy kernel keeps the
    stream busy past cache_step's host poll limit; the step reports
    MOE_ERR_TIMEOUT and changes nothing, and once the device is done the
    retried step is exactly the oracle's."""
    m = Model(H=256, F=256, E=16, k=2, L=1, capacity=4, max_tokens=2, window=8, poll_timeout_ms=30)
    try:
        for _ in _run_steps(m, 6, lambda s: 1):
            pass
        _assert_state(m)
        before = qec.moe_stats(m.ctx)
        x, lg = m.wl.x(0, 50, 1), m.wl.logits(0, 50, 1)
        idx, w = m.route(lg)
        m.forward(0, x, idx, w)
        qec.moe_debug_busy(m.ctx, 400000)  # 0.4 s, far past the 30 ms poll limit
        with pytest.raises(qec.MoeError) as ex:
            qec.cache_step(m.ctx, 1)
        assert ex.value.code == -5
        torch.cuda.synchronize()  # the busy kernel ends by itself
        assert qec.moe_stats(m.ctx) == before
        qec.cache_step(m.ctx, 1)
        used = idx.cpu().numpy().ravel().tolist()
        m.policy.step(1, {kd: used for kd in range(3)})
        _assert_state(m)
        st = qec.moe_stats(m.ctx)
        assert st["steps"] == before["steps"] + 1 and st["misses"] == m.policy.stats["misses"]
    finally:
        m.close()


@pytest.mark.parametrize("T", [1, 40])
def test_bad_expert_id_is_reported_once_and_the_context_recovers(T):
    """An expert id outside [0, E) is caught by the kernels' own range checks
    (read as expert 0, error bit set); the next promotion pass reports
    MOE_ERR_FAULT once and clears it, and later steps are normal."""
    m = Model(H=256, F=256, E=16, k=2, L=1, capacity=4, max_tokens=40, window=8)
    try:
        x, lg = m.wl.x(0, 7, T), m.wl.logits(0, 7, T)
        idx, w = m.route(lg)
        bad = idx.clone()
        bad[0, 1] = m.E + 3
        m.forward(0, x, bad, w)
        with pytest.raises(qec.MoeError) as ex:
            qec.cache_step(m.ctx, T)
        assert ex.value.code == -8 and "expert id" in str(ex.value)
        y = m.forward(0, x, idx, w)
        torch.cuda.synchronize()
        check_layer_parity(m, 0, x, lg, y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy())
        qec.cache_step(m.ctx, T)  # no error left
    finally:
        m.close()
