"""GPU parity of the shared expert (one expert every token runs next to its
routed ones, weight 1, inside the same launches) through the C ABI, against
the oracle: whole layers at decode and prompt sizes with hot and cold routed
experts (mat-vec kernels and the grouped GEMM), the shared expert's block
dots, the miss log (the shared expert is never cold), the cache state after
every promotion pass, and the Q8_0 / Q5_0 formats."""
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


@pytest.mark.parametrize("H,F,E,k,T", [(256, 512, 8, 2, 4), (512, 384, 64, 4, 1), (512, 384, 64, 4, 9),
                                       (512, 384, 64, 4, 33), (512, 384, 64, 4, 100), (640, 1440, 16, 3, 40),
                                       (2048, 1152, 64, 8, 1)])
def test_shared_expert_layer_parity_hot_and_cold(H, F, E, k, T):
    m = Model(H=H, F=F, E=E, k=k, L=2, capacity=E // 2, max_tokens=T, zipf_s=0.6, shared=True)
    try:
        for layer in range(2):
            x, lg = m.wl.x(layer, 1, T), m.wl.logits(layer, 1, T)
            idx, w = m.route(lg)
            y = m.forward(layer, x, idx, w)
            torch.cuda.synchronize()
            idx_np = idx.cpu().numpy()
            check_layer_parity(m, layer, x, lg, y.cpu().numpy(), idx_np, w.cpu().numpy())
            # only routed experts are ever cold
            used = sorted(set(idx_np.ravel().tolist()))
            expect = [((layer * 3 + kd) << 12) | e for kd in range(3) for e in used
                      if m.policy.snapshot(layer * 3 + kd)["slot_of"][e] < 0]
            assert qec.miss_drain(m.ctx).tolist() == sorted(expect)
    finally:
        m.close()


def test_shared_expert_block_dots_and_errors():
    m = Model(H=256, F=512, E=8, k=2, L=1, capacity=4, max_tokens=4, routing="normal", shared=True)
    try:
        rng = np.random.default_rng(8)
        for tid in range(3):
            cols = 256 if tid < 2 else 512
            qa = rng.integers(-127, 128, cols).astype(np.int8)
            out = torch.empty((9, cols // 32), dtype=torch.int32, device="cuda")
            qec.moe_debug_block_dots(m.ctx, tid, m.E, 3, 9, torch.from_numpy(qa).cuda(), out)
            W = m.shared[(0, tid)]
            ref = np.array([[oracle.block_dot(W[3 + r, b], qa[32 * b:32 * b + 32]) for b in range(cols // 32)]
                            for r in range(9)])
            assert np.array_equal(out.cpu().numpy(), ref)
        with pytest.raises(qec.MoeError) as ex:
            qec.register_shared_expert(m.ctx, 0, 0, m.shared[(0, 0)], 512, 256)
        assert ex.value.code == -1
    finally:
        m.close()
    # a context without shared experts refuses one; one with them needs all three first
    ctx = qec.moe_layer_init(256, 256, 8, 2, 1, 4, 4, stream=torch.cuda.current_stream().cuda_stream)
    try:
        with pytest.raises(qec.MoeError) as ex:
            qec.register_shared_expert(ctx, 0, 0, np.zeros((256, 8, 18), np.uint8), 256, 256)
        assert ex.value.code == -7
    finally:
        qec.moe_destroy(ctx)


def test_shared_expert_cache_steps_and_borrow():
    m = Model(H=512, F=384, E=32, k=4, L=2, capacity=8, max_tokens=48, window=8, zipf_s=1.1, shared=True,
              slots_per_tensor=8)
    try:
        for step in range(24):
            T = 1 if step % 5 else 3
            used = {}
            for layer in range(m.L):
                x, lg = m.wl.x(layer, step, T), m.wl.logits(layer, step, T)
                idx, w = m.route(lg)
                y = m.forward(layer, x, idx, w)
                idx_np = idx.cpu().numpy()
                if step % 8 == 0:
                    torch.cuda.synchronize()
                    check_layer_parity(m, layer, x, lg, y.cpu().numpy(), idx_np, w.cpu().numpy())
                for kd in range(3):
                    used[layer * 3 + kd] = idx_np.ravel().tolist()
            qec.cache_step(m.ctx, T)
            m.policy.step(T, used)
            for tid in range(3 * m.L):
                snap = qec.moe_cache_snapshot(m.ctx, tid, m.E, m.spt)
                o = m.policy.snapshot(tid)
                assert snap["slot_of"].tolist() == o["slot_of"] and snap["last_seen"].tolist() == o["last_seen"]
                assert np.array_equal(snap["tbl"], m.expected_tbl(tid))
        st = qec.moe_stats(m.ctx)
        assert st["admissions"] == m.policy.stats["admissions"] > 0
        assert st["hits"] == m.policy.stats["hits"] and st["misses"] == m.policy.stats["misses"]
        # a prompt pass through the grouped GEMM with lent slots (staging)
        qec.moe_pool_borrow(m.ctx, 10)
        m.policy.borrow(10)
        x, lg = m.wl.x(1, 500, 48), m.wl.logits(1, 500, 48)
        idx, w = m.route(lg)
        y = m.forward(1, x, idx, w)
        torch.cuda.synchronize()
        check_layer_parity(m, 1, x, lg, y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy())
        qec.moe_pool_return(m.ctx)
        m.policy.give_back()
        qec.moe_cache_reset(m.ctx, False)
        x, lg = m.wl.x(0, 600, 2), m.wl.logits(0, 600, 2)
        idx, w = m.route(lg)
        y = m.forward(0, x, idx, w)
        torch.cuda.synchronize()
        m.reset(False)
        check_layer_parity(m, 0, x, lg, y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy())
    finally:
        m.close()


@pytest.mark.parametrize("fmt", [qec.FMT_Q8_0, qec.FMT_Q5_0, qec.FMT_Q4_K, qec.FMT_Q6_K, qec.FMT_Q5_K])
def test_shared_expert_other_formats(fmt):
    F = 512 if fmt in (qec.FMT_Q4_K, qec.FMT_Q6_K, qec.FMT_Q5_K) else 384
    m = Model(H=512, F=F, E=16, k=4, L=1, capacity=8, max_tokens=40, zipf_s=0.8, shared=True, weight_format=fmt)
    try:
        for T in (1, 5, 40):
            x, lg = m.wl.x(0, T, T), m.wl.logits(0, T, T)
            idx, w = m.route(lg)
            y = m.forward(0, x, idx, w)
            torch.cuda.synchronize()
            check_layer_parity(m, 0, x, lg, y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy())
            qec.miss_drain(m.ctx)
    finally:
        m.close()


@pytest.mark.parametrize("fmt", [qec.FMT_Q4_0, qec.FMT_Q8_0, qec.FMT_Q5_0, qec.FMT_Q4_K, qec.FMT_Q6_K, qec.FMT_Q5_K])
def test_shared_expert_routed_single_token(fmt):
    """One routed token per layer through the single-launch layer, whose last
    pick is the shared expert (its weights requested at kernel entry, before
    the routing is done): ids and weights against the oracle's top-k, x and h
    codes and y against the oracle's layer with the shared expert, the cache
    state and counts after every promotion pass, in every weight format."""
    F = 512 if fmt in (qec.FMT_Q4_K, qec.FMT_Q6_K, qec.FMT_Q5_K) else 384
    m = Model(H=512, F=F, E=32, k=4, L=2, capacity=8, max_tokens=4, window=8, zipf_s=1.1, shared=True,
              weight_format=fmt)
    try:
        for step in range(16):
            used = {}
            for layer in range(m.L):
                x, lg = m.wl.x(layer, step, 1), m.wl.logits(layer, step, 1)
                idx = torch.empty((1, m.k), dtype=torch.int32, device="cuda")
                w = torch.empty((1, m.k), device="cuda")
                y = torch.empty((1, m.H), device="cuda")
                qec.moe_ffn_forward_routed(m.ctx, layer, m.dev(x), m.dev(lg), 1, idx, w, y)
                torch.cuda.synchronize()
                idx_np = idx.cpu().numpy()
                if step % 4 == 0 or step == 15:
                    check_layer_parity(m, layer, x, lg, y.cpu().numpy(), idx_np, w.cpu().numpy())
                else:
                    io, _ = oracle.topk(lg, m.k)
                    assert np.array_equal(idx_np, io)
                for kd in range(3):
                    used[layer * 3 + kd] = idx_np.ravel().tolist()
            qec.cache_step(m.ctx, 1)
            m.policy.step(1, used)
            for tid in range(3 * m.L):
                snap = qec.moe_cache_snapshot(m.ctx, tid, m.E, m.spt)
                o = m.policy.snapshot(tid)
                assert snap["slot_of"].tolist() == o["slot_of"] and snap["last_seen"].tolist() == o["last_seen"]
                assert np.array_equal(snap["tbl"], m.expected_tbl(tid))
        st = qec.moe_stats(m.ctx)
        assert st["admissions"] == m.policy.stats["admissions"] > 0
        assert st["hits"] == m.policy.stats["hits"] and st["misses"] == m.policy.stats["misses"] > 0
    finally:
        m.close()
