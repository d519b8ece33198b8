"""GPU parity of the prefill path (grouped tcgen05 GEMM over tokens sorted by
expert) against the oracle, through the C ABI: several token tiles per
expert, ragged weight-row tiles, hot and cold experts, misses and stamps."""
import numpy as np
import pytest

import quantized_expert_cache_gb300 as qec
from gpu_helpers import Model, check_layer_parity

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    qec.build.build()
    qec.load()


@pytest.mark.parametrize("H,F,E,k,T,cap", [
    (256, 512, 8, 2, 600, 8),        # ~150 tokens per expert: several token tiles, all hot
    (512, 384, 64, 4, 120, 32),      # half of the experts cold (zero-copy reads)
    (2048, 1152, 64, 8, 256, 48),    # decode-model shape, 2048 assignments
    (768, 1216, 16, 2, 97, 12),      # ragged row tiles (1216 = 9.5 x 128), odd token count
])
def test_prefill_layer_parity(H, F, E, k, T, cap):
    m = Model(H=H, F=F, E=E, k=k, L=1, capacity=cap, max_tokens=T, zipf_s=0.8)
    try:
        x, lg = m.wl.x(0, 3, T), m.wl.logits(0, 3, T)
        idx, w = m.route(lg)
        y = m.forward(0, x, idx, w)
        torch.cuda.synchronize()
        idx_np = idx.cpu().numpy()
        n_alt = check_layer_parity(m, 0, x, lg, y.cpu().numpy(), idx_np, w.cpu().numpy())
        used = sorted(set(idx_np.ravel().tolist()))
        expect = []
        for kind in range(3):
            slot_of = m.policy.snapshot(kind)["slot_of"]
            expect += [(kind << 12) | e for e in used if slot_of[e] < 0]
        assert qec.miss_drain(m.ctx).tolist() == sorted(expect)
        for kind in range(3):
            snap = qec.moe_cache_snapshot(m.ctx, kind, m.E, m.spt)
            for e in used:
                s = snap["slot_of"][e]
                if s >= 0:
                    assert snap["stamps"][s] == T
        assert n_alt <= max(4, T * k * F // 20000)
    finally:
        m.close()


def test_prefill_repeat_is_deterministic():
    m = Model(H=512, F=384, E=16, k=4, L=1, capacity=16, max_tokens=300, zipf_s=1.0)
    try:
        x, lg = m.wl.x(0, 0, 300), m.wl.logits(0, 0, 300)
        idx, w = m.route(lg)
        y1 = m.forward(0, x, idx, w).clone()
        y2 = m.forward(0, x, idx, w)
        torch.cuda.synchronize()
        assert torch.equal(y1, y2)
    finally:
        m.close()


@pytest.mark.parametrize("n_borrow", [2, 7, 30])
def test_prefill_with_lent_slots_stages_cold_experts(n_borrow):
    """With pool slots lent to the prompt pass, the layer's cold expert
    tensors are staged into them (as many as fit) and read from HBM; the
    result is unchanged and the miss log still lists every cold read."""
    m = Model(H=512, F=384, E=16, k=2, L=2, capacity=8, max_tokens=600, zipf_s=0.5, slots_per_tensor=8)
    try:
        qec.moe_pool_borrow(m.ctx, n_borrow)
        m.policy.borrow(n_borrow)
        for layer in range(2):
            T = 600
            x, lg = m.wl.x(layer, 5, T), m.wl.logits(layer, 5, T)
            idx, w = m.route(lg)
            y = m.forward(layer, x, idx, w)
            torch.cuda.synchronize()
            idx_np = idx.cpu().numpy()
            check_layer_parity(m, layer, x, lg, y.cpu().numpy(), idx_np, w.cpu().numpy())
            used = sorted(set(idx_np.ravel().tolist()))
            expect = sorted(((layer * 3 + kd) << 12) | e for kd in range(3) for e in used
                            if m.policy.snapshot(layer * 3 + kd)["slot_of"][e] < 0)
            assert qec.miss_drain(m.ctx).tolist() == expect
        qec.moe_pool_return(m.ctx)
        m.policy.give_back()
        for tid in range(6):
            snap = qec.moe_cache_snapshot(m.ctx, tid, m.E, m.spt)
            assert snap["slot_of"].tolist() == m.policy.snapshot(tid)["slot_of"]
            assert np.array_equal(snap["tbl"], m.expected_tbl(tid))
    finally:
        m.close()


def test_prefill_lookahead_prefetch_matches_plain_run():
    """Lookahead prefetch: a prompt forward of layer l uploads layer l + 1's
    cold expert tensors, and that layer reads them from the prefetch buffer.
    Outputs, stats and cache state equal those of the same run without
    prefetch, also across promotion passes that change the cold sets while a
    prefetch is pending (admissions on the second sighting); the prefetching
    run's outputs match the oracle on every pass.  (The layers' token counts
    differ from the promotion pass's n_tokens here, so stamps follow each
    forward's own count; the two runs' states are compared with each other.)"""
    # a wide window: prompt-length steps then admit on the second sighting;
    # the layers' token counts differ, so some stamps are older than the clock
    kw = dict(H=512, F=384, E=16, k=2, L=3, capacity=8, max_tokens=400, zipf_s=0.5, window=10000)
    a, b = Model(**kw), Model(**kw)
    try:
        qec.moe_set_lookahead(b.ctx, True)
        for p in range(3):
            for layer in range(3):
                T = 400 - 37 * layer
                x, lg = a.wl.x(layer, p, T), a.wl.logits(layer, p, T)
                ia, wa = a.route(lg)
                ib, wb = b.route(lg)
                ya = a.forward(layer, x, ia, wa)
                yb = b.forward(layer, x, ib, wb)
                torch.cuda.synchronize()
                assert torch.equal(ya, yb), (p, layer)
                check_layer_parity(b, layer, x, lg, yb.cpu().numpy(), ib.cpu().numpy(), wb.cpu().numpy())
            qec.cache_step(a.ctx, 400)
            qec.cache_step(b.ctx, 400)
        sa, sb = qec.moe_stats(a.ctx), qec.moe_stats(b.ctx)
        for key in ("hits", "misses", "admissions", "evictions", "cold_bytes"):
            assert sa[key] == sb[key], key
        assert sa["admissions"] > 0
        for tid in range(9):
            xa = qec.moe_cache_snapshot(a.ctx, tid, a.E, a.spt)
            xb = qec.moe_cache_snapshot(b.ctx, tid, b.E, b.spt)
            for key in ("slot_of", "last_seen", "owner", "stamps"):
                assert np.array_equal(xa[key], xb[key]), (tid, key)
    finally:
        a.close()
        b.close()
