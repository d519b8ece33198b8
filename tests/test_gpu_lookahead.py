"""Decode lookahead (mihailescu2m/llama.cpp, MoE expert streaming, lookahead
prefetch: layer L+1's router predicts its experts from layer L's input, so
their reads start a layer early).

The synthetic model with a residual stream and linear routers (synth's
router model): with the routers registered and lookahead on, every batch-1
routed forward of layer l predicts layer l + 1's picks and prefetches their
pool-resident weights into L2.  Outputs, top-k, statistics and cache state
must equal those of the same run without it; outputs also match the oracle;
the prediction counters must show predictions and hits."""
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


def _routed(m, layer, x, lg):
    xd, ld = m.dev(x), m.dev(lg)
    idx = torch.empty((1, m.k), dtype=torch.int32, device="cuda")
    w = torch.empty((1, m.k), device="cuda")
    y = torch.empty((1, m.H), device="cuda")
    qec.moe_ffn_forward_routed(m.ctx, layer, xd, ld, 1, idx, w, y)
    torch.cuda.synchronize()
    return idx, w, y


@pytest.mark.parametrize("H,F,E,k,L,cap", [(512, 384, 64, 4, 4, 40), (2048, 1152, 512, 8, 3, 300)])
def test_decode_lookahead_matches_plain_run(H, F, E, k, L, cap):
    kw = dict(H=H, F=F, E=E, k=k, L=L, capacity=cap, max_tokens=1, zipf_s=1.1, window=16)
    a, b = Model(**kw), Model(**kw)
    try:
        for m in (a, b):
            m.wl.residual_rho = 0.9
        for l in range(L):
            qec.moe_set_router(b.ctx, l, b.wl.router_scale * b.wl.router(l), b.wl.router_bias(l))
        qec.moe_set_lookahead(b.ctx, True)
        check = {(0, 1), (3, L - 1), (5, 2 % L)}
        for s in range(6):
            used = {}
            for l in range(L):
                x, lg = a.wl.x(l, s, 1), a.wl.logits(l, s, 1)
                ia, wa, ya = _routed(a, l, x, lg)
                ib, wb, yb = _routed(b, l, x, lg)
                assert torch.equal(ia, ib) and torch.equal(wa, wb) and torch.equal(ya, yb), (s, l)
                if (s, l) in check:
                    check_layer_parity(b, l, x, lg, yb.cpu().numpy(), ib.cpu().numpy(), wb.cpu().numpy())
                for kind in range(3):
                    used[3 * l + kind] = ib.cpu().numpy().ravel().tolist()
            qec.cache_step(a.ctx, 1)
            qec.cache_step(b.ctx, 1)
            a.policy.step(1, used)
            b.policy.step(1, used)
        sa, sb = qec.moe_stats(a.ctx), qec.moe_stats(b.ctx)
        for key in ("hits", "misses", "admissions", "evictions", "cold_bytes"):
            assert sa[key] == sb[key] == b.policy.stats.get(key, sb[key]), key
        assert sa["lookahead_predicted"] == 0
        # layers 1..L-1 are predicted in every step
        assert sb["lookahead_predicted"] == 6 * (L - 1) * k
        assert 0 < sb["lookahead_hits"] <= sb["lookahead_predicted"]
        for tid in range(3 * L):
            xa = qec.moe_cache_snapshot(a.ctx, tid, a.E, a.spt)
            xb = qec.moe_cache_snapshot(b.ctx, tid, b.E, b.spt)
            for key in ("slot_of", "last_seen", "owner", "stamps"):
                assert np.array_equal(xa[key], xb[key]), (tid, key)
            o = b.policy.snapshot(tid)
            assert xb["slot_of"].tolist() == o["slot_of"], tid
            assert np.array_equal(xa["tbl"], a.expected_tbl(tid)) and np.array_equal(xb["tbl"], b.expected_tbl(tid))
    finally:
        a.close()
        b.close()
