"""The allocation-free layer entry point (moe_expert_ffn_noalloc).

Some callers cannot allocate device memory at the moment they run a layer
(their device memory belongs to another allocator, or allocation is
forbidden where they run); for them the library keeps every intermediate of
this entry point in one fixed device array.  Checked here, two calls in a
row on three shapes: its y against the oracle (through the h codes the
context entry point produces on the same inputs, validated against the
oracle's binary64 h) and against the context entry point (moe_ffn_forward);
and that a fault its kernel detects (an out-of-range expert id) is reported
by moe_expert_ffn_noalloc_status.  This file is collected last on purpose."""
import numpy as np
import pytest

import oracle
import quantized_expert_cache_gb300 as qec
from gpu_helpers import Model, assert_close, check_h_codes

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    qec.build.build()
    qec.load()


def _oracle_y(m, x, lg, idx, w):
    """The oracle's y for this forward: its own y when every h code of the
    context forward matches, else its down projection and combine applied to
    the context's (validated) codes."""
    T = x.shape[0]
    idx_o, w_o = oracle.topk(lg, m.k)
    assert np.array_equal(idx.cpu().numpy(), idx_o)
    used = sorted(set(idx_o.ravel().tolist()))
    g = {e: m.tensor(0, 0)[e] for e in used}
    u = {e: m.tensor(0, 1)[e] for e in used}
    d = {e: m.tensor(0, 2)[e] for e in used}
    y_o, it = oracle.layer(x, idx_o, w_o, g, u, d, m.H, m.F, want_intermediates=True)
    xq, xd, hq, hd = m.read_debug(T)
    assert np.array_equal(xq, it["xq"]) and np.array_equal(xd, it["xd"])
    n_alt = check_h_codes(hq, hd, it, m.H // 32)
    return oracle.down_combine(idx_o, w_o, d, hq, hd, m.H, m.F) if n_alt else y_o


@pytest.mark.parametrize("H,F,E,k,T", [(512, 384, 64, 4, 3), (2048, 1152, 64, 8, 1), (640, 1440, 16, 3, 9)])
def test_noalloc_matches_oracle_and_context_forward_twice(H, F, E, k, T):
    m = Model(H=H, F=F, E=E, k=k, L=1, capacity=E // 2, max_tokens=T, zipf_s=0.7)
    try:
        x, lg = m.wl.x(0, 2, T), m.wl.logits(0, 2, T)
        idx, w = m.route(lg)
        y_ctx = m.forward(0, x, idx, w)
        torch.cuda.synchronize()
        y_ctx = y_ctx.cpu().numpy().astype(np.float64)
        y_ref = _oracle_y(m, x, lg, idx, w)
        assert_close(y_ctx, y_ref, "context y")
        tbl = np.stack([qec.moe_cache_snapshot(m.ctx, kind, E, m.spt)["tbl"] for kind in range(3)])
        d_tbl = torch.from_numpy(tbl.view(np.int64)).cuda()
        d_x = torch.from_numpy(x).cuda()
        for _ in range(2):
            y = torch.full((T, H), float("nan"), device="cuda")
            qec.moe_expert_ffn_noalloc(d_x, T, idx, w, d_tbl, H, F, E, k, y)
            qec.moe_expert_ffn_noalloc_status()
            y_np = y.cpu().numpy()
            assert_close(y_np, y_ref, "noalloc y vs oracle")
            assert_close(y_np, y_ctx, "noalloc y vs context forward")
    finally:
        m.close()


def test_noalloc_reports_a_bad_expert_id():
    H, F, E, k, T = 512, 384, 64, 4, 3
    m = Model(H=H, F=F, E=E, k=k, L=1, capacity=E, max_tokens=T)
    try:
        x, lg = m.wl.x(0, 0, T), m.wl.logits(0, 0, T)
        idx, w = m.route(lg)
        tbl = np.stack([qec.moe_cache_snapshot(m.ctx, kind, E, m.spt)["tbl"] for kind in range(3)])
        d_tbl = torch.from_numpy(tbl.view(np.int64)).cuda()
        d_x = torch.from_numpy(x).cuda()
        y = torch.empty((T, H), device="cuda")
        bad = idx.clone()
        bad[1, 2] = E + 5  # the kernel range-checks ids and reads this one as expert 0
        qec.moe_expert_ffn_noalloc(d_x, T, bad, w, d_tbl, H, F, E, k, y)
        with pytest.raises(qec.MoeError) as ei:
            qec.moe_expert_ffn_noalloc_status()
        assert ei.value.code == -8 and "outside" in qec.moe_last_error(None)
        # the next call clears the word
        qec.moe_expert_ffn_noalloc(d_x, T, idx, w, d_tbl, H, F, E, k, y)
        assert qec.moe_expert_ffn_noalloc_status() == 0
    finally:
        m.close()


def test_noalloc_rejects_oversized_calls():
    dummy = 1 << 20  # never dereferenced: the size check comes first
    with pytest.raises(qec.MoeError) as ei:
        qec.moe_expert_ffn_noalloc(dummy, 32, dummy, dummy, dummy, 8192, 1024, 64, 8, dummy)
    assert ei.value.code == -6 and "maximum" in qec.moe_last_error(None)
    with pytest.raises(qec.MoeError) as ei:
        qec.moe_expert_ffn_noalloc(dummy, 33, dummy, dummy, dummy, 512, 384, 64, 4, dummy)
    assert ei.value.code == -1
