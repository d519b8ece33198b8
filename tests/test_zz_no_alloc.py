"""The allocation-free layer entry point (moe_expert_ffn_noalloc) against the
context entry point (moe_ffn_forward) on the same inputs, two calls in a row.

Callers that cannot allocate device memory when they run a layer use the
allocation-free entry point; its intermediates live in a fixed device array
of the library.  This file is collected last on purpose."""
import numpy as np
import pytest

import quantized_expert_cache_gb300 as qec
from gpu_helpers import Model, assert_close

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    qec.build.build()
    qec.load()


@pytest.mark.parametrize("H,F,E,k,T", [(512, 384, 64, 4, 3), (2048, 1152, 64, 8, 1), (640, 1440, 16, 3, 9)])
def test_noalloc_matches_context_forward_twice(H, F, E, k, T):
    m = Model(H=H, F=F, E=E, k=k, L=1, capacity=E // 2, max_tokens=T, zipf_s=0.7)
    try:
        x, lg = m.wl.x(0, 2, T), m.wl.logits(0, 2, T)
        idx, w = m.route(lg)
        y_ref = m.forward(0, x, idx, w)
        torch.cuda.synchronize()
        y_ref = y_ref.cpu().numpy().astype(np.float64)
        tbl = np.stack([qec.moe_cache_snapshot(m.ctx, kind, E, m.spt)["tbl"] for kind in range(3)])
        d_tbl = torch.from_numpy(tbl.view(np.int64)).cuda()
        d_x = torch.from_numpy(x).cuda()
        for _ in range(2):
            y = torch.full((T, H), float("nan"), device="cuda")
            qec.moe_expert_ffn_noalloc(d_x, T, idx, w, d_tbl, H, F, E, k, y)
            torch.cuda.synchronize()
            assert_close(y.cpu().numpy(), y_ref, "noalloc y")
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
