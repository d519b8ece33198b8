"""GPU parity of the other expert weight formats through the C ABI, against
the oracle: Q8_0 (blocks of 32 signed 8-bit codes and one binary16 scale,
w = d * q), Q5_0 (5-bit codes, w = d * (q - 16)), Q4_K (256-weight
super-blocks, 6-bit sub-block scales and mins, w = d*sc*q - dmin*m) and Q6_K
(256-weight super-blocks, signed 8-bit scales of 16-weight sub-blocks, 6-bit
codes, w = d*sc*(q - 32)) and Q5_K (Q4_K with a fifth code bit, q in 0..31).
Integer block dots
bit-exact from pool slots and from pinned host memory, whole layers (decode
and prompt-sized batches, hot and cold experts, ragged shapes), the miss
log, and the cache state after every promotion pass."""
import numpy as np
import pytest

import oracle
import quantized_expert_cache_gb300 as qec
import synth
from gpu_helpers import Model, check_layer_parity

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
FMTS = [pytest.param(qec.FMT_Q8_0, id="q8_0"), pytest.param(qec.FMT_Q5_0, id="q5_0"),
        pytest.param(qec.FMT_Q4_K, id="q4_k"), pytest.param(qec.FMT_Q6_K, id="q6_k"),
        pytest.param(qec.FMT_Q5_K, id="q5_k")]
K_QUANTS = (qec.FMT_Q4_K, qec.FMT_Q6_K, qec.FMT_Q5_K)


def _fits(fmt, H, F):
    """The K-quants need hidden and FFN widths that are multiples of their 256-weight super-blocks."""
    return fmt not in K_QUANTS or (H % 256 == 0 and F % 256 == 0)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    qec.build.build()
    qec.load()


@pytest.mark.parametrize("fmt", FMTS)
def test_block_dots_bit_exact_hot_and_cold(fmt):
    m = Model(H=256, F=512, E=8, k=2, L=1, capacity=4, max_tokens=4, routing="normal", weight_format=fmt)
    try:
        rng = np.random.default_rng(5)
        for tid in (0, 1, 2):
            rows, cols = (512, 256) if tid < 2 else (256, 512)
            snap = qec.moe_cache_snapshot(m.ctx, tid, m.E, m.spt)
            hot = [e for e in range(8) if snap["slot_of"][e] >= 0]
            cold = [e for e in range(8) if snap["slot_of"][e] < 0]
            assert hot and cold
            for e in (hot[0], cold[-1]):
                qa = rng.integers(-127, 128, cols).astype(np.int8)
                qa[:32] = -127  # extreme activations against the block's codes
                n_rows = 37
                out = torch.empty((n_rows, cols // 32), dtype=torch.int32, device="cuda")
                qec.moe_debug_block_dots(m.ctx, tid, e, 5, n_rows, torch.from_numpy(qa).cuda(), out)
                W = m.tensors[tid][e]
                assert W.shape[-1] == synth.BLOCK_BYTES[fmt]
                if fmt == qec.FMT_Q4_K:
                    # raw sub-block dots: 8 per 256-weight super-block
                    ref = np.array([np.concatenate([oracle.subblock_dots(W[5 + r, u], qa[256 * u:256 * u + 256])
                                                    for u in range(cols // 256)]) for r in range(n_rows)])
                elif fmt == qec.FMT_Q5_K:
                    # raw sub-block dots (q in 0..31): 8 per super-block
                    ref = np.array([np.concatenate([oracle.q5k_subdots(W[5 + r, u], qa[256 * u:256 * u + 256])
                                                    for u in range(cols // 256)]) for r in range(n_rows)])
                elif fmt == qec.FMT_Q6_K:
                    # per 32 weights: the two 16-weight sub-blocks' scaled dots
                    ref = np.array([np.concatenate([oracle.q6k_blockdots(W[5 + r, u], qa[256 * u:256 * u + 256])
                                                    for u in range(cols // 256)]) for r in range(n_rows)])
                else:
                    ref = np.array([[oracle.block_dot(W[5 + r, b], qa[32 * b:32 * b + 32])
                                     for b in range(cols // 32)] for r in range(n_rows)])
                assert np.array_equal(out.cpu().numpy(), ref)
    finally:
        m.close()


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("H,F,E,k,T", [(256, 512, 8, 2, 4), (512, 384, 64, 4, 1), (512, 384, 64, 4, 7),
                                       (512, 384, 64, 4, 33), (640, 1440, 16, 3, 5), (640, 1440, 16, 3, 40),
                                       (2048, 1152, 64, 8, 1), (512, 768, 64, 4, 1), (512, 768, 64, 4, 9),
                                       (768, 1024, 16, 3, 40), (2048, 1536, 64, 8, 1)])
def test_layer_parity_hot_and_cold(H, F, E, k, T, fmt):
    if not _fits(fmt, H, F):
        pytest.skip("the K-quants need widths that are multiples of 256")
    m = Model(H=H, F=F, E=E, k=k, L=2, capacity=E // 2, max_tokens=T, zipf_s=0.6, weight_format=fmt)
    try:
        for layer in range(2):
            x, lg = m.wl.x(layer, 1, T), m.wl.logits(layer, 1, T)
            idx, w = m.route(lg)
            y = m.forward(layer, x, idx, w)
            torch.cuda.synchronize()
            idx_np = idx.cpu().numpy()
            check_layer_parity(m, layer, x, lg, y.cpu().numpy(), idx_np, w.cpu().numpy())
            used = sorted(set(idx_np.ravel().tolist()))
            expect = [((layer * 3 + kd) << 12) | e for kd in range(3) for e in used
                      if m.policy.snapshot(layer * 3 + kd)["slot_of"][e] < 0]
            assert qec.miss_drain(m.ctx).tolist() == sorted(expect)
    finally:
        m.close()


@pytest.mark.parametrize("fmt", FMTS)
def test_routed_forward_and_cache_steps(fmt):
    F = 512 if fmt in K_QUANTS else 384
    m = Model(H=512, F=F, E=32, k=4, L=2, capacity=8, max_tokens=4, window=8, zipf_s=1.1, weight_format=fmt)
    try:
        for step in range(30):
            T = 1 if step % 6 else 3
            used = {}
            for layer in range(m.L):
                x, lg = m.wl.x(layer, step, T), m.wl.logits(layer, step, T)
                idx = torch.empty((T, m.k), dtype=torch.int32, device="cuda")
                w = torch.empty((T, m.k), device="cuda")
                y = torch.empty((T, m.H), device="cuda")
                qec.moe_ffn_forward_routed(m.ctx, layer, m.dev(x), m.dev(lg), T, idx, w, y)
                torch.cuda.synchronize()
                idx_np = idx.cpu().numpy()
                if step % 10 == 0:
                    check_layer_parity(m, layer, x, lg, y.cpu().numpy(), idx_np, w.cpu().numpy())
                for kd in range(3):
                    used[layer * 3 + kd] = idx_np.ravel().tolist()
            qec.cache_step(m.ctx, T)
            m.policy.step(T, used)
            for tid in range(3 * m.L):
                snap = qec.moe_cache_snapshot(m.ctx, tid, m.E, m.spt)
                o = m.policy.snapshot(tid)
                assert snap["slot_of"].tolist() == o["slot_of"]
                assert snap["last_seen"].tolist() == o["last_seen"]
                assert snap["stamps"].tolist()[: len(o["stamp"])] == o["stamp"]
                assert np.array_equal(snap["tbl"], m.expected_tbl(tid))
        st = qec.moe_stats(m.ctx)
        assert st["admissions"] == m.policy.stats["admissions"] > 0
        assert st["hits"] == m.policy.stats["hits"] and st["misses"] == m.policy.stats["misses"]
        # admitted experts were uploaded whole: a layer after the promotions
        x, lg = m.wl.x(0, 99, 2), m.wl.logits(0, 99, 2)
        idx, w = m.route(lg)
        y = m.forward(0, x, idx, w)
        torch.cuda.synchronize()
        check_layer_parity(m, 0, x, lg, y.cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy())
    finally:
        m.close()


def test_format_is_checked():
    with pytest.raises(qec.MoeError) as ex:
        qec.moe_layer_init(256, 256, 8, 2, 1, 4, 4, weight_format=7,
                           stream=torch.cuda.current_stream().cuda_stream)
    assert ex.value.code == -1
    # a Q8_0 context has no prompt tensor-core path, so no lookahead either
    m = Model(H=256, F=256, E=8, k=2, L=1, capacity=4, max_tokens=64, weight_format=qec.FMT_Q8_0)
    try:
        with pytest.raises(qec.MoeError) as ex:
            qec.moe_set_lookahead(m.ctx, True)
        assert ex.value.code == -7
    finally:
        m.close()
