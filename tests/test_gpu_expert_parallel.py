"""Expert parallelism through the C ABI, on one GPU: the two ranks of a
world-size-2 partition run one after the other as two shard contexts
(moe_set_expert_shard), each registered with its own half of every layer's
experts and with its own pool; the exchange between them (the sum
all-reduce of replicated tokens, the dispatch / combine of distributed
ones) is done on the host here -- the collectives themselves are covered by
the gloo tests of the same module.

Checked against the oracle, at every step:
- the top-k ids (global, bit-exact) and weights each rank routes;
- every rank's partial y: the oracle's layer with the other rank's picks
  weighted 0, x codes bit-exact and h codes validated as in every layer test;
- the sum of the partials against the whole layer;
- each rank's table / slot / stamp / sighting state after every promotion
  pass, and its hit / miss / admission counts, against the policy oracle
  over its own experts (local ids), fed with the picks of its experts;
  distributed tokens stamp with the clock of the whole step.
"""
import numpy as np
import pytest

import oracle
import quantized_expert_cache_gb300 as qec
import synth
from gpu_helpers import ATOL, RTOL, check_h_codes
from quantized_expert_cache_gb300 import expert_parallel as ep

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    qec.build.build()
    qec.load()


class Shard:
    """Rank `rank`'s context: experts [base, base + n) of every layer."""

    def __init__(self, wl, tensors, rank, world, cap, max_tokens):
        self.wl = wl
        E, L = wl.n_experts, wl.n_layers
        self.base, self.n = ep.shard_range(E, rank, world)
        self.spt = cap
        self.ctx = qec.moe_layer_init(wl.hidden, wl.ffn, self.n, wl.top_k, L, cap, max_tokens,
                                      weight_format=wl.weight_format)
        qec.moe_set_expert_shard(self.ctx, self.base, E)
        self.policy = oracle.PolicyOracle(self.n, window=64, slots_per_tensor=cap, n_tensors=3 * L)
        for layer in range(L):
            order = [int(e) - self.base for e in wl.seed_order(layer) if self.owns(e)]
            for kind in range(3):
                rows, cols = wl.tensor_shapes[kind]
                mine = np.ascontiguousarray(tensors[(layer, kind)][self.base:self.base + self.n])
                tid = qec.register_expert_tensor(self.ctx, layer, kind, mine, rows, cols, cap, order, cap)
                assert tid == 3 * layer + kind
                self.policy.add_tensor(tid, cap, order, cap)

    def owns(self, e):
        return self.base <= int(e) < self.base + self.n

    def used(self, layer, idx):
        ids = [int(e) - self.base for e in np.asarray(idx).ravel() if self.owns(e)]
        return {3 * layer + kind: ids for kind in range(3)}

    def check_state(self, where):
        L = self.wl.n_layers
        for tid in range(3 * L):
            snap = qec.moe_cache_snapshot(self.ctx, tid, self.n, self.spt)
            o = self.policy.snapshot(tid)
            assert snap["slot_of"].tolist() == o["slot_of"], (where, tid)
            assert snap["last_seen"].tolist() == o["last_seen"], (where, tid)
            assert snap["stamps"].tolist() == o["stamp"], (where, tid)
            lay = qec.moe_cache_layout(self.ctx, tid)
            want = np.array([lay["pool_base"] + (s * lay["n_tensors"] + tid) * lay["slot_bytes"] if s >= 0 else
                             (lay["host_base"] + e * lay["slot_bytes"]) | 1
                             for e, s in enumerate(o["slot_of"])], np.uint64)
            assert np.array_equal(snap["tbl"], want), (where, tid)
        st = qec.moe_stats(self.ctx)
        for key in ("hits", "misses", "admissions", "evictions"):
            assert st[key] == self.policy.stats[key], (where, key)

    def close(self):
        qec.moe_destroy(self.ctx)


def _debug(ctx, T, k, H, F):
    xq, xd = np.empty((T, H), np.int8), np.empty((T, H // 32), np.uint16)
    hq, hd = np.empty((T * k, F), np.int8), np.empty((T * k, F // 32), np.uint16)
    for what, arr in ((0, xq), (1, xd), (2, hq), (3, hd)):
        qec.moe_debug_read(ctx, what, arr)
    return xq, xd, hq, hd


def _check_partial(sh, tensors, layer, x, idx, w, y_gpu):
    """One rank's partial layer against the oracle's (other picks weigh 0).
    Returns the reference it matched (binary64: the oracle's partial, or its
    down projection and combine of the GPU's h codes where a code took the
    other valid rounding) and the number of such codes."""
    wl = sh.wl
    H, F, k = wl.hidden, wl.ffn, wl.top_k
    T = x.shape[0]
    idx = np.asarray(idx, np.int32)
    mine = (idx >= sh.base) & (idx < sh.base + sh.n)
    wm = np.where(mine, np.asarray(w, np.float64), 0.0)
    used = sorted(set(idx.ravel().tolist()))
    g, u, d = ({e: tensors[(layer, kd)][e] for e in used} for kd in range(3))
    y_o, it = oracle.layer(x, idx, wm, g, u, d, H, F, want_intermediates=True)
    xq, xd, hq, hd = _debug(sh.ctx, T, k, H, F)
    # the x copy covers the tokens this shard computes (one of its picks or more)
    rows = mine.any(axis=1)
    assert np.array_equal(xq[rows], it["xq"][rows]) and np.array_equal(xd[rows], it["xd"][rows]), "x codes differ"
    # h of the other rank's assignments is not computed here: take the oracle's
    other = ~mine.ravel()
    hq[other], hd[other] = it["hq"][other], it["hd"][other]
    extra = 2 if wl.weight_format in (synth.FMT_Q4_K, synth.FMT_Q5_K) else 0
    n_alt = check_h_codes(hq, hd, it, H // 32 + extra)
    y_ref = oracle.down_combine(idx, wm, d, hq, hd, H, F) if n_alt else y_o
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    tol = ATOL + RTOL * np.abs(y_ref)
    assert (err <= tol).all(), f"partial y: worst {(err / tol).max():.3g}x"
    return y_ref, n_alt


def _check_sum(y_sum, ref_sum, ref_abs, n_alt, y_full):
    """The GPU's sum of the partials is within both partials' tolerances of
    the sum of their references; with no h code on its other valid rounding,
    those references add up to the oracle's whole layer."""
    assert (np.abs(y_sum - ref_sum) <= 2 * ATOL + RTOL * ref_abs + 1e-7).all()
    if n_alt == 0:
        np.testing.assert_allclose(ref_sum, y_full, rtol=1e-9, atol=1e-12)


def _dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    return (t.to(dtype) if dtype is not None else t).cuda()


@pytest.mark.parametrize("fmt,H,F,E,k,cap,Ts,Td", [
    (synth.FMT_Q4, 256, 512, 16, 3, 3, (1, 4, 40), (37, 60)),   # fused layer, GEMM rows
    (synth.FMT_Q4, 512, 384, 13, 2, 2, (1, 9), (5, 29)),         # ragged shards (6 + 7 experts)
    (synth.FMT_Q8_0, 256, 320, 10, 2, 2, (1, 3), (6, 11)),       # mat-vec kernels
])
def test_two_shards_sum_to_the_layer_and_keep_their_own_caches(fmt, H, F, E, k, cap, Ts, Td):
    L, steps = 2, 6
    wl = synth.Workload("ep", H, E, k, F, L, routing="zipf", zipf_s=0.9, seed=21, weight_format=fmt)
    tensors = {(l, kd): wl.expert_tensor(l, kd) for l in range(L) for kd in range(3)}
    max_tokens = max(max(Ts), sum(Td))
    shards = [Shard(wl, tensors, r, 2, cap, max_tokens) for r in range(2)]
    try:
        for s in range(steps):
            used = [{} for _ in shards]
            if s % 2 == 0:
                # replicated tokens: both ranks route the same tokens
                T = Ts[(s // 2) % len(Ts)]
                for layer in range(L):
                    x, lg = wl.x(layer, s, T), wl.logits(layer, s, T)
                    io, wo = oracle.topk(lg, k)
                    y_sum, p_ref, p_abs = np.zeros((T, H)), np.zeros((T, H)), np.zeros((T, H))
                    n_alt = 0
                    for sh in shards:
                        idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
                        w = torch.empty((T, k), device="cuda")
                        y = torch.empty((T, H), device="cuda")
                        qec.moe_ffn_forward_routed(sh.ctx, layer, _dev(x), _dev(lg), T, idx, w, y)
                        torch.cuda.synchronize()
                        assert np.array_equal(idx.cpu().numpy(), io), (s, layer)
                        np.testing.assert_allclose(w.cpu().numpy(), wo, rtol=1e-5, atol=1e-7)
                        yp = y.cpu().numpy()
                        ref, alt = _check_partial(sh, tensors, layer, x, io, wo, yp)
                        y_sum += yp
                        p_ref += ref
                        p_abs += np.abs(ref)
                        n_alt += alt
                    _check_sum(y_sum, p_ref, p_abs, n_alt,
                               oracle.layer(x, io, wo, *(tensors[(layer, kd)] for kd in range(3)), H, F))
                    for r, sh in enumerate(shards):
                        used[r].update(sh.used(layer, io))
                n_step = T
            else:
                # distributed tokens: rank r holds Td[r] tokens; each rank gets
                # the rows with one of its experts among the picks
                n_step = sum(Td)
                for layer in range(L):
                    toks = []
                    for r, sh in enumerate(shards):
                        x, lg = wl.x(layer, 100 * s + r, Td[r]), wl.logits(layer, 100 * s + r, Td[r])
                        idx = torch.empty((Td[r], k), dtype=torch.int32, device="cuda")
                        w = torch.empty((Td[r], k), device="cuda")
                        qec.route_topk(sh.ctx, _dev(lg), Td[r], E, k, idx, w)
                        torch.cuda.synchronize()
                        io, wo = oracle.topk(lg, k)
                        assert np.array_equal(idx.cpu().numpy(), io)
                        toks.append((x, io, w.cpu().numpy()))
                    X = np.concatenate([t[0] for t in toks])
                    I = np.concatenate([t[1] for t in toks])
                    W = np.concatenate([t[2] for t in toks])
                    y_home, ref_home, abs_home = (np.zeros((n_step, H)) for _ in range(3))
                    n_alt = 0
                    for r, sh in enumerate(shards):
                        rows = np.nonzero(((I >= sh.base) & (I < sh.base + sh.n)).any(axis=1))[0]
                        n = len(rows)
                        y = torch.empty((max(n, 1), H), device="cuda")
                        qec.moe_ffn_forward_rows(sh.ctx, layer, _dev(X[rows]), n, _dev(I[rows]), _dev(W[rows]), y,
                                                 n_step)
                        torch.cuda.synchronize()
                        if n:
                            yp = y.cpu().numpy()[:n]
                            ref, alt = _check_partial(sh, tensors, layer, X[rows], I[rows], W[rows], yp)
                            y_home[rows] += yp
                            ref_home[rows] += ref
                            abs_home[rows] += np.abs(ref)
                            n_alt += alt
                        used[r].update(sh.used(layer, I))
                    _check_sum(y_home, ref_home, abs_home, n_alt,
                               oracle.layer(X, I, W, *(tensors[(layer, kd)] for kd in range(3)), H, F))
            for r, sh in enumerate(shards):
                qec.cache_step(sh.ctx, n_step)
                sh.policy.step(n_step, used[r])
                sh.check_state((s, sh.base))
        for sh in shards:
            assert sh.policy.stats["misses"] > 0 and sh.policy.stats["hits"] > 0
    finally:
        for sh in shards:
            sh.close()


def test_shard_argument_checks():
    ctx = qec.moe_layer_init(256, 256, 8, 2, 1, 2, 4)
    try:
        for base, n_route in ((-1, 16), (9, 16), (0, 7), (0, 5000)):
            with pytest.raises(qec.MoeError):
                qec.moe_set_expert_shard(ctx, base, n_route)
        qec.moe_set_expert_shard(ctx, 8, 16)
        qec.moe_set_expert_shard(ctx, 0, 8)  # back to unsharded
        x = torch.zeros((2, 256), device="cuda")
        with pytest.raises(qec.MoeError):  # step_tokens below the rows
            qec.moe_ffn_forward_rows(ctx, 0, x, 2, x, x, x, 1)
    finally:
        qec.moe_destroy(ctx)
