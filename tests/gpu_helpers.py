"""Helpers for the GPU parity tests: build a context from a small workload
spec, run the oracle on the same seeded inputs, and compare.

Tolerances (from the parity contract of the path):
- bit-exact: top-k indices, quantized x (codes and binary16 scales), int32
  block dots, miss-log contents (sorted unique), table / stamp / sighting
  state after every promotion pass;
- fp32 layer outputs: |y_gpu - y_ref| <= 1e-4 + 2e-3 * |y_ref| elementwise.

Quantized h: h is computed in fp32 in a different summation order (and with
CUDA's expf) than the oracle's binary64 value, so a code whose value sits
within rounding error of a half-step may legitimately round either way.
Such a code is accepted only if it is the rounding of some h' within the
derived error bound of the oracle's h (below); y is then compared against
the oracle's down projection and combine applied to the GPU's quantized h
(when every code matches, that is exactly the oracle's own y).
"""
from __future__ import annotations

import numpy as np

import oracle
import quantized_expert_cache_gb300 as qec
import synth

U32 = 2.0 ** -24  # unit roundoff of binary32
RTOL, ATOL = 2e-3, 1e-4


def f16(bits):
    return np.asarray(bits, np.uint16).view(np.float16).astype(np.float64)


def h_error_bound(g, u, gabs, uabs, nb):
    """Bound on |h_gpu - h| for h = silu(g) u, given binary64 g, u and the
    sums of |terms| of their block sums: fp32 accumulation of nb scaled block
    terms (one rounding per product and per addition), then a few fp32 ops
    and expf (<= 2 ulp) for h."""
    gam = (nb + 2) * U32 * 1.01
    Eg, Eu = gam * gabs, gam * uabs
    sg = 1.0 / (1.0 + np.exp(-np.clip(g, -700, 700)))
    dh_dg = np.abs(u * sg * (1.0 + g * (1.0 - sg))) + np.abs(u) * 1e-30
    silu = np.abs(g * sg)
    h = g * u * sg
    return dh_dg * (Eg + 1e-30) + silu * Eu + 8 * U32 * np.abs(h) + 1e-38


def check_h_codes(hq_gpu, hd_gpu, it, nbh):
    """Validate the GPU's quantized h against the oracle's binary64 h.
    Returns the number of codes that differ from the oracle's (all valid)."""
    A, F = it["h"].shape
    h = it["h"]
    E = h_error_bound(it["g"], it["u"], it["gabs"], it["uabs"], nbh)
    hb = h.reshape(A, F // 32, 32)
    Eb = E.reshape(A, F // 32, 32)
    amax = np.abs(hb.astype(np.float32).astype(np.float64)).max(axis=2)
    Ea = np.abs(Eb).max(axis=2)
    lo = f16(np.float16(np.float32(np.maximum(amax - Ea, 0)) / np.float32(127)).view(np.uint16))
    hi = f16(np.float16(np.float32(amax + Ea) / np.float32(127)).view(np.uint16))
    dd = f16(hd_gpu)
    bad_d = (dd < lo) | (dd > hi)
    assert not bad_d.any(), f"h scale outside its valid range at {np.argwhere(bad_d)[:5]}"
    ddb = dd[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        clo = np.where(ddb > 0, np.clip(np.rint((hb - Eb) / ddb), -127, 127), 0)
        chi = np.where(ddb > 0, np.clip(np.rint((hb + Eb) / ddb), -127, 127), 0)
    c = hq_gpu.reshape(A, F // 32, 32).astype(np.float64)
    bad = (c < clo) | (c > chi)
    assert not bad.any(), f"h code outside its valid range at {np.argwhere(bad)[:5]}"
    return int((hq_gpu != it["hq"]).sum()) + int((hd_gpu != it["hd"]).sum())


def assert_close(y_gpu, y_ref, what="y"):
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    tol = ATOL + RTOL * np.abs(y_ref)
    bad = err > tol
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; worst "
                           f"{(err / tol).max():.3g}x at {np.unravel_index((err / tol).argmax(), err.shape)}")


class Model:
    """A small stack of expert tensors registered in one context."""

    def __init__(self, H, F, E, k, L, capacity, max_tokens, seed=0, routing="zipf", zipf_s=1.1, window=64,
                 slots_per_tensor=None, max_swaps=0, stream=None, global_pool=False, preheat=False,
                 weight_format=0, shared=False, poll_timeout_ms=10000):
        import torch
        self.torch = torch
        self.wl = synth.Workload("test", H, E, k, F, L, routing=routing, zipf_s=zipf_s, seed=seed,
                                 capacity=[capacity] * L if isinstance(capacity, int) else list(capacity),
                                 weight_format=weight_format)
        self.H, self.F, self.E, self.k, self.L = H, F, E, k, L
        self.spt = slots_per_tensor if slots_per_tensor is not None else max(self.wl.capacity)
        # one stream for torch's copies / allocations and the library's kernels
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        self.ctx = qec.moe_layer_init(H, F, E, k, L, self.spt, max_tokens, window_tokens=window,
                                      max_swaps_per_step=max_swaps, stream=stream, weight_format=weight_format,
                                      shared_experts=int(shared), poll_timeout_ms=poll_timeout_ms)
        self.shared = None
        if shared:
            # one shared expert per layer, from its own seeded stream
            sw = synth.Workload("shared", H, 1, 1, F, L, seed=seed + 101, weight_format=weight_format)
            self.shared = {}
            for layer in range(L):
                for kind in range(3):
                    t = sw.expert_tensor(layer, kind)[0]
                    rows, cols = sw.tensor_shapes[kind]
                    qec.register_shared_expert(self.ctx, layer, kind, t, rows, cols)
                    self.shared[(layer, kind)] = t
        self.tensors = {}
        self.global_pool = global_pool
        if global_pool:
            qec.moe_set_global_pool(self.ctx, True)
        if preheat:
            qec.moe_set_preheat(self.ctx, True)
        self.window, self.max_swaps = window, max_swaps
        self._new_policy()
        for layer in range(L):
            order = self.wl.seed_order(layer)
            cap = self.wl.layer_capacity(layer)
            for kind in range(3):
                t = self.wl.expert_tensor(layer, kind)
                rows, cols = self.wl.tensor_shapes[kind]
                tid = qec.register_expert_tensor(self.ctx, layer, kind, t, rows, cols, cap, order, cap)
                assert tid == layer * 3 + kind
                self.tensors[tid] = t
                self.policy.add_tensor(tid, cap, order, cap)

    def _new_policy(self):
        self.policy = oracle.PolicyOracle(self.E, window=self.window, max_swaps_per_step=self.max_swaps,
                                          slots_per_tensor=self.spt, n_tensors=3 * self.L,
                                          global_pool=self.global_pool)

    def reset(self, global_pool):
        """Registered state again (library and oracle), in a pool mode."""
        qec.moe_cache_reset(self.ctx, global_pool)
        self.global_pool = global_pool
        self._new_policy()
        for layer in range(self.L):
            cap = self.wl.layer_capacity(layer)
            for kind in range(3):
                self.policy.add_tensor(layer * 3 + kind, cap, self.wl.seed_order(layer), cap)

    def close(self):
        qec.moe_destroy(self.ctx)
        self.ctx = None

    def tensor(self, layer, kind):
        return self.tensors[layer * 3 + kind]

    # -- device helpers --------------------------------------------------------
    def dev(self, a):
        return self.torch.from_numpy(np.ascontiguousarray(a)).cuda()

    def route(self, logits_np):
        torch = self.torch
        T = logits_np.shape[0]
        lg = self.dev(logits_np)
        idx = torch.empty((T, self.k), dtype=torch.int32, device="cuda")
        w = torch.empty((T, self.k), dtype=torch.float32, device="cuda")
        qec.route_topk(self.ctx, lg, T, self.E, self.k, idx, w)
        torch.cuda.synchronize()
        return idx, w

    def forward(self, layer, x_np, idx, w):
        torch = self.torch
        T = x_np.shape[0]
        x = self.dev(x_np)
        y = torch.empty((T, self.H), dtype=torch.float32, device="cuda")
        qec.moe_ffn_forward(self.ctx, layer, x, T, idx, w, y)
        return y

    @property
    def ka(self):
        """Assignments per token (the routed k, plus the shared expert)."""
        return self.k + (1 if getattr(self, "shared", None) else 0)

    def read_debug(self, T):
        H, F, k = self.H, self.F, self.ka
        xq = np.empty((T, H), np.int8)
        xd = np.empty((T, H // 32), np.uint16)
        hq = np.empty((T * k, F), np.int8)
        hd = np.empty((T * k, F // 32), np.uint16)
        for what, arr in ((0, xq), (1, xd), (2, hq), (3, hd)):
            qec.moe_debug_read(self.ctx, what, arr)
        return xq, xd, hq, hd

    def expected_tbl(self, tid):
        lay = qec.moe_cache_layout(self.ctx, tid)
        snap = self.policy.snapshot(tid)
        out = np.empty(self.E, np.uint64)
        for e in range(self.E):
            s = snap["slot_of"][e]
            if s >= 0:
                g = s if self.global_pool else s * lay["n_tensors"] + tid
                out[e] = lay["pool_base"] + g * lay["slot_bytes"]
            else:
                out[e] = (lay["host_base"] + e * lay["slot_bytes"]) | 1
        return out


def check_layer_parity(m: Model, layer, x_np, logits_np, y_gpu, idx_gpu, w_gpu):
    """Full-layer parity of one forward against the oracle."""
    T = x_np.shape[0]
    idx_o, w_o = oracle.topk(logits_np, m.k)
    assert np.array_equal(idx_gpu, idx_o), "top-k indices differ"
    np.testing.assert_allclose(w_gpu, w_o, rtol=1e-5, atol=1e-7)
    used = sorted(set(idx_o.ravel().tolist()))
    g = {e: m.tensor(layer, 0)[e] for e in used}
    u = {e: m.tensor(layer, 1)[e] for e in used}
    d = {e: m.tensor(layer, 2)[e] for e in used}
    if getattr(m, "shared", None):
        idx_o, w_o, g, u, d = oracle.with_shared(idx_o, w_o, g, u, d,
                                                 tuple(m.shared[(layer, kd)] for kd in range(3)), e_shared=m.E)
        # the shared expert is id E (one past the routed ids)
        assert (idx_o[:, -1] == m.E).all()
    y_o, it = oracle.layer(x_np, idx_o, w_o, g, u, d, m.H, m.F, want_intermediates=True)
    xq, xd, hq, hd = m.read_debug(T)
    assert np.array_equal(xq, it["xq"]), "quantized x codes differ"
    assert np.array_equal(xd, it["xd"]), "quantized x scales differ"
    # Q4_K's block term has two products and a difference before the scale
    # (two more roundings per block than the other formats)
    extra = 2 if m.wl.weight_format in (synth.FMT_Q4_K, synth.FMT_Q5_K) else 0
    n_alt = check_h_codes(hq, hd, it, m.H // 32 + extra)
    y_ref = oracle.down_combine(idx_o, w_o, d, hq, hd, m.H, m.F) if n_alt else y_o
    assert_close(y_gpu, y_ref)
    return n_alt


class _LazyExperts:
    """Expert tensor whose experts are regenerated on demand from their
    seeded streams (full-size workloads do not keep every weight in RAM)."""

    def __init__(self, wl, layer, kind):
        self.wl, self.layer, self.kind = wl, layer, kind
        self.cache = {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self.cache:
            self.cache[e] = self.wl.expert_tensor(self.layer, self.kind, e, e + 1)[0]
        return self.cache[e]


class FullModel(Model):
    """A whole workload of synth.WORKLOADS registered in one context, with
    the library's seeding (capacity and routing-frequency order per layer)."""

    def __init__(self, wl, max_tokens, slots_per_tensor=None, window=64, stream=None):
        import torch
        self.torch = torch
        self.wl = wl
        self.H, self.F, self.E, self.k, self.L = wl.hidden, wl.ffn, wl.n_experts, wl.top_k, wl.n_layers
        self.spt = slots_per_tensor or max(wl.layer_capacity(l) for l in range(wl.n_layers))
        self.global_pool = False
        if stream is None:
            stream = torch.cuda.current_stream().cuda_stream
        self.ctx = qec.moe_layer_init(self.H, self.F, self.E, self.k, self.L, self.spt, max_tokens,
                                      window_tokens=window, stream=stream)
        self.policy = oracle.PolicyOracle(self.E, window=window, slots_per_tensor=self.spt, n_tensors=3 * self.L)
        self.tensors = {}
        bufs = {}
        for layer in range(self.L):
            order = wl.seed_order(layer)
            cap = wl.layer_capacity(layer)
            for kind in range(3):
                rows, cols = wl.tensor_shapes[kind]
                if (rows, cols) not in bufs:
                    bufs[(rows, cols)] = np.empty((self.E, rows, cols // 32, 18), np.uint8)
                wl.expert_tensor(layer, kind, out=bufs[(rows, cols)])
                tid = qec.register_expert_tensor(self.ctx, layer, kind, bufs[(rows, cols)], rows, cols, cap, order,
                                                 cap)
                self.tensors[tid] = _LazyExperts(wl, layer, kind)
                self.policy.add_tensor(tid, cap, order, cap)
        del bufs


def check_sampled_rows(m, layer, x_np, logits_np, y_gpu, idx_gpu, w_gpu, rows):
    """Parity of selected tokens (rows) of one forward against the oracle:
    idx of every token bit-exact, and for the sampled tokens x codes, h codes
    (validated) and y."""
    T = x_np.shape[0]
    idx_o, w_o = oracle.topk(logits_np, m.k)
    assert np.array_equal(idx_gpu, idx_o), "top-k indices differ"
    np.testing.assert_allclose(w_gpu, w_o, rtol=1e-5, atol=1e-7)
    rows = np.asarray(sorted(set(int(r) for r in rows)))
    xs, io, wo = x_np[rows], idx_o[rows], w_o[rows]
    used = sorted(set(io.ravel().tolist()))
    g = {e: m.tensor(layer, 0)[e] for e in used}
    u = {e: m.tensor(layer, 1)[e] for e in used}
    d = {e: m.tensor(layer, 2)[e] for e in used}
    y_o, it = oracle.layer(xs, io, wo, g, u, d, m.H, m.F, want_intermediates=True)
    xq, xd, hq, hd = m.read_debug(T)
    assert np.array_equal(xq[rows], it["xq"]) and np.array_equal(xd[rows], it["xd"]), "x codes differ"
    arows = (rows[:, None] * m.k + np.arange(m.k)[None, :]).ravel()
    n_alt = check_h_codes(hq[arows], hd[arows], it, m.H // 32)
    y_ref = oracle.down_combine(io, wo, d, hq[arows], hd[arows], m.H, m.F) if n_alt else y_o
    assert_close(y_gpu[rows], y_ref)
    return n_alt
