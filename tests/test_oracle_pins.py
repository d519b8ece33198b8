"""Pins of the numeric oracle against things other than itself: the IEEE
binary16 definition and numpy's independent float16, hand-worked block dots,
brute force over all codes, numpy stable sorts, scipy closed forms and fp64
dense matmuls of independently dequantized weights.

Each pin is chosen so that a plausible mistake in the oracle (a dropped
term, a wrong sign or offset, swapped nibbles, swapped gate/up, a wrong
index) fails at least one of them.
"""
import math

import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle
import synth

RNG = np.random.default_rng(1234)


# ---------------------------------------------------------------- binary16
def test_h2d_golden(golden):
    for bits, val, _ in golden("f16_values.txt"):
        got = oracle.h2d(int(bits, 16))
        assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val)), bits


def test_h2d_all_bit_patterns_vs_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.h2d(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_f2h_vs_numpy_random_and_ties():
    # random magnitudes over the whole binary16 range, incl. subnormals/overflow
    mags = np.exp2(RNG.uniform(-30, 17, 20000)).astype(np.float32)
    vals = np.concatenate([mags, -mags]).astype(np.float32)
    # exact midpoints between neighbouring binary16 values (ties to even)
    h = np.arange(0, 0x7bff, 7, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)
    assert np.array_equal(mid.astype(np.float64), (lo + hi) / 2)  # exact in binary32
    vals = np.concatenate([vals, mid, -mid, np.float32([0.0, -0.0, 65504, 65519.99, 65520, 1e-8, 2.0 ** -25])])
    with np.errstate(over="ignore"):  # values past 65520 round to infinity, as they should
        ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f2h(float(v)) for v in vals], np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(float(vals[i]), hex(got[i]), hex(ref[i])) for i in bad[:5]]


# ---------------------------------------------------------------- top-k
def _stable_topk(logits, k):
    # numpy's stable sort on -logit keeps index order among equal keys
    order = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")
    return order[:, :k]


@pytest.mark.parametrize("E,k", [(8, 2), (512, 8), (128, 4), (64, 1), (16, 16)])
def test_topk_matches_stable_sort(E, k):
    T = 37
    logits = RNG.standard_normal((T, E)).astype(np.float32)
    # force ties: quantize a third of the rows coarsely
    logits[::3] = np.round(logits[::3] * 2) / 2
    idx, w = oracle.topk(logits, k)
    assert np.array_equal(idx, _stable_topk(logits, k))


def test_topk_signed_zero_tie_goes_to_lower_index():
    logits = np.array([[-1.0, 0.0, -0.0, -2.0], [-1.0, -0.0, 0.0, -2.0]], np.float32)
    idx, _ = oracle.topk(logits, 2)
    assert idx.tolist() == [[1, 2], [1, 2]]


def test_topk_brute_force_subsets():
    # the chosen set maximizes the sum of logits among all k-subsets (E=8)
    import itertools
    logits = RNG.standard_normal((20, 8)).astype(np.float32)
    idx, _ = oracle.topk(logits, 3)
    for t in range(20):
        best = max(itertools.combinations(range(8), 3), key=lambda s: sum(float(logits[t, i]) for i in s))
        assert sorted(best) == sorted(idx[t].tolist())


def test_topk_weights_closed_forms():
    logits = RNG.standard_normal((50, 64)).astype(np.float32)
    idx, w = oracle.topk(logits, 6, renorm=True)
    sel = np.take_along_axis(logits.astype(np.float64), idx, 1)
    np.testing.assert_allclose(w, softmax(sel, axis=1), rtol=1e-14, atol=0)
    idx2, w2 = oracle.topk(logits, 6, renorm=False)
    full = softmax(logits.astype(np.float64), axis=1)
    np.testing.assert_allclose(w2, np.take_along_axis(full, idx2, 1), rtol=1e-13)


# ---------------------------------------------------------------- quantizer
def _exact_nearest_codes(xb, dd):
    """Brute force: the code c in [-127,127] minimizing |x - c*d| (exact,
    ties to the even code), for every element of a block."""
    cands = np.arange(-127, 128, dtype=np.float64)
    err = np.abs(xb[:, None].astype(np.float64) - cands[None, :] * dd)
    best = err.min(axis=1, keepdims=True)
    ties = err == best
    out = []
    for row in ties:
        cs = cands[row]
        even = cs[np.mod(cs, 2) == 0]
        out.append(even[0] if len(cs) > 1 and len(even) else cs[0])
    return np.array(out)


def test_quantizer_brute_force_and_scale():
    x = (RNG.standard_normal((64, 32)) * np.exp2(RNG.uniform(-6, 6, (64, 1)))).astype(np.float32)
    x[5] = 0.0
    x[7, :] = np.float32(0.5)
    q, d = oracle.quantize(x)
    for b in range(x.shape[0]):
        amax = np.float32(np.abs(x[b]).max())
        d_ref = np.float16(np.float32(amax) / np.float32(127.0)).view(np.uint16)
        assert d[b, 0] == d_ref
        dd = float(np.uint16(d[b, 0]).view(np.float16))
        if dd == 0:
            assert not q[b].any()
            continue
        ref = _exact_nearest_codes(x[b], dd)
        quot = x[b].astype(np.float64) / dd
        near_tie = np.abs(np.abs(quot - np.floor(quot)) - 0.5) < 1e-6 * np.maximum(1, np.abs(quot))
        mism = (q[b] != ref) & ~near_tie
        assert not mism.any(), (b, q[b][mism], ref[mism])
        assert np.abs(q[b]).max() <= 127
        assert np.abs(q[b]).max() >= 126  # the largest element maps to the end of the range


def test_quantizer_zero_and_tiny_blocks():
    x = np.zeros((2, 32), np.float32)
    x[1, 3] = 1e-30  # scale underflows binary16 -> zero block
    q, d = oracle.quantize(x)
    assert not q.any() and not d.any()


# ---------------------------------------------------------------- Q4 blocks
def _np_dequant(blocks):
    """Independent dequantization of canonical Q4 blocks [..., 18]."""
    d = blocks[..., 0:2].copy().view(np.float16)[..., 0].astype(np.float64)
    qs = blocks[..., 2:18]
    codes = np.concatenate([qs & 15, qs >> 4], axis=-1).astype(np.int64)  # elements 0..15, 16..31
    return codes, d


def test_block_dot_golden(golden):
    for qs_hex, acts, expect in golden("q4_block_dot.txt"):
        blk = np.zeros(18, np.uint8)
        blk[2:] = np.frombuffer(bytes.fromhex(qs_hex), np.uint8)
        a = np.array([int(v) for v in acts.split(",")], np.int8)
        assert oracle.block_dot(blk, a) == int(expect)


def test_block_dot_brute_force():
    blocks = synth.q4_blocks(synth.key(7, 99), 500)
    acts = RNG.integers(-127, 128, (500, 32)).astype(np.int8)
    codes, _ = _np_dequant(blocks)
    ref = ((codes - 8) * acts.astype(np.int64)).sum(axis=1)
    got = np.array([oracle.block_dot(blocks[i], acts[i]) for i in range(500)])
    assert np.array_equal(got, ref)
    assert np.abs(ref).max() <= 32512


def test_dequant_vs_independent():
    blocks = synth.q4_blocks(synth.key(7, 100), 300).reshape(10, 30, 18)
    codes, d = _np_dequant(blocks)
    ref = (d[..., None] * (codes - 8)).reshape(10, 30 * 32)
    assert np.array_equal(oracle.dequant(blocks), ref)


def test_row_dot_vs_dense_fp64():
    nb = 64
    row = synth.q4_blocks(synth.key(7, 101), nb)
    x = RNG.standard_normal(nb * 32).astype(np.float32)
    qa, da = oracle.quantize(x)
    r, abs_sum = oracle.row_dot(row, qa, da)
    w = oracle.dequant(row)
    codes, dw = _np_dequant(row)
    w_ind = (dw[:, None] * (codes - 8)).reshape(-1)
    a = qa.astype(np.float64) * np.repeat(da.view(np.float16).astype(np.float64), 32)
    ref = float(np.dot(w_ind, a))
    assert abs(r - ref) <= 4 * nb * 2.0 ** -52 * abs_sum
    assert np.array_equal(w, w_ind)


# ---------------------------------------------------------------- layer
def _tiny_layer(seed=0):
    wl = synth.WORKLOADS["tiny"]
    H, F, E, k, T = wl.hidden, wl.ffn, wl.n_experts, wl.top_k, 4
    gate = wl.expert_tensor(0, synth.KIND_GATE)
    up = wl.expert_tensor(0, synth.KIND_UP)
    down = wl.expert_tensor(0, synth.KIND_DOWN)
    x = wl.x(0, 0, T)
    logits = wl.logits(0, 0, T)
    return wl, H, F, E, k, T, gate, up, down, x, logits


def test_layer_vs_dense_fp64_brute_force():
    wl, H, F, E, k, T, gate, up, down, x, logits = _tiny_layer()
    idx, w = oracle.topk(logits, k)
    y, it = oracle.layer(x, idx, w, gate, up, down, H, F, want_intermediates=True)

    def deq(t):  # [E, rows, nb, 18] -> [E, rows, cols]
        codes, d = _np_dequant(t)
        return (d[..., None] * (codes - 8)).reshape(t.shape[0], t.shape[1], -1)

    Wg, Wu, Wd = deq(gate), deq(up), deq(down)
    # the oracle's quantized x is pinned by the quantizer tests
    xa = it["xq"].astype(np.float64) * np.repeat(it["xd"].view(np.float16).astype(np.float64), 32, axis=1)
    y_bf = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            a = t * k + j
            e = idx[t, j]
            g = Wg[e] @ xa[t]
            u = Wu[e] @ xa[t]
            np.testing.assert_allclose(it["g"][a], g, rtol=0, atol=1e-12 * np.abs(g).max())
            np.testing.assert_allclose(it["u"][a], u, rtol=0, atol=1e-12 * np.abs(u).max())
            h = g * u * expit(g)  # silu(gate) * up
            np.testing.assert_allclose(it["h"][a], h, rtol=1e-12, atol=1e-12)
            # quantized h, recomputed through the (pinned) quantizer from binary32 h
            hq, hd = oracle.quantize(h.astype(np.float32))
            assert np.array_equal(hq, it["hq"][a]) and np.array_equal(hd, it["hd"][a])
            ha = hq.astype(np.float64) * np.repeat(hd.view(np.float16).astype(np.float64), 32)
            y_bf[t] += w[t, j] * (Wd[e] @ ha)
    np.testing.assert_allclose(y, y_bf, rtol=1e-12, atol=1e-12 * np.abs(y_bf).max())
    # quantization-error envelope against unquantized activations (reported, loose)
    y_fp = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            g = Wg[e] @ x[t].astype(np.float64)
            u = Wu[e] @ x[t].astype(np.float64)
            y_fp[t] += w[t, j] * (Wd[e] @ (g * u * expit(g)))
    rel = np.linalg.norm(y - y_fp) / np.linalg.norm(y_fp)
    assert rel < 0.05


def test_down_combine_matches_layer():
    wl, H, F, E, k, T, gate, up, down, x, logits = _tiny_layer()
    idx, w = oracle.topk(logits, k)
    y, it = oracle.layer(x, idx, w, gate, up, down, H, F, want_intermediates=True)
    y2 = oracle.down_combine(idx, w, down, it["hq"], it["hd"], H, F)
    assert np.array_equal(y, y2)


def test_layer_experts_as_dict_equal_array():
    wl, H, F, E, k, T, gate, up, down, x, logits = _tiny_layer()
    idx, w = oracle.topk(logits, k)
    y = oracle.layer(x, idx, w, gate, up, down, H, F)
    used = sorted(set(idx.ravel().tolist()))
    y2 = oracle.layer(x, idx, w, {e: gate[e] for e in used}, {e: up[e] for e in used},
                      {e: down[e] for e in used}, H, F)
    assert np.array_equal(y, y2)


def test_generator_determinism():
    wl = synth.WORKLOADS["decode_b1_pool25"]
    a = wl.expert_tensor(3, synth.KIND_DOWN, 10, 14, threads=3)
    b = wl.expert_tensor(3, synth.KIND_DOWN, 12, 13, threads=1)
    assert np.array_equal(a[2], b[0])
    codes, d = _np_dequant(a)
    assert d.min() >= 0.005 - 1e-5 and d.max() <= 0.02 + 1e-5
    assert codes.min() == 0 and codes.max() == 15


def test_quantizer_exact_ties_round_half_even():
    # d = 2^-4 exactly: amax = 127/16 gives amax/127 = 1/16 (exact in binary16).
    # Elements at (n + 1/2) * d are exact ties; round-half-even picks the even code.
    d = 1.0 / 16
    halves = [0.5, 1.5, 2.5, 3.5, -0.5, -1.5, -2.5, 125.5, -126.5]
    expect = [0, 2, 2, 4, 0, -2, -2, 126, -126]
    x = np.zeros(32, np.float32)
    x[0] = 127 * d
    x[1:1 + len(halves)] = np.float32(halves) * np.float32(d)
    q, dd = oracle.quantize(x[None])
    assert dd[0, 0] == np.float16(d).view(np.uint16)
    assert q[0, 0] == 127
    assert q[0, 1:1 + len(halves)].tolist() == expect


def test_request_drift_is_a_seeded_jitter_of_the_table():
    wl = synth.WORKLOADS["prompt_then_decode_pool25"]
    base = synth.Workload("b", wl.hidden, wl.n_experts, wl.top_k, wl.ffn, wl.n_layers, routing="zipf",
                          zipf_s=wl.zipf_s, capacity=wl.capacity)
    for layer in (0, 17):
        p, q = wl.perm(layer), wl.request_perm(layer)
        assert np.array_equal(p, base.perm(layer)) and np.array_equal(base.request_perm(layer), p)
        assert sorted(q.tolist()) == list(range(wl.n_experts)) and not np.array_equal(p, q)
        assert np.array_equal(q, wl.request_perm(layer))
        # rank noise 0.15 E: the hot sets overlap but are not the same
        top = len(set(p[:128].tolist()) & set(q[:128].tolist()))
        assert 64 < top < 128
        assert np.array_equal(wl.seed_order(layer), p)


# ---------------------------------------------------------------- Q8_0 weights
def _np_dequant_q8(blocks):
    """Independent Q8_0 decode: numpy's float16 scale and int8 view of the codes."""
    d = np.ascontiguousarray(blocks[..., :2]).view(np.float16)[..., 0].astype(np.float64)
    codes = np.ascontiguousarray(blocks[..., 2:]).view(np.int8).astype(np.int64)
    return codes, d


def test_q8_block_dot_golden(golden):
    for qs_hex, acts, expect in golden("q8_block_dot.txt"):
        blk = np.zeros(34, np.uint8)
        blk[2:] = np.frombuffer(bytes.fromhex(qs_hex), np.uint8)
        a = np.array([int(v) for v in acts.split(",")], np.int8)
        assert oracle.block_dot(blk, a) == int(expect)


def test_q8_block_dot_brute_force_and_extremes():
    blocks = synth.q8_blocks(synth.key(7, 199), 500)
    acts = RNG.integers(-127, 128, (500, 32)).astype(np.int8)
    codes, _ = _np_dequant_q8(blocks)
    ref = (codes * acts.astype(np.int64)).sum(axis=1)
    got = np.array([oracle.block_dot(blocks[i], acts[i]) for i in range(500)])
    assert np.array_equal(got, ref)
    # every code value, against every activation value, one element at a time
    for qv in (-128, -127, -1, 0, 1, 126, 127):
        for av in (-127, -3, 0, 5, 127):
            blk = np.zeros(34, np.uint8)
            blk[2 + 13] = np.uint8(qv & 0xFF)
            a = np.zeros(32, np.int8)
            a[13] = av
            assert oracle.block_dot(blk, a) == qv * av


def test_q8_dequant_vs_independent():
    blocks = synth.q8_blocks(synth.key(7, 200), 300).reshape(10, 30, 34)
    codes, d = _np_dequant_q8(blocks)
    ref = (d[..., None] * codes).reshape(10, 30 * 32)
    assert np.array_equal(oracle.dequant(blocks), ref)
    assert codes.min() >= -127 and codes.max() <= 127 and np.abs(ref).max() <= 127 * 0.02 / 16 * 1.001


def test_q8_row_dot_vs_dense_fp64():
    nb = 64
    row = synth.q8_blocks(synth.key(7, 201), nb)
    x = RNG.standard_normal(nb * 32).astype(np.float32)
    qa, da = oracle.quantize(x)
    r, abs_sum = oracle.row_dot(row, qa, da)
    codes, dw = _np_dequant_q8(row)
    w_ind = (dw[:, None] * codes).reshape(-1)
    a = qa.astype(np.float64) * np.repeat(da.view(np.float16).astype(np.float64), 32)
    assert abs(r - float(np.dot(w_ind, a))) <= 4 * nb * 2.0 ** -52 * abs_sum


def test_q8_layer_vs_dense_fp64_brute_force():
    wl = synth.Workload("tiny_q8", 256, 8, 2, 512, 1, routing="normal", weight_format=synth.FMT_Q8_0)
    H, F, k, T = wl.hidden, wl.ffn, wl.top_k, 4
    gate, up, down = (wl.expert_tensor(0, kd) for kd in range(3))
    x, logits = wl.x(0, 0, T), wl.logits(0, 0, T)
    idx, w = oracle.topk(logits, k)
    y, it = oracle.layer(x, idx, w, gate, up, down, H, F, want_intermediates=True)

    def deq(t):
        codes, d = _np_dequant_q8(t)
        return (d[..., None] * codes).reshape(t.shape[0], t.shape[1], -1)

    Wg, Wu, Wd = deq(gate), deq(up), deq(down)
    xa = it["xq"].astype(np.float64) * np.repeat(it["xd"].view(np.float16).astype(np.float64), 32, axis=1)
    y_bf = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            a, e = t * k + j, idx[t, j]
            g, u = Wg[e] @ xa[t], Wu[e] @ xa[t]
            np.testing.assert_allclose(it["g"][a], g, rtol=0, atol=1e-12 * np.abs(g).max())
            np.testing.assert_allclose(it["u"][a], u, rtol=0, atol=1e-12 * np.abs(u).max())
            h = g * u * expit(g)
            hq, hd = oracle.quantize(h.astype(np.float32))
            assert np.array_equal(hq, it["hq"][a]) and np.array_equal(hd, it["hd"][a])
            ha = hq.astype(np.float64) * np.repeat(hd.view(np.float16).astype(np.float64), 32)
            y_bf[t] += w[t, j] * (Wd[e] @ ha)
    np.testing.assert_allclose(y, y_bf, rtol=1e-12, atol=1e-12 * np.abs(y_bf).max())
    assert np.array_equal(oracle.down_combine(idx, w, down, it["hq"], it["hd"], H, F), y)
    # the same weights in Q4 would give another layer: the format is really used
    q4 = synth.Workload("tiny", 256, 8, 2, 512, 1, routing="normal")
    y4 = oracle.layer(x, idx, w, *(q4.expert_tensor(0, kd) for kd in range(3)), H, F)
    assert not np.allclose(y4, y)


# ---------------------------------------------------------------- Q5_0 weights
def _np_dequant_q5(blocks):
    """Independent Q5_0 decode with numpy: float16 scale, 32-bit high-bit word,
    nibble planes unpacked with shifts."""
    d = np.ascontiguousarray(blocks[..., :2]).view(np.float16)[..., 0].astype(np.float64)
    qh = np.ascontiguousarray(blocks[..., 2:6]).view(np.uint32)[..., 0].astype(np.int64)
    qs = blocks[..., 6:22].astype(np.int64)
    lo = np.concatenate([qs & 15, qs >> 4], axis=-1)
    hi = (qh[..., None] >> np.arange(32)) & 1
    return lo + 16 * hi - 16, d


def test_q5_block_dot_golden(golden):
    for qh_hex, qs_hex, acts, expect in golden("q5_block_dot.txt"):
        blk = np.zeros(22, np.uint8)
        blk[2:6] = np.frombuffer(bytes.fromhex(qh_hex), np.uint8)
        blk[6:] = np.frombuffer(bytes.fromhex(qs_hex), np.uint8)
        a = np.array([int(v) for v in acts.split(",")], np.int8)
        assert oracle.block_dot(blk, a) == int(expect)


def test_q5_block_dot_brute_force_every_code():
    blocks = synth.q5_blocks(synth.key(7, 299), 500)
    acts = RNG.integers(-127, 128, (500, 32)).astype(np.int8)
    codes, _ = _np_dequant_q5(blocks)
    assert codes.min() == -16 and codes.max() == 15
    ref = (codes * acts.astype(np.int64)).sum(axis=1)
    got = np.array([oracle.block_dot(blocks[i], acts[i]) for i in range(500)])
    assert np.array_equal(got, ref)
    # each of the 32 codes at each element position picks out that element
    for q in range(32):
        for i in (0, 7, 15, 16, 30, 31):
            blk = np.zeros(22, np.uint8)
            blk[2 + i // 8] = ((q >> 4) & 1) << (i % 8)
            blk[6 + i % 16] = (q & 15) << (4 if i >= 16 else 0)
            a = np.zeros(32, np.int8)
            a[i] = 3
            # every other element has q = 0 (w = -16) against a = 0
            assert oracle.block_dot(blk, a) == 3 * (q - 16)


def test_q5_dequant_and_layer_vs_dense_fp64():
    blocks = synth.q5_blocks(synth.key(7, 300), 300).reshape(10, 30, 22)
    codes, d = _np_dequant_q5(blocks)
    assert np.array_equal(oracle.dequant(blocks), (d[..., None] * codes).reshape(10, 30 * 32))
    wl = synth.Workload("tiny_q5", 256, 8, 2, 512, 1, routing="normal", weight_format=synth.FMT_Q5_0)
    H, F, k, T = wl.hidden, wl.ffn, wl.top_k, 3
    gate, up, down = (wl.expert_tensor(0, kd) for kd in range(3))
    x, logits = wl.x(0, 0, T), wl.logits(0, 0, T)
    idx, w = oracle.topk(logits, k)
    y, it = oracle.layer(x, idx, w, gate, up, down, H, F, want_intermediates=True)

    def deq(t):
        c, dd = _np_dequant_q5(t)
        return (dd[..., None] * c).reshape(t.shape[0], t.shape[1], -1)

    Wg, Wu, Wd = deq(gate), deq(up), deq(down)
    xa = it["xq"].astype(np.float64) * np.repeat(it["xd"].view(np.float16).astype(np.float64), 32, axis=1)
    y_bf = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            a, e = t * k + j, idx[t, j]
            g, u = Wg[e] @ xa[t], Wu[e] @ xa[t]
            np.testing.assert_allclose(it["g"][a], g, rtol=0, atol=1e-12 * np.abs(g).max())
            h = g * u * expit(g)
            hq, hd = oracle.quantize(h.astype(np.float32))
            assert np.array_equal(hq, it["hq"][a]) and np.array_equal(hd, it["hd"][a])
            ha = hq.astype(np.float64) * np.repeat(hd.view(np.float16).astype(np.float64), 32)
            y_bf[t] += w[t, j] * (Wd[e] @ ha)
    np.testing.assert_allclose(y, y_bf, rtol=1e-12, atol=1e-12 * np.abs(y_bf).max())


# ---------------------------------------------------------------- shared expert
def test_shared_expert_layer_vs_dense_fp64():
    wl, H, F, E, k, T, gate, up, down, x, logits = _tiny_layer()
    sh = synth.Workload("shared", H, 1, 1, F, 1, routing="normal", seed=9)
    shared = tuple(sh.expert_tensor(0, kd)[0] for kd in range(3))
    idx, w = oracle.topk(logits, k)
    idx2, w2, g2, u2, d2 = oracle.with_shared(idx, w, gate, up, down, shared)
    assert idx2.shape == (T, k + 1) and (idx2[:, k] == E).all() and (w2[:, k] == 1.0).all()
    y, it = oracle.layer(x, idx2, w2, g2, u2, d2, H, F, want_intermediates=True)
    y0 = oracle.layer(x, idx, w, gate, up, down, H, F)

    def deq(b):
        codes, d = _np_dequant(b)
        return (d[..., None] * (codes - 8)).reshape(b.shape[0], -1)

    Sg, Su, Sd = (deq(t) for t in shared)
    xa = it["xq"].astype(np.float64) * np.repeat(it["xd"].view(np.float16).astype(np.float64), 32, axis=1)
    for t in range(T):
        g, u = Sg @ xa[t], Su @ xa[t]
        h = g * u * expit(g)
        hq, hd = oracle.quantize(h.astype(np.float32))
        a = t * (k + 1) + k
        assert np.array_equal(hq, it["hq"][a]) and np.array_equal(hd, it["hd"][a])
        o = Sd @ (hq.astype(np.float64) * np.repeat(hd.view(np.float16).astype(np.float64), 32))
        # y = (routed sum) + o_shared: the routed part is the plain layer
        np.testing.assert_allclose(y[t], y0[t] + o, rtol=1e-12, atol=1e-12 * np.abs(o).max())


# ---------------------------------------------------------------- Q4_K weights
def _np_dequant_q4k(sb):
    """Independent Q4_K decode with numpy: [..., 144] super-blocks -> codes
    [..., 256], per-sub-block scales and mins [..., 8], d and dmin."""
    sb = np.asarray(sb, np.uint8)
    d = np.ascontiguousarray(sb[..., 0:2]).view(np.float16)[..., 0].astype(np.float64)
    dmin = np.ascontiguousarray(sb[..., 2:4]).view(np.float16)[..., 0].astype(np.float64)
    b = sb[..., 4:16].astype(np.int64)
    sc = np.concatenate([b[..., 0:4] & 63, (b[..., 8:12] & 15) | ((b[..., 0:4] >> 6) << 4)], axis=-1)
    mn = np.concatenate([b[..., 4:8] & 63, (b[..., 8:12] >> 4) | ((b[..., 4:8] >> 6) << 4)], axis=-1)
    qs = sb[..., 16:144].astype(np.int64).reshape(sb.shape[:-1] + (4, 32))
    codes = np.stack([qs & 15, qs >> 4], axis=-2).reshape(sb.shape[:-1] + (256,))
    return codes, sc, mn, d, dmin


def _q4k_weights(sb):
    codes, sc, mn, d, dmin = _np_dequant_q4k(sb)
    scale = np.repeat(d[..., None] * sc, 32, axis=-1)
    mins = np.repeat(dmin[..., None] * mn, 32, axis=-1)
    return scale * codes - mins


def test_q4k_golden(golden):
    (d, dmin, scales, codes, over, dots, weights), = golden("q4k_superblock.txt")
    sb = np.zeros(144, np.uint8)
    sb[0:2] = np.array([int(d, 16) & 0xFF, int(d, 16) >> 8], np.uint8)  # little endian
    sb[2:4] = np.array([int(dmin, 16) & 0xFF, int(dmin, 16) >> 8], np.uint8)
    sb[4:16] = np.frombuffer(bytes.fromhex(scales.replace(" ", "")), np.uint8)
    hexs = "".join(h * int(n) for h, n in (t.split("*") for t in codes.split()))
    sb[16:] = np.frombuffer(bytes.fromhex(hexs), np.uint8)
    a = np.ones(256, np.int8)
    for kv in over.split(","):
        i, v = kv.split("=")
        a[int(i)] = int(v)
    assert oracle.subblock_dots(sb, a).tolist() == [int(v) for v in dots.split(",")]
    w = oracle.dequant(sb.reshape(1, 144))
    for kv in weights.split(","):
        i, v = kv.split("=")
        assert w[int(i)] == float(v)


def test_q4k_brute_force_vs_independent_decode():
    sbs = synth.q4k_blocks(synth.key(7, 400), 60)
    codes, *_ = _np_dequant_q4k(sbs)
    acts = RNG.integers(-127, 128, (60, 256)).astype(np.int8)
    for i in range(60):
        ref = (codes[i].reshape(8, 32) * acts[i].astype(np.int64).reshape(8, 32)).sum(axis=1)
        assert np.array_equal(oracle.subblock_dots(sbs[i], acts[i]), ref)
    assert np.array_equal(oracle.dequant(sbs.reshape(3, 20, 144)), _q4k_weights(sbs).reshape(3, 20 * 256))
    _, sc, mn, _, _ = _np_dequant_q4k(sbs)
    assert sc.min() == 0 and sc.max() == 63 and mn.min() == 0 and mn.max() == 63


def test_q4k_layer_vs_dense_fp64():
    wl = synth.Workload("tiny_q4k", 512, 8, 2, 256, 1, routing="normal", weight_format=synth.FMT_Q4_K)
    H, F, k, T = wl.hidden, wl.ffn, wl.top_k, 3
    gate, up, down = (wl.expert_tensor(0, kd) for kd in range(3))
    assert gate.shape == (8, F, H // 256, 144) and down.shape == (8, H, F // 256, 144)
    x, logits = wl.x(0, 0, T), wl.logits(0, 0, T)
    idx, w = oracle.topk(logits, k)
    y, it = oracle.layer(x, idx, w, gate, up, down, H, F, want_intermediates=True)

    def deq(t):
        return _q4k_weights(t).reshape(t.shape[0], t.shape[1], -1)

    Wg, Wu, Wd = deq(gate), deq(up), deq(down)
    xa = it["xq"].astype(np.float64) * np.repeat(it["xd"].view(np.float16).astype(np.float64), 32, axis=1)
    y_bf = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            a, e = t * k + j, idx[t, j]
            g, u = Wg[e] @ xa[t], Wu[e] @ xa[t]
            np.testing.assert_allclose(it["g"][a], g, rtol=0, atol=1e-12 * np.abs(g).max())
            h = g * u * expit(g)
            hq, hd = oracle.quantize(h.astype(np.float32))
            assert np.array_equal(hq, it["hq"][a]) and np.array_equal(hd, it["hd"][a])
            ha = hq.astype(np.float64) * np.repeat(hd.view(np.float16).astype(np.float64), 32)
            y_bf[t] += w[t, j] * (Wd[e] @ ha)
    np.testing.assert_allclose(y, y_bf, rtol=1e-12, atol=1e-12 * np.abs(y_bf).max())


# ---------------------------------------------------------------- Q5_K weights
def _np_q5k(sb):
    """Independent Q5_K decode with numpy: [..., 176] super-blocks -> codes
    [..., 256] (0..31), per-sub-block scales and mins [..., 8], d and dmin.
    The scale/min bytes and the code bytes decode as in Q4_K; bit j of qh[l]
    adds 16 to element l of sub-block j."""
    sb = np.asarray(sb, np.uint8)
    as_q4k = np.concatenate([sb[..., 0:16], sb[..., 48:176]], axis=-1)
    lo, sc, mn, d, dmin = _np_dequant_q4k(as_q4k)
    qh = sb[..., 16:48].astype(np.int64)                                  # [..., 32]
    hi = (qh[..., None, :] >> np.arange(8)[:, None]) & 1                 # [..., 8, 32]
    codes = lo + 16 * hi.reshape(sb.shape[:-1] + (256,))
    return codes, sc, mn, d, dmin


def _q5k_weights(sb):
    codes, sc, mn, d, dmin = _np_q5k(sb)
    scale = np.repeat(d[..., None] * sc, 32, axis=-1)
    mins = np.repeat(dmin[..., None] * mn, 32, axis=-1)
    return scale * codes - mins


def test_q5k_golden(golden):
    (d, dmin, scales, qh_over, codes, over, dots, weights), = golden("q5k_superblock.txt")
    sb = np.zeros(176, np.uint8)
    sb[0:2] = np.array([int(d, 16) & 0xFF, int(d, 16) >> 8], np.uint8)  # little endian
    sb[2:4] = np.array([int(dmin, 16) & 0xFF, int(dmin, 16) >> 8], np.uint8)
    sb[4:16] = np.frombuffer(bytes.fromhex(scales.replace(" ", "")), np.uint8)
    for kv in qh_over.split(","):
        i, v = kv.split("=")
        sb[16 + int(i)] = int(v, 16)
    hexs = "".join(h * int(n) for h, n in (t.split("*") for t in codes.split()))
    sb[48:] = np.frombuffer(bytes.fromhex(hexs), np.uint8)
    a = np.ones(256, np.int8)
    for kv in over.split(","):
        i, v = kv.split("=")
        a[int(i)] = int(v)
    assert oracle.q5k_subdots(sb, a).tolist() == [int(v) for v in dots.split(",")]
    w = oracle.dequant(sb.reshape(1, 176))
    for kv in weights.split(","):
        i, v = kv.split("=")
        assert w[int(i)] == float(v)


def test_q5k_brute_force_vs_independent_decode():
    sbs = synth.q5k_blocks(synth.key(7, 600), 60)
    codes, sc, mn, _, _ = _np_q5k(sbs)
    assert codes.min() == 0 and codes.max() == 31 and sc.max() == 63 and mn.max() == 63
    acts = RNG.integers(-127, 128, (60, 256)).astype(np.int8)
    for i in range(60):
        ref = (codes[i].reshape(8, 32) * acts[i].astype(np.int64).reshape(8, 32)).sum(axis=1)
        assert np.array_equal(oracle.q5k_subdots(sbs[i], acts[i]), ref)
    assert np.array_equal(oracle.dequant(sbs.reshape(3, 20, 176)), _q5k_weights(sbs).reshape(3, 20 * 256))


def test_q5k_layer_vs_dense_fp64():
    wl = synth.Workload("tiny_q5k", 512, 8, 2, 256, 1, routing="normal", weight_format=synth.FMT_Q5_K)
    H, F, k, T = wl.hidden, wl.ffn, wl.top_k, 3
    gate, up, down = (wl.expert_tensor(0, kd) for kd in range(3))
    assert gate.shape == (8, F, H // 256, 176) and down.shape == (8, H, F // 256, 176)
    x, logits = wl.x(0, 0, T), wl.logits(0, 0, T)
    idx, w = oracle.topk(logits, k)
    y, it = oracle.layer(x, idx, w, gate, up, down, H, F, want_intermediates=True)

    def deq(t):
        return _q5k_weights(t).reshape(t.shape[0], t.shape[1], -1)

    Wg, Wu, Wd = deq(gate), deq(up), deq(down)
    xa = it["xq"].astype(np.float64) * np.repeat(it["xd"].view(np.float16).astype(np.float64), 32, axis=1)
    y_bf = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            a, e = t * k + j, idx[t, j]
            g, u = Wg[e] @ xa[t], Wu[e] @ xa[t]
            np.testing.assert_allclose(it["g"][a], g, rtol=0, atol=1e-12 * np.abs(g).max())
            h = g * u * expit(g)
            hq, hd = oracle.quantize(h.astype(np.float32))
            assert np.array_equal(hq, it["hq"][a]) and np.array_equal(hd, it["hd"][a])
            ha = hq.astype(np.float64) * np.repeat(hd.view(np.float16).astype(np.float64), 32)
            y_bf[t] += w[t, j] * (Wd[e] @ ha)
    np.testing.assert_allclose(y, y_bf, rtol=1e-12, atol=1e-12 * np.abs(y_bf).max())


# ---------------------------------------------------------------- Q2_K weights
def _np_q2k(sb):
    """Independent Q2_K decode with numpy: [..., 84] super-blocks -> codes
    [..., 256] (0..3), scales and mins [..., 16], d and dmin.  Per
    128-weight half, code byte t carries element t of each 32-weight quarter
    m in bits 2m..2m+1."""
    sb = np.asarray(sb, np.uint8)
    sc = (sb[..., 0:16] & 15).astype(np.int64)
    mn = (sb[..., 0:16] >> 4).astype(np.int64)
    parts = []
    for n in range(2):
        qs = sb[..., 16 + 32 * n:16 + 32 * n + 32].astype(np.int64)
        parts += [(qs >> (2 * m)) & 3 for m in range(4)]
    codes = np.concatenate(parts, axis=-1)
    d = np.ascontiguousarray(sb[..., 80:82]).view(np.float16)[..., 0].astype(np.float64)
    dmin = np.ascontiguousarray(sb[..., 82:84]).view(np.float16)[..., 0].astype(np.float64)
    return codes, sc, mn, d, dmin


def _q2k_weights(sb):
    codes, sc, mn, d, dmin = _np_q2k(sb)
    return (np.repeat(d[..., None] * sc, 16, axis=-1) * codes - np.repeat(dmin[..., None] * mn, 16, axis=-1))


def test_q2k_golden(golden):
    (scales, qs_over, d, dmin, over, dots, weights), = golden("q2k_superblock.txt")
    sb = np.zeros(84, np.uint8)
    sb[0:16] = np.frombuffer(bytes.fromhex(scales), np.uint8)
    for kv in qs_over.split(","):
        i, v = kv.split("=")
        sb[16 + int(i)] = int(v, 16)
    sb[80:82] = np.array([int(d, 16) & 0xFF, int(d, 16) >> 8], np.uint8)  # little endian
    sb[82:84] = np.array([int(dmin, 16) & 0xFF, int(dmin, 16) >> 8], np.uint8)
    a = np.ones(256, np.int8)
    for kv in over.split(","):
        i, v = kv.split("=")
        a[int(i)] = int(v)
    assert oracle.q2k_subdots(sb, a).tolist() == [int(v) for v in dots.split(",")]
    w = oracle.dequant(sb.reshape(1, 84))
    for kv in weights.split(","):
        i, v = kv.split("=")
        assert w[int(i)] == float(v)


def test_q2k_brute_force_vs_independent_decode():
    sbs = synth.q2k_blocks(synth.key(7, 700), 60)
    codes, sc, mn, _, _ = _np_q2k(sbs)
    assert codes.min() == 0 and codes.max() == 3 and sc.max() == 15 and mn.max() == 15
    acts = RNG.integers(-127, 128, (60, 256)).astype(np.int8)
    for i in range(60):
        ref = (codes[i].reshape(16, 16) * acts[i].astype(np.int64).reshape(16, 16)).sum(axis=1)
        assert np.array_equal(oracle.q2k_subdots(sbs[i], acts[i]), ref)
    assert np.array_equal(oracle.dequant(sbs.reshape(3, 20, 84)), _q2k_weights(sbs).reshape(3, 20 * 256))


def test_q2k_layer_vs_dense_fp64():
    wl = synth.Workload("tiny_q2k", 512, 8, 2, 256, 1, routing="normal", weight_format=synth.FMT_Q2_K)
    H, F, k, T = wl.hidden, wl.ffn, wl.top_k, 3
    gate, up, down = (wl.expert_tensor(0, kd) for kd in range(3))
    assert gate.shape == (8, F, H // 256, 84) and down.shape == (8, H, F // 256, 84)
    x, logits = wl.x(0, 0, T), wl.logits(0, 0, T)
    idx, w = oracle.topk(logits, k)
    y, it = oracle.layer(x, idx, w, gate, up, down, H, F, want_intermediates=True)

    def deq(t):
        return _q2k_weights(t).reshape(t.shape[0], t.shape[1], -1)

    Wg, Wu, Wd = deq(gate), deq(up), deq(down)
    xa = it["xq"].astype(np.float64) * np.repeat(it["xd"].view(np.float16).astype(np.float64), 32, axis=1)
    y_bf = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            a, e = t * k + j, idx[t, j]
            g, u = Wg[e] @ xa[t], Wu[e] @ xa[t]
            np.testing.assert_allclose(it["g"][a], g, rtol=0, atol=1e-12 * np.abs(g).max())
            h = g * u * expit(g)
            hq, hd = oracle.quantize(h.astype(np.float32))
            assert np.array_equal(hq, it["hq"][a]) and np.array_equal(hd, it["hd"][a])
            ha = hq.astype(np.float64) * np.repeat(hd.view(np.float16).astype(np.float64), 32)
            y_bf[t] += w[t, j] * (Wd[e] @ ha)
    np.testing.assert_allclose(y, y_bf, rtol=1e-12, atol=1e-12 * np.abs(y_bf).max())


# ---------------------------------------------------------------- Q3_K weights
def _np_q3k(sb):
    """Independent Q3_K decode with numpy: [..., 110] super-blocks -> signed
    codes [..., 256] (-4..3), signed scales [..., 16], d.  Per 128-weight half
    n, code byte t and hmask byte t carry element t of each quarter m (bits
    2m..2m+1 of the code byte, bit 4n + m of the hmask byte)."""
    sb = np.asarray(sb, np.uint8)
    hm = sb[..., 0:32].astype(np.int64)
    parts = []
    for n in range(2):
        qs = sb[..., 32 + 32 * n:32 + 32 * n + 32].astype(np.int64)
        for m in range(4):
            low = (qs >> (2 * m)) & 3
            hbit = (hm >> (4 * n + m)) & 1
            parts.append(np.where(hbit == 1, low, low - 4))
    codes = np.concatenate(parts, axis=-1)
    b = sb[..., 96:108].astype(np.int64)
    low4 = np.concatenate([b[..., 0:8] & 15, b[..., 0:8] >> 4], axis=-1)          # j = 0..7, 8..15
    high2 = np.concatenate([(b[..., 8:12] >> (2 * q)) & 3 for q in range(4)], axis=-1)  # j = 4q + r
    sc = (low4 | (high2 << 4)) - 32
    d = np.ascontiguousarray(sb[..., 108:110]).view(np.float16)[..., 0].astype(np.float64)
    return codes, sc, d


def _q3k_weights(sb):
    codes, sc, d = _np_q3k(sb)
    return d[..., None] * np.repeat(sc, 16, axis=-1) * codes


def test_q3k_golden(golden):
    (hm_over, qs_over, scales, d, over, dots, weights), = golden("q3k_superblock.txt")
    sb = np.zeros(110, np.uint8)
    for kv in hm_over.split(","):
        i, v = kv.split("=")
        sb[int(i)] = int(v, 16)
    for kv in qs_over.split(","):
        i, v = kv.split("=")
        sb[32 + int(i)] = int(v, 16)
    sb[96:108] = np.frombuffer(bytes.fromhex(scales.replace(" ", "")), np.uint8)
    sb[108:110] = np.array([int(d, 16) & 0xFF, int(d, 16) >> 8], np.uint8)  # little endian
    a = np.ones(256, np.int8)
    for kv in over.split(","):
        i, v = kv.split("=")
        a[int(i)] = int(v)
    assert oracle.q3k_blockdots(sb, a).tolist() == [int(v) for v in dots.split(",")]
    w = oracle.dequant(sb.reshape(1, 110))
    for kv in weights.split(","):
        i, v = kv.split("=")
        assert w[int(i)] == float(v)


def test_q3k_brute_force_vs_independent_decode():
    sbs = synth.q3k_blocks(synth.key(7, 800), 60)
    codes, sc, _ = _np_q3k(sbs)
    assert codes.min() == -4 and codes.max() == 3 and sc.min() == -32 and sc.max() == 31
    acts = RNG.integers(-127, 128, (60, 256)).astype(np.int8)
    for i in range(60):
        t = (codes[i] * acts[i].astype(np.int64)).reshape(16, 16).sum(axis=1) * sc[i]
        assert np.array_equal(oracle.q3k_blockdots(sbs[i], acts[i]), t.reshape(8, 2).sum(axis=1))
    assert np.array_equal(oracle.dequant(sbs.reshape(3, 20, 110)), _q3k_weights(sbs).reshape(3, 20 * 256))


def test_q3k_layer_vs_dense_fp64():
    wl = synth.Workload("tiny_q3k", 512, 8, 2, 256, 1, routing="normal", weight_format=synth.FMT_Q3_K)
    H, F, k, T = wl.hidden, wl.ffn, wl.top_k, 3
    gate, up, down = (wl.expert_tensor(0, kd) for kd in range(3))
    assert gate.shape == (8, F, H // 256, 110) and down.shape == (8, H, F // 256, 110)
    x, logits = wl.x(0, 0, T), wl.logits(0, 0, T)
    idx, w = oracle.topk(logits, k)
    y, it = oracle.layer(x, idx, w, gate, up, down, H, F, want_intermediates=True)

    def deq(t):
        return _q3k_weights(t).reshape(t.shape[0], t.shape[1], -1)

    Wg, Wu, Wd = deq(gate), deq(up), deq(down)
    xa = it["xq"].astype(np.float64) * np.repeat(it["xd"].view(np.float16).astype(np.float64), 32, axis=1)
    y_bf = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            a, e = t * k + j, idx[t, j]
            g, u = Wg[e] @ xa[t], Wu[e] @ xa[t]
            np.testing.assert_allclose(it["g"][a], g, rtol=0, atol=1e-12 * np.abs(g).max())
            h = g * u * expit(g)
            hq, hd = oracle.quantize(h.astype(np.float32))
            assert np.array_equal(hq, it["hq"][a]) and np.array_equal(hd, it["hd"][a])
            ha = hq.astype(np.float64) * np.repeat(hd.view(np.float16).astype(np.float64), 32)
            y_bf[t] += w[t, j] * (Wd[e] @ ha)
    np.testing.assert_allclose(y, y_bf, rtol=1e-12, atol=1e-12 * np.abs(y_bf).max())


@pytest.mark.parametrize("fmt", [synth.FMT_Q8_0, synth.FMT_Q5_0, synth.FMT_Q4_K, synth.FMT_Q6_K, synth.FMT_Q5_K,
                                 synth.FMT_Q2_K, synth.FMT_Q3_K])
def test_generators_of_every_format_are_range_and_thread_independent(fmt):
    # the same expert's bytes whether generated alone or in a range, with any
    # thread count (the oracle and the library register the same weights)
    wl = synth.Workload("g", 512, 16, 2, 512, 2, weight_format=fmt)
    a = wl.expert_tensor(1, synth.KIND_DOWN, 3, 9, threads=4)
    b = wl.expert_tensor(1, synth.KIND_DOWN, 6, 7, threads=1)
    assert np.array_equal(a[3], b[0])
    assert a.shape[-1] == synth.BLOCK_BYTES[fmt] and a.shape[-2] == 512 // synth.BLOCK_ELEMS[fmt]
    # another tensor of the same layer draws other bytes
    c = wl.expert_tensor(1, synth.KIND_UP, 6, 7, threads=1)
    assert not np.array_equal(c, b)
    # every weight within the shared |w| <= 0.16 envelope
    w = oracle.dequant(a.reshape(-1, a.shape[-2], a.shape[-1]))
    assert np.abs(w).max() <= 0.16 * 1.01


# ---------------------------------------------------------------- Q6_K weights
def _np_q6k(sb):
    """Independent Q6_K decode with numpy: [..., 210] -> codes q [..., 256],
    signed scales [..., 16], d.  Per 128-weight half: ql bytes 0..31 give the
    low nibbles of quarter 0 (low) and 2 (high), bytes 32..63 those of
    quarters 1 and 3; qh byte l gives the high pairs of element l of every
    quarter (bits 0-1, 2-3, 4-5, 6-7 for quarters 0..3)."""
    sb = np.asarray(sb, np.uint8)
    lo_parts, hi_parts = [], []
    for n in range(2):
        ql = sb[..., 64 * n:64 * n + 64].astype(np.int64)
        qh = sb[..., 128 + 32 * n:128 + 32 * n + 32].astype(np.int64)
        lo_parts += [ql[..., 0:32] & 15, ql[..., 32:64] & 15, ql[..., 0:32] >> 4, ql[..., 32:64] >> 4]
        hi_parts += [(qh >> (2 * m)) & 3 for m in range(4)]
    lo = np.concatenate(lo_parts, axis=-1)
    hi = np.concatenate(hi_parts, axis=-1)
    sc = np.ascontiguousarray(sb[..., 192:208]).view(np.int8).astype(np.int64)
    d = np.ascontiguousarray(sb[..., 208:210]).view(np.float16)[..., 0].astype(np.float64)
    return lo | (hi << 4), sc, d


def _q6k_weights(sb):
    q, sc, d = _np_q6k(sb)
    return d[..., None] * np.repeat(sc, 16, axis=-1) * (q - 32)


def test_q6k_golden(golden):
    (ql_over, qh_over, d, dots, weights), = golden("q6k_superblock.txt")
    sb = np.zeros(210, np.uint8)
    for kv in ql_over.split(","):
        i, v = kv.split("=")
        sb[int(i)] = int(v, 16)
    for kv in qh_over.split(","):
        i, v = kv.split("=")
        sb[128 + int(i)] = int(v, 16)
    sb[192:208] = (np.arange(16) - 8).astype(np.int8).view(np.uint8)
    sb[208:210] = np.array([int(d, 16) & 0xFF, int(d, 16) >> 8], np.uint8)
    a = np.ones(256, np.int8)
    assert oracle.q6k_blockdots(sb, a).tolist() == [int(v) for v in dots.split(",")]
    w = oracle.dequant(sb.reshape(1, 210))
    for kv in weights.split(","):
        i, v = kv.split("=")
        assert w[int(i)] == float(v)


def test_q6k_brute_force_vs_independent_decode():
    sbs = synth.q6k_blocks(synth.key(7, 500), 60)
    q, sc, _ = _np_q6k(sbs)
    assert q.min() == 0 and q.max() == 63 and sc.min() == -64 and sc.max() == 63
    acts = RNG.integers(-127, 128, (60, 256)).astype(np.int8)
    for i in range(60):
        t = ((q[i] - 32) * acts[i].astype(np.int64)).reshape(16, 16).sum(axis=1) * sc[i]
        assert np.array_equal(oracle.q6k_blockdots(sbs[i], acts[i]), t.reshape(8, 2).sum(axis=1))
    assert np.array_equal(oracle.dequant(sbs.reshape(3, 20, 210)), _q6k_weights(sbs).reshape(3, 20 * 256))


def test_q6k_layer_vs_dense_fp64():
    wl = synth.Workload("tiny_q6k", 512, 8, 2, 256, 1, routing="normal", weight_format=synth.FMT_Q6_K)
    H, F, k, T = wl.hidden, wl.ffn, wl.top_k, 3
    gate, up, down = (wl.expert_tensor(0, kd) for kd in range(3))
    assert gate.shape == (8, F, H // 256, 210) and down.shape == (8, H, F // 256, 210)
    x, logits = wl.x(0, 0, T), wl.logits(0, 0, T)
    idx, w = oracle.topk(logits, k)
    y, it = oracle.layer(x, idx, w, gate, up, down, H, F, want_intermediates=True)

    def deq(t):
        return _q6k_weights(t).reshape(t.shape[0], t.shape[1], -1)

    Wg, Wu, Wd = deq(gate), deq(up), deq(down)
    xa = it["xq"].astype(np.float64) * np.repeat(it["xd"].view(np.float16).astype(np.float64), 32, axis=1)
    y_bf = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            a, e = t * k + j, idx[t, j]
            g, u = Wg[e] @ xa[t], Wu[e] @ xa[t]
            np.testing.assert_allclose(it["g"][a], g, rtol=0, atol=1e-12 * np.abs(g).max())
            h = g * u * expit(g)
            hq, hd = oracle.quantize(h.astype(np.float32))
            assert np.array_equal(hq, it["hq"][a]) and np.array_equal(hd, it["hd"][a])
            ha = hq.astype(np.float64) * np.repeat(hd.view(np.float16).astype(np.float64), 32)
            y_bf[t] += w[t, j] * (Wd[e] @ ha)
    np.testing.assert_allclose(y, y_bf, rtol=1e-12, atol=1e-12 * np.abs(y_bf).max())
