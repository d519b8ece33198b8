"""Seeded synthetic inputs for the routed-expert MoE FFN workloads.

Shared, as data, by the CPU oracle and the CUDA path.  Nothing here computes
any step of the method: the module draws random numbers and lays them out in
the canonical input formats (fp32 activations and logits, canonical 18-byte Q4
blocks, expert permutations, seeding orders and pool capacities).

The C core (``synth.c``) is compiled on first use with the system C compiler.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_OUT = os.path.join(_HERE, "_build", "libsynth.so")
_lib = None

# Stream ids of the key tuple (seed, stream, a, b, c).
STREAM_WEIGHTS = 1
STREAM_X = 2
STREAM_LOGITS = 3
STREAM_PERM = 4
STREAM_DRIFT = 5
STREAM_ROUTER = 6

KIND_GATE, KIND_UP, KIND_DOWN = 0, 1, 2
Q4_BLOCK_BYTES = 18
Q8_BLOCK_BYTES = 34
Q5_BLOCK_BYTES = 22
Q4K_BLOCK_BYTES = 144  # one super-block of 256 weights
Q6K_BLOCK_BYTES = 210  # one super-block of 256 weights
Q5K_BLOCK_BYTES = 176  # one super-block of 256 weights
Q2K_BLOCK_BYTES = 84   # one super-block of 256 weights
Q3K_BLOCK_BYTES = 110  # one super-block of 256 weights
FMT_Q4, FMT_Q8_0, FMT_Q5_0, FMT_Q4_K, FMT_Q6_K, FMT_Q5_K, FMT_Q2_K, FMT_Q3_K = 0, 1, 2, 3, 4, 5, 6, 7
BLOCK_BYTES = {FMT_Q4: Q4_BLOCK_BYTES, FMT_Q8_0: Q8_BLOCK_BYTES, FMT_Q5_0: Q5_BLOCK_BYTES,
               FMT_Q4_K: Q4K_BLOCK_BYTES, FMT_Q6_K: Q6K_BLOCK_BYTES, FMT_Q5_K: Q5K_BLOCK_BYTES,
               FMT_Q2_K: Q2K_BLOCK_BYTES, FMT_Q3_K: Q3K_BLOCK_BYTES}
BLOCK_ELEMS = {FMT_Q4: 32, FMT_Q8_0: 32, FMT_Q5_0: 32, FMT_Q4_K: 256, FMT_Q6_K: 256, FMT_Q5_K: 256,
               FMT_Q2_K: 256, FMT_Q3_K: 256}
# scale ranges: |w| <= 0.16 in every format (|q - 8| <= 8 for Q4, |q| <= 127
# for Q8_0, |q - 16| <= 16 for Q5_0; Q4_K: d * 63 * 15 and dmin * 63 <= 0.16;
# Q6_K: d * 64 * 32 <= 0.16; Q5_K: d * 63 * 31 <= 0.16; Q2_K: d * 15 * 3 and
# dmin * 15 <= 0.16; Q3_K: d * 32 * 4 <= 0.16)
D_RANGE = {FMT_Q4: (0.005, 0.02), FMT_Q8_0: (0.005 / 16, 0.02 / 16), FMT_Q5_0: (0.0025, 0.01),
           FMT_Q4_K: (0.0000625, 0.00017), FMT_Q6_K: (0.00002, 0.000078), FMT_Q5_K: (0.00003, 0.000082),
           FMT_Q2_K: (0.001, 0.0035), FMT_Q3_K: (0.0004, 0.00125)}


def build(force: bool = False) -> str:
    """Compile the C generator into synth/_build/libsynth.so (if stale)."""
    if (not force and os.path.exists(_OUT)
            and os.path.getmtime(_OUT) >= os.path.getmtime(_SRC)):
        return _OUT
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    tmp = _OUT + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
           "-pthread", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _OUT)
    return _OUT


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        u64, i32, sz = ctypes.c_uint64, ctypes.c_int, ctypes.c_size_t
        vp, dbl = ctypes.c_void_p, ctypes.c_double
        L.synth_key.restype = u64
        L.synth_key.argtypes = [u64, u64, u64, u64, u64]
        L.synth_uniform_f64.argtypes = [u64, vp, sz]
        L.synth_normal_f32.argtypes = [u64, vp, sz]
        L.synth_q4_blocks.argtypes = [u64, vp, sz, dbl, dbl]
        L.synth_q4_experts.argtypes = [u64, u64, i32, i32, sz, vp, dbl, dbl, i32]
        L.synth_q8_blocks.argtypes = [u64, vp, sz, dbl, dbl]
        L.synth_q5_blocks.argtypes = [u64, vp, sz, dbl, dbl]
        L.synth_q4k_blocks.argtypes = [u64, vp, sz, dbl, dbl, dbl, dbl]
        L.synth_q6k_blocks.argtypes = [u64, vp, sz, dbl, dbl]
        L.synth_q5k_blocks.argtypes = [u64, vp, sz, dbl, dbl, dbl, dbl]
        L.synth_q2k_blocks.argtypes = [u64, vp, sz, dbl, dbl, dbl, dbl]
        L.synth_q3k_blocks.argtypes = [u64, vp, sz, dbl, dbl]
        L.synth_experts.argtypes = [u64, u64, i32, i32, sz, vp, dbl, dbl, i32, i32]
        L.synth_permutation.argtypes = [u64, vp, i32]
        L.synth_gumbel_logits.argtypes = [u64, vp, i32, i32, vp]
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def key(seed: int, stream: int, a: int = 0, b: int = 0, c: int = 0) -> int:
    return int(lib().synth_key(seed, stream, a, b, c))


def uniform(k: int, n: int) -> np.ndarray:
    out = np.empty(n, np.float64)
    lib().synth_uniform_f64(k, _ptr(out), n)
    return out


def normal(k: int, shape) -> np.ndarray:
    out = np.empty(shape, np.float32)
    lib().synth_normal_f32(k, _ptr(out), out.size)
    return out


def q4_blocks(k: int, n_blocks: int, dlo: float = 0.005, dhi: float = 0.02) -> np.ndarray:
    out = np.empty((n_blocks, Q4_BLOCK_BYTES), np.uint8)
    lib().synth_q4_blocks(k, _ptr(out), n_blocks, dlo, dhi)
    return out


def q8_blocks(k: int, n_blocks: int, dlo: float = D_RANGE[FMT_Q8_0][0],
              dhi: float = D_RANGE[FMT_Q8_0][1]) -> np.ndarray:
    out = np.empty((n_blocks, Q8_BLOCK_BYTES), np.uint8)
    lib().synth_q8_blocks(k, _ptr(out), n_blocks, dlo, dhi)
    return out


def q5_blocks(k: int, n_blocks: int, dlo: float = D_RANGE[FMT_Q5_0][0],
              dhi: float = D_RANGE[FMT_Q5_0][1]) -> np.ndarray:
    out = np.empty((n_blocks, Q5_BLOCK_BYTES), np.uint8)
    lib().synth_q5_blocks(k, _ptr(out), n_blocks, dlo, dhi)
    return out


def q4k_blocks(k: int, n_super: int, dlo: float = D_RANGE[FMT_Q4_K][0], dhi: float = D_RANGE[FMT_Q4_K][1],
               mlo: float = 0.0006, mhi: float = 0.0025) -> np.ndarray:
    out = np.empty((n_super, Q4K_BLOCK_BYTES), np.uint8)
    lib().synth_q4k_blocks(k, _ptr(out), n_super, dlo, dhi, mlo, mhi)
    return out


def q5k_blocks(k: int, n_super: int, dlo: float = D_RANGE[FMT_Q5_K][0], dhi: float = D_RANGE[FMT_Q5_K][1],
               mlo: float = 0.0006, mhi: float = 0.0025) -> np.ndarray:
    out = np.empty((n_super, Q5K_BLOCK_BYTES), np.uint8)
    lib().synth_q5k_blocks(k, _ptr(out), n_super, dlo, dhi, mlo, mhi)
    return out


def q2k_blocks(k: int, n_super: int, dlo: float = D_RANGE[FMT_Q2_K][0], dhi: float = D_RANGE[FMT_Q2_K][1],
               mlo: float = 0.002, mhi: float = 0.0106) -> np.ndarray:
    out = np.empty((n_super, Q2K_BLOCK_BYTES), np.uint8)
    lib().synth_q2k_blocks(k, _ptr(out), n_super, dlo, dhi, mlo, mhi)
    return out


def q3k_blocks(k: int, n_super: int, dlo: float = D_RANGE[FMT_Q3_K][0],
               dhi: float = D_RANGE[FMT_Q3_K][1]) -> np.ndarray:
    out = np.empty((n_super, Q3K_BLOCK_BYTES), np.uint8)
    lib().synth_q3k_blocks(k, _ptr(out), n_super, dlo, dhi)
    return out


def q6k_blocks(k: int, n_super: int, dlo: float = D_RANGE[FMT_Q6_K][0],
               dhi: float = D_RANGE[FMT_Q6_K][1]) -> np.ndarray:
    out = np.empty((n_super, Q6K_BLOCK_BYTES), np.uint8)
    lib().synth_q6k_blocks(k, _ptr(out), n_super, dlo, dhi)
    return out


def q4_experts(seed: int, tensor_tag: int, e_begin: int, e_end: int, rows: int, cols: int,
               out: np.ndarray | None = None, dlo: float | None = None, dhi: float | None = None,
               threads: int | None = None, fmt: int = FMT_Q4) -> np.ndarray:
    """Canonical weights (Q4, Q8_0 with fmt = 1, Q5_0 with fmt = 2) of experts
    [e_begin, e_end) of one expert tensor.

    Shape [n, rows, cols/32, 18, 34 or 22] uint8; expert e's bytes do not depend
    on the range it was generated in, nor on the thread count.
    """
    bb, per = BLOCK_BYTES[fmt], BLOCK_ELEMS[fmt]
    assert cols % per == 0
    dlo = D_RANGE[fmt][0] if dlo is None else dlo
    dhi = D_RANGE[fmt][1] if dhi is None else dhi
    n = e_end - e_begin
    nbe = rows * (cols // per)
    if out is None:
        out = np.empty((n, rows, cols // per, bb), np.uint8)
    assert out.nbytes == n * nbe * bb and out.flags["C_CONTIGUOUS"]
    if threads is None:
        threads = max(1, min(16, os.cpu_count() or 1))
    lib().synth_experts(seed, tensor_tag, e_begin, e_end, nbe, _ptr(out), dlo, dhi, threads, fmt)
    return out


def permutation(k: int, n: int) -> np.ndarray:
    out = np.empty(n, np.int32)
    lib().synth_permutation(k, _ptr(out), n)
    return out


def gumbel_logits(k: int, base: np.ndarray, T: int) -> np.ndarray:
    base = np.ascontiguousarray(base, np.float64)
    E = base.shape[0]
    out = np.empty((T, E), np.float32)
    lib().synth_gumbel_logits(k, _ptr(base), T, E, _ptr(out))
    return out


def zipf_probs(E: int, s: float) -> np.ndarray:
    """p(r) proportional to r^-s for ranks r = 1..E."""
    w = np.arange(1, E + 1, dtype=np.float64) ** (-s)
    return w / w.sum()


# ---------------------------------------------------------------------------
# Workloads.  Each names its shapes, routing popularity and pool residency.
# ---------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    hidden: int
    n_experts: int
    top_k: int
    ffn: int
    n_layers: int
    # popularity of the expert ranked r (1-based) under a per-layer
    # permutation: "normal" (plain N(0,1) logits), "zipf", or "mix".
    routing: str = "normal"
    zipf_s: float = 1.1
    mix_uniform: float = 0.0
    seed: int = 0
    # pool slots per layer (same for gate/up/down of a layer); None = all.
    capacity: list | None = None
    phases: list = field(default_factory=list)  # (label, n_tokens, n_steps)
    # request drift: the routed popularity ranks are the seeding table's
    # ranks plus N(0, (drift * E)^2) noise, re-ranked (0 = the table exactly)
    drift: float = 0.0
    # expert weight format: FMT_Q4 (canonical Q4 blocks), FMT_Q8_0 or FMT_Q5_0
    weight_format: int = FMT_Q4
    # router model (residual_rho > 0): each step's token runs through a
    # residual-stream stand-in, x_l = rho x_(l-1) + sqrt(1 - rho^2) xi_l with
    # x_0, xi_l ~ N(0, I), and layer l's logits are linear in its input,
    # bias_l + router_scale * R_l x_l (R_l: seeded rows of unit length, so
    # R_l x_l ~ N(0, 1) per expert; bias_l = the log popularity by rank);
    # layer l + 1's router applied to x_l then predicts its picks
    residual_rho: float = 0.0
    router_scale: float = math.pi / math.sqrt(6.0)

    def __post_init__(self):
        self._xcache = {}
        self._rcache = {}

    @property
    def tensor_shapes(self):
        H, F = self.hidden, self.ffn
        return {KIND_GATE: (F, H), KIND_UP: (F, H), KIND_DOWN: (H, F)}

    def tensor_tag(self, layer: int, kind: int) -> int:
        return layer * 3 + kind

    def expert_tensor(self, layer: int, kind: int, e_begin: int = 0, e_end: int | None = None,
                      out=None, threads=None) -> np.ndarray:
        rows, cols = self.tensor_shapes[kind]
        if e_end is None:
            e_end = self.n_experts
        return q4_experts(self.seed, self.tensor_tag(layer, kind), e_begin, e_end, rows, cols,
                          out=out, threads=threads, fmt=self.weight_format)

    def popularity(self) -> np.ndarray | None:
        E = self.n_experts
        if self.routing == "zipf":
            return zipf_probs(E, self.zipf_s)
        if self.routing == "mix":
            return self.mix_uniform / E + (1.0 - self.mix_uniform) * zipf_probs(E, self.zipf_s)
        return None

    def perm(self, layer: int) -> np.ndarray:
        """perm[r] = the expert holding popularity rank r+1 in this layer."""
        return permutation(key(self.seed, STREAM_PERM, layer), self.n_experts)

    def request_perm(self, layer: int) -> np.ndarray:
        """The permutation the logits are drawn with: perm(layer), or with
        drift its ranks jittered by seeded Gaussian noise and re-ranked."""
        base = self.perm(layer)
        if self.drift <= 0.0:
            return base
        z = normal(key(self.seed, STREAM_DRIFT, layer), (self.n_experts,)).astype(np.float64)
        order = np.argsort(np.arange(self.n_experts) + self.drift * self.n_experts * z, kind="stable")
        return base[order]

    def seed_order(self, layer: int) -> np.ndarray:
        """Synthetic routing-frequency table: experts by expected pick
        frequency, most frequent first (rank order of the popularity)."""
        if self.routing == "normal":
            return np.arange(self.n_experts, dtype=np.int32)
        return self.perm(layer).astype(np.int32)

    def layer_capacity(self, layer: int) -> int:
        if self.capacity is None:
            return self.n_experts
        return int(self.capacity[layer])

    def x(self, layer: int, step: int, T: int, phase: int = 0) -> np.ndarray:
        if self.residual_rho <= 0.0:
            return normal(key(self.seed, STREAM_X, layer, step, phase), (T, self.hidden))
        # residual chain, cached per (step, T, phase) from the last layer asked
        ck = (step, T, phase)
        l0, x = self._xcache.get(ck, (-1, None))
        if l0 > layer:
            l0, x = -1, None
        rho = self.residual_rho
        c = math.sqrt(1.0 - rho * rho)
        for l in range(l0 + 1, layer + 1):
            xi = normal(key(self.seed, STREAM_X, l, step, phase), (T, self.hidden))
            x = xi if l == 0 else (rho * x + c * xi).astype(np.float32)
        self._xcache = {ck: (layer, x)}
        return x.copy()

    def router(self, layer: int) -> np.ndarray:
        """R_l: [E][H] fp32, seeded rows of unit length (router model only)."""
        if layer not in self._rcache:
            r = normal(key(self.seed, STREAM_ROUTER, layer), (self.n_experts, self.hidden)).astype(np.float64)
            r /= np.linalg.norm(r, axis=1, keepdims=True)
            if len(self._rcache) >= 64:
                self._rcache.clear()
            self._rcache[layer] = r.astype(np.float32)
        return self._rcache[layer]

    def router_bias(self, layer: int) -> np.ndarray:
        """bias_l[e] = log popularity of e's rank in layer l (router model)."""
        base = np.empty(self.n_experts, np.float64)
        base[self.request_perm(layer)] = np.log(self.popularity())
        return base.astype(np.float32)

    def logits(self, layer: int, step: int, T: int, phase: int = 0) -> np.ndarray:
        if self.residual_rho > 0.0:
            x = self.x(layer, step, T, phase).astype(np.float64)
            z = x @ self.router(layer).astype(np.float64).T
            return (self.router_bias(layer).astype(np.float64)[None, :] + self.router_scale * z).astype(np.float32)
        k = key(self.seed, STREAM_LOGITS, layer, step, phase)
        p = self.popularity()
        if p is None:
            return normal(k, (T, self.n_experts))
        perm = self.request_perm(layer)
        base = np.empty(self.n_experts, np.float64)
        base[perm] = np.log(p)
        return gumbel_logits(k, base, T)

    def tensor_bytes(self, kind: int) -> int:
        rows, cols = self.tensor_shapes[kind]
        return rows * (cols // BLOCK_ELEMS[self.weight_format]) * BLOCK_BYTES[self.weight_format]


def _c1_capacity(L=48, E=512):
    # 40 layers fully resident, the other 8 hold a 60% hot set.
    part = int(math.floor(0.6 * E))
    return [part] * 8 + [E] * (L - 8)


WORKLOADS = {
    "tiny": Workload("tiny", hidden=256, n_experts=8, top_k=2, ffn=512, n_layers=1,
                     routing="normal", seed=0, phases=[("decode", 4, 1)]),
    "decode_b1_resident": Workload("decode_b1_resident", 2048, 512, 8, 1152, 48, routing="zipf",
                                   zipf_s=1.1, capacity=_c1_capacity(), phases=[("decode", 1, 128)]),
    # the decode workload with the router model (residual stream, linear
    # router, rho 0.9): layer l + 1's router on layer l's input predicts
    # its picks, for lookahead prefetch
    "decode_b1_resident_router": Workload("decode_b1_resident_router", 2048, 512, 8, 1152, 48, routing="zipf",
                                          zipf_s=1.1, capacity=_c1_capacity(), phases=[("decode", 1, 128)],
                                          residual_rho=0.9),
    "decode_b1_pool25": Workload("decode_b1_pool25", 2048, 512, 8, 1152, 48, routing="zipf",
                                 zipf_s=1.1, capacity=[128] * 48, phases=[("decode", 1, 256)]),
    # a 4096-token prompt, then decode, on the 25% pool; the request's expert
    # popularity drifts from the seeding table (rank noise 0.15 E)
    "prompt_then_decode_pool25": Workload("prompt_then_decode_pool25", 2048, 512, 8, 1152, 48, routing="zipf",
                                          zipf_s=1.1, capacity=[128] * 48, drift=0.15,
                                          phases=[("prefill", 4096, 1), ("decode", 1, 256)]),
    # Q8_0 expert weights: 16 layers of the decode shape, every expert resident
    "decode_b1_q8_resident16": Workload("decode_b1_q8_resident16", 2048, 512, 8, 1152, 16, routing="zipf",
                                        zipf_s=1.1, capacity=[512] * 16, phases=[("decode", 1, 64)],
                                        weight_format=FMT_Q8_0),
    # Q5_0 expert weights: the same 16 resident layers
    "decode_b1_q5_resident16": Workload("decode_b1_q5_resident16", 2048, 512, 8, 1152, 16, routing="zipf",
                                        zipf_s=1.1, capacity=[512] * 16, phases=[("decode", 1, 64)],
                                        weight_format=FMT_Q5_0),
    # Q4_K expert weights: 16 resident layers, FFN 1280 (the decode shape's
    # 1152 rounded up to whole 256-weight super-blocks)
    "decode_b1_q4k_resident16": Workload("decode_b1_q4k_resident16", 2048, 512, 8, 1280, 16, routing="zipf",
                                         zipf_s=1.1, capacity=[512] * 16, phases=[("decode", 1, 64)],
                                         weight_format=FMT_Q4_K),
    # Q6_K expert weights: the same 16 resident layers, FFN 1280
    "decode_b1_q6k_resident16": Workload("decode_b1_q6k_resident16", 2048, 512, 8, 1280, 16, routing="zipf",
                                         zipf_s=1.1, capacity=[512] * 16, phases=[("decode", 1, 64)],
                                         weight_format=FMT_Q6_K),
    # Q5_K expert weights: the same 16 resident layers, FFN 1280
    "decode_b1_q5k_resident16": Workload("decode_b1_q5k_resident16", 2048, 512, 8, 1280, 16, routing="zipf",
                                         zipf_s=1.1, capacity=[512] * 16, phases=[("decode", 1, 64)],
                                         weight_format=FMT_Q5_K),
    # Q4 weights with a shared expert per layer: the same 16 resident layers
    "decode_b1_shared_resident16": Workload("decode_b1_shared_resident16", 2048, 512, 8, 1152, 16,
                                            routing="zipf", zipf_s=1.1, capacity=[512] * 16,
                                            phases=[("decode", 1, 64)]),
    "prefill_t4096": Workload("prefill_t4096", 2048, 512, 8, 1152, 48, routing="zipf", zipf_s=1.1,
                              capacity=[384] * 48, phases=[("prefill", 4096, 1)]),
    "large_expert": Workload("large_expert", 2880, 128, 4, 2880, 36, routing="mix", zipf_s=0.8,
                             mix_uniform=0.5, capacity=[64] * 36,
                             phases=[("prefill", 512, 1), ("prefill", 4096, 1), ("prefill", 12288, 1),
                                     ("decode", 1, 16), ("decode", 8, 16), ("decode", 32, 16)]),
}
