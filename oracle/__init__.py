"""ORACLE (test infrastructure only).

A plain, slow, single-threaded CPU restatement of the routed-expert MoE FFN
with a quantized expert cache, used to check the CUDA path.  Only the tests,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import
it.  It shares no code with the CUDA library, and the library never calls it.

- ``moe_oracle.c``: numerics (top-k, activation quantization, Q4, Q8_0, Q5_0, Q4_K and Q6_K block dots,
  SwiGLU, down projection and combine), binary64 with the integer-deciding
  steps in binary32 (see the header of that file);
- ``policy.py``: the admission / eviction policy of the expert pools.

Parity pins: every function here is checked by ``tests/test_oracle_*.py``
against brute force, closed forms, library routines or hand-traced
sequences; nothing here is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from .policy import PolicyOracle  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_OUT = os.path.join(_HERE, "_build", "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into oracle/_build/liboracle.so (if stale)."""
    if (not force and os.path.exists(_OUT)
            and os.path.getmtime(_OUT) >= os.path.getmtime(_SRC)):
        return _OUT
    os.makedirs(os.path.dirname(_OUT), exist_ok=True)
    tmp = _OUT + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _OUT)
    return _OUT


def configure(L):
    """Set the argument and result types of a loaded oracle library."""
    i32, vp, f32 = ctypes.c_int, ctypes.c_void_p, ctypes.c_float
    L.orc_h2d.restype = ctypes.c_double
    L.orc_h2d.argtypes = [ctypes.c_uint16]
    L.orc_f2h.restype = ctypes.c_uint16
    L.orc_f2h.argtypes = [f32]
    L.orc_topk.argtypes = [vp, i32, i32, i32, i32, vp, vp]
    L.orc_quantize_blocks.argtypes = [vp, i32, vp, vp]
    L.orc_dequant_fmt.argtypes = [vp, i32, i32, vp]
    L.orc_block_dot_fmt.restype = ctypes.c_int32
    L.orc_block_dot_fmt.argtypes = [vp, vp, i32]
    L.orc_row_dot_fmt.restype = ctypes.c_double
    L.orc_row_dot_fmt.argtypes = [vp, vp, vp, i32, i32, vp]
    L.orc_k4_subdots.argtypes = [vp, vp, vp]
    L.orc_k6_blockdots.argtypes = [vp, vp, vp]
    L.orc_k5_subdots.argtypes = [vp, vp, vp]
    L.orc_k2_subdots.argtypes = [vp, vp, vp]
    L.orc_k3_blockdots.argtypes = [vp, vp, vp]
    L.orc_expert.argtypes = [vp, vp, vp, i32, i32, vp, vp] + [vp] * 8 + [i32]
    L.orc_down_combine.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, i32]
    L.orc_layer.argtypes = [i32, i32, i32, i32, vp, vp, vp, vp, vp, vp, vp] + [vp] * 9 + [i32]
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = configure(ctypes.CDLL(build()))
    return _lib


def _p(a):
    if a is None:
        return None
    assert isinstance(a, np.ndarray) and a.flags["C_CONTIGUOUS"], "needs a C-contiguous array"
    return a.ctypes.data


def h2d(bits: int) -> float:
    return float(lib().orc_h2d(int(bits)))


def f2h(x: float) -> int:
    return int(lib().orc_f2h(float(x)))


def topk(logits: np.ndarray, k: int, renorm: bool = True):
    logits = np.ascontiguousarray(logits, np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    lib().orc_topk(_p(logits), T, E, k, int(renorm), _p(idx), _p(w))
    return idx, w


def quantize(x: np.ndarray):
    """x fp32 [..., n] (n % 32 == 0) -> (q int8 [..., n], d uint16 [..., n/32])."""
    x = np.ascontiguousarray(x, np.float32)
    n = x.size
    q = np.empty(x.shape, np.int8)
    d = np.empty(x.shape[:-1] + (x.shape[-1] // 32,), np.uint16)
    lib().orc_quantize_blocks(_p(x), n, _p(q), _p(d))
    return q, d


# canonical block size -> format (0: Q4, 1: Q8_0, 2: Q5_0, 3: Q4_K, 4: Q6_K, 5: Q5_K, 6: Q2_K, 7: Q3_K)
BLOCK_BYTES = {18: 0, 34: 1, 22: 2, 144: 3, 210: 4, 176: 5, 84: 6, 110: 7}
ELEMS = {0: 32, 1: 32, 2: 32, 3: 256, 4: 256, 5: 256, 6: 256, 7: 256}  # weights per canonical block


def _fmt(blocks) -> int:
    """Format of canonical blocks from their last dimension (18: Q4, 34: Q8_0, 22: Q5_0,
    144: Q4_K, 210: Q6_K, 176: Q5_K, 84: Q2_K and 110: Q3_K super-blocks of 256 weights)."""
    if blocks.shape[-1] not in BLOCK_BYTES:
        raise ValueError(f"unknown block size {blocks.shape[-1]}")
    return BLOCK_BYTES[blocks.shape[-1]]


def dequant(blocks: np.ndarray) -> np.ndarray:
    """Canonical blocks [..., nb, 18 (Q4), 34 (Q8_0) or 22 (Q5_0)] -> float64 [..., nb*32]."""
    blocks = np.ascontiguousarray(blocks, np.uint8)
    f = _fmt(blocks)
    n32 = blocks.size // blocks.shape[-1] * (ELEMS[f] // 32)
    out = np.empty(blocks.shape[:-2] + (blocks.shape[-2] * ELEMS[f],), np.float64)
    lib().orc_dequant_fmt(_p(blocks), n32, f, _p(out))
    return out


def subblock_dots(superblock: np.ndarray, qa: np.ndarray) -> np.ndarray:
    """Q4_K: raw integer dots sum q*a of the 8 sub-blocks of one super-block."""
    sb = np.ascontiguousarray(superblock, np.uint8)
    assert sb.size == 144 and qa.size == 256
    qa = np.ascontiguousarray(qa, np.int8)
    out = np.empty(8, np.int32)
    lib().orc_k4_subdots(_p(sb), _p(qa), _p(out))
    return out


def q5k_subdots(superblock: np.ndarray, qa: np.ndarray) -> np.ndarray:
    """Q5_K: raw integer dots sum q*a (q in 0..31) of the 8 sub-blocks of one super-block."""
    sb = np.ascontiguousarray(superblock, np.uint8)
    assert sb.size == 176 and qa.size == 256
    qa = np.ascontiguousarray(qa, np.int8)
    out = np.empty(8, np.int32)
    lib().orc_k5_subdots(_p(sb), _p(qa), _p(out))
    return out


def q2k_subdots(superblock: np.ndarray, qa: np.ndarray) -> np.ndarray:
    """Q2_K: raw integer dots sum q*a (q in 0..3) of the 16 sub-blocks of 16 of one super-block."""
    sb = np.ascontiguousarray(superblock, np.uint8)
    assert sb.size == 84 and qa.size == 256
    qa = np.ascontiguousarray(qa, np.int8)
    out = np.empty(16, np.int32)
    lib().orc_k2_subdots(_p(sb), _p(qa), _p(out))
    return out


def q3k_blockdots(superblock: np.ndarray, qa: np.ndarray) -> np.ndarray:
    """Q3_K: the integer dots of the 8 32-weight blocks of one super-block
    (each = the two 16-weight halves' sums of q * a times their scales)."""
    sb = np.ascontiguousarray(superblock, np.uint8)
    assert sb.size == 110 and qa.size == 256
    qa = np.ascontiguousarray(qa, np.int8)
    out = np.empty(8, np.int32)
    lib().orc_k3_blockdots(_p(sb), _p(qa), _p(out))
    return out


def q6k_blockdots(superblock: np.ndarray, qa: np.ndarray) -> np.ndarray:
    """Q6_K: the integer dots of the 8 32-weight blocks of one super-block
    (each = the two 16-weight halves' sums of (q - 32) * a times their scales)."""
    sb = np.ascontiguousarray(superblock, np.uint8)
    assert sb.size == 210 and qa.size == 256
    qa = np.ascontiguousarray(qa, np.int8)
    out = np.empty(8, np.int32)
    lib().orc_k6_blockdots(_p(sb), _p(qa), _p(out))
    return out


def block_dot(block: np.ndarray, qa: np.ndarray) -> int:
    block = np.ascontiguousarray(block, np.uint8)
    qa = np.ascontiguousarray(qa, np.int8)
    return int(lib().orc_block_dot_fmt(_p(block), _p(qa), _fmt(block)))


def row_dot(row: np.ndarray, qa: np.ndarray, da: np.ndarray):
    row = np.ascontiguousarray(row, np.uint8)
    qa = np.ascontiguousarray(qa, np.int8)
    da = np.ascontiguousarray(da, np.uint16)
    a = np.zeros(1, np.float64)
    f = _fmt(row)
    r = lib().orc_row_dot_fmt(_p(row), _p(qa), _p(da), row.size // row.shape[-1] * (ELEMS[f] // 32), f, _p(a))
    return float(r), float(a[0])


def _expert_ptrs(tensor):
    """Expert tensor given as an array [E, rows, nb, B] or a dict {e: [rows, nb, B]}
    (B = 18: Q4, 34: Q8_0, 22: Q5_0).  Returns (pointers, kept arrays, format)."""
    if isinstance(tensor, dict):
        E = max(tensor) + 1
        arrs = {e: np.ascontiguousarray(v, np.uint8) for e, v in tensor.items()}
        ptrs = (ctypes.c_void_p * E)(*[arrs[e].ctypes.data if e in arrs else None for e in range(E)])
        fmts = {_fmt(v) for v in arrs.values()}
        assert len(fmts) == 1, "one weight format per tensor"
        return ptrs, arrs, fmts.pop()
    t = np.ascontiguousarray(tensor, np.uint8)
    ptrs = (ctypes.c_void_p * t.shape[0])(*[t[e].ctypes.data for e in range(t.shape[0])])
    return ptrs, t, _fmt(t)


def layer(x, idx, w, gate, up, down, H, F, want_intermediates=False):
    """Whole layer: y float64 [T,H] (+ intermediates per assignment)."""
    x = np.ascontiguousarray(x, np.float32)
    idx = np.ascontiguousarray(idx, np.int32)
    w = np.ascontiguousarray(w, np.float64)
    T, k = idx.shape
    gp, g_keep, fg = _expert_ptrs(gate)
    upp, u_keep, fu = _expert_ptrs(up)
    dp, d_keep, fd = _expert_ptrs(down)
    assert fg == fu == fd, "gate, up and down share one weight format"
    y = np.empty((T, H), np.float64)
    out = {}
    if want_intermediates:
        A = T * k
        out = dict(xq=np.empty((T, H), np.int8), xd=np.empty((T, H // 32), np.uint16),
                   g=np.empty((A, F)), u=np.empty((A, F)), gabs=np.empty((A, F)), uabs=np.empty((A, F)),
                   h=np.empty((A, F)), hq=np.empty((A, F), np.int8), hd=np.empty((A, F // 32), np.uint16))
    o = out
    lib().orc_layer(T, H, F, k, _p(x), _p(idx), _p(w), ctypes.cast(gp, ctypes.c_void_p),
                    ctypes.cast(upp, ctypes.c_void_p), ctypes.cast(dp, ctypes.c_void_p), _p(y),
                    _p(o.get("xq")), _p(o.get("xd")), _p(o.get("g")), _p(o.get("u")), _p(o.get("gabs")),
                    _p(o.get("uabs")), _p(o.get("h")), _p(o.get("hq")), _p(o.get("hd")), fg)
    del g_keep, u_keep, d_keep
    return (y, out) if want_intermediates else y


def with_shared(idx, w, gate, up, down, shared, e_shared=None):
    """Routing and expert tensors of a layer with a shared expert (the
    shared-expert block among the fusion arguments of the dot kernels,
    Zapdev-labs/a6000-custom-kernels): every token also runs the shared
    expert on the same quantized x, and y = sum_j w_j o_j + o_shared.  The
    shared expert is appended as one more assignment per token, after the
    routed ones, with weight 1 and expert id E (one past the routed ids).
    shared: (gate, up, down) canonical tensors [rows, nb, B] of one expert;
    e_shared: the id to give it (default: one past every routed id given)."""
    idx = np.ascontiguousarray(idx, np.int32)
    T, k = idx.shape
    E = gate.shape[0] if not isinstance(gate, dict) else max(gate) + 1
    E = max(E, int(idx.max()) + 1 if idx.size else 0)
    if e_shared is not None:
        assert e_shared >= E, "the shared id must not collide with a routed one"
        E = int(e_shared)
    idx2 = np.concatenate([idx, np.full((T, 1), E, np.int32)], axis=1)
    w2 = np.concatenate([np.asarray(w, np.float64), np.ones((T, 1))], axis=1)

    def ext(t, s):
        d = dict(t) if isinstance(t, dict) else {e: t[e] for e in sorted(set(idx.ravel().tolist()))}
        d[E] = s
        return d

    return idx2, w2, ext(gate, shared[0]), ext(up, shared[1]), ext(down, shared[2])


def down_combine(idx, w, down, hq, hd, H, F):
    idx = np.ascontiguousarray(idx, np.int32)
    w = np.ascontiguousarray(w, np.float64)
    hq = np.ascontiguousarray(hq, np.int8)
    hd = np.ascontiguousarray(hd, np.uint16)
    T, k = idx.shape
    dp, keep, fd = _expert_ptrs(down)
    y = np.empty((T, H), np.float64)
    lib().orc_down_combine(T, H, F, k, _p(idx), _p(w), ctypes.cast(dp, ctypes.c_void_p), _p(hq), _p(hd), _p(y), fd)
    del keep
    return y
