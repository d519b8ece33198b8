"""The library's weight-format path, built for the host from its own sources
(the registration repack and the per-block code and scale traits the
kernels use, `tests/host/format_path_host.cpp`), against the oracle on the
CPU: for every format, canonical blocks from the seeded generators are
repacked into a plane blob exactly as registration does, and each block's
integer dot must equal the oracle's bit for bit (Q4_0 / Q8_0 / Q5_0: the
block dot with its offset; Q4_K / Q5_K: the raw sub-block dot; Q6_K: the
two sub-block dots folded with their scales); each block's fp32 term must
lie within the rounding of the fp32 expression the traits evaluate of the
exact binary64 value computed from independently decoded scales; and no
load may leave the blob or its natural alignment.  The GPU tests check the
same path on the device; this one runs wherever the CPU suite runs."""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
import synth
from test_oracle_pins import _np_dequant_q4k, _np_q5k

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "host", "format_path_host.cpp")
CSRC = os.path.join(ROOT, "quantized_expert_cache_gb300", "csrc")
OUT = os.path.join(ROOT, "tests", "host", "_build", "libformat_path_host.so")
U = 2.0 ** -24  # unit roundoff of binary32

FORMATS = [pytest.param(synth.FMT_Q4, id="q4_0"), pytest.param(synth.FMT_Q8_0, id="q8_0"),
           pytest.param(synth.FMT_Q5_0, id="q5_0"), pytest.param(synth.FMT_Q4_K, id="q4_k"),
           pytest.param(synth.FMT_Q6_K, id="q6_k"), pytest.param(synth.FMT_Q5_K, id="q5_k")]


def _cuda_include():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_fp16.h")):
            return os.path.join(cand, "include")
    return None


@pytest.fixture(scope="module")
def lib():
    inc = _cuda_include()
    if inc is None or shutil.which("g++") is None:
        pytest.skip("needs g++ and the CUDA headers")
    deps = [SRC] + [os.path.join(CSRC, h) for h in ("common.cuh", "repack.h")]
    if not os.path.exists(OUT) or any(os.path.getmtime(d) > os.path.getmtime(OUT) for d in deps):
        os.makedirs(os.path.dirname(OUT), exist_ok=True)
        tmp = OUT + f".{os.getpid()}.tmp"
        subprocess.run(["g++", "-std=c++17", "-O1", "-fPIC", "-shared", "-Wno-unknown-pragmas",
                        "-Wno-class-memaccess", "-I" + inc, "-I" + CSRC, SRC, "-o", tmp, "-lpthread"], check=True)
        os.replace(tmp, OUT)
    L = ctypes.CDLL(OUT)
    L.fp_blob_bytes.restype = ctypes.c_size_t
    L.fp_blob_bytes.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int]
    L.fp_repack.restype = None
    L.fp_repack.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                            ctypes.c_int, ctypes.c_size_t]
    L.fp_block_terms.restype = ctypes.c_long
    L.fp_block_terms.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return L


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _f16(b2):
    return np.ascontiguousarray(b2).view(np.float16)[..., 0].astype(np.float64)


def _host_path(lib, fmt, W, rows, nb, qa, da):
    """Repack one expert's canonical rows and evaluate every block."""
    size = lib.fp_blob_bytes(fmt, rows, nb)
    # the plane blob sits 16-byte aligned, as pool slots and host copies do
    raw = np.zeros(size + 64, np.uint8)
    off = (-raw.ctypes.data) % 16
    blob = raw[off:off + size]
    assert blob.ctypes.data % 16 == 0
    src = np.ascontiguousarray(W, np.uint8)
    lib.fp_repack(_ptr(src), _ptr(blob), fmt, 1, rows, nb, size)
    dots = np.zeros((rows, nb), np.int32)
    terms = np.zeros((rows, nb), np.float32)
    bad = lib.fp_block_terms(fmt, _ptr(blob), size, rows, nb, _ptr(qa), _ptr(da), _ptr(dots), _ptr(terms))
    return dots, terms.astype(np.float64), bad


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("rows,cols", [(40, 512), (7, 1024)])
def test_repack_and_traits_match_the_oracle(lib, fmt, rows, cols):
    wl = synth.Workload("host_fmt", cols, 3, 1, rows, 1, weight_format=fmt, seed=31 + fmt)
    W = wl.expert_tensor(0, 0)[2]          # one expert of a gate tensor: [rows][cols / 32 or / 256][bytes]
    assert W.shape[0] == rows
    nb = cols // 32
    rng = np.random.default_rng(100 + fmt)
    qa = rng.integers(-127, 128, cols).astype(np.int8)
    qa[:32] = -127                          # extreme activations against the first block
    qa[32:64] = 127
    # activation scales: binary16 values held in fp32, as the quantizer stores them
    da = rng.uniform(1e-3, 4e-2, nb).astype(np.float16).astype(np.float32)
    dots, terms, bad = _host_path(lib, fmt, W, rows, nb, qa, da)
    assert bad == 0, "a load left the blob or its alignment"

    asum = qa.astype(np.int64).reshape(nb, 32).sum(axis=1)
    dA = da.astype(np.float64)
    if fmt in (synth.FMT_Q4, synth.FMT_Q8_0, synth.FMT_Q5_0):
        ref_dot = np.array([[oracle.block_dot(W[r, b], qa[32 * b:32 * b + 32]) for b in range(nb)]
                            for r in range(rows)])
        d = _f16(W[..., 0:2])                                   # [rows][nb]
        exact = d * dA[None, :] * ref_dot
        bound = 3 * U * np.abs(exact)                           # (float)dot * (d * d_a): two roundings
    elif fmt == synth.FMT_Q6_K:
        ref_dot = np.array([np.concatenate([oracle.q6k_blockdots(W[r, u], qa[256 * u:256 * u + 256])
                                            for u in range(nb // 8)]) for r in range(rows)])
        d = np.repeat(_f16(W[..., 208:210]), 8, axis=1)         # the super-block's d for each of its blocks
        exact = d * dA[None, :] * ref_dot
        bound = 3 * U * np.abs(exact)
    else:
        sub = oracle.subblock_dots if fmt == synth.FMT_Q4_K else oracle.q5k_subdots
        ref_dot = np.array([np.concatenate([sub(W[r, u], qa[256 * u:256 * u + 256]) for u in range(nb // 8)])
                            for r in range(rows)])
        dec = _np_dequant_q4k if fmt == synth.FMT_Q4_K else _np_q5k
        _, sc, mn, dd, dmin = dec(W)                            # [rows][nb/8][8], [rows][nb/8]
        scale = (dd[..., None] * sc).reshape(rows, nb)          # d * sc_j, exact in binary32
        mins = (dmin[..., None] * mn).reshape(rows, nb)         # dmin * m_j, exact in binary32
        p1, p2 = scale * ref_dot, mins * asum[None, :]
        exact = dA[None, :] * (p1 - p2)
        # two products, a difference and the scale multiply, each rounded once
        bound = 4 * U * dA[None, :] * (np.abs(p1) + np.abs(p2))
    assert np.array_equal(dots, ref_dot), "integer block dots differ from the oracle"
    err = np.abs(terms - exact)
    assert (err <= bound + 1e-45).all(), float((err - bound).max())
    # the row sums the kernels accumulate equal the oracle's exact row dot
    # against the dequantized activations within the fp32 summation bound
    Wd = oracle.dequant(W[None])[0]                             # [rows][cols] binary64
    row_exact = Wd @ (np.repeat(dA, 32) * qa.astype(np.float64))
    assert np.allclose(exact.sum(axis=1), row_exact, rtol=1e-12, atol=1e-15)


def test_out_of_range_loads_are_counted(lib):
    # the check itself: a blob shorter than the layout needs is caught
    fmt, rows, cols = synth.FMT_Q4, 4, 64
    wl = synth.Workload("host_fmt", cols, 2, 1, rows, 1, weight_format=fmt, seed=5)
    W = wl.expert_tensor(0, 0)[0]
    nb = cols // 32
    size = lib.fp_blob_bytes(fmt, rows, nb)
    blob = np.zeros(size, np.uint8)
    lib.fp_repack(_ptr(np.ascontiguousarray(W)), _ptr(blob), fmt, 1, rows, nb, size)
    qa = np.ones(cols, np.int8)
    da = np.ones(nb, np.float32)
    dots = np.zeros((rows, nb), np.int32)
    terms = np.zeros((rows, nb), np.float32)
    assert lib.fp_block_terms(fmt, _ptr(blob), size - 2, rows, nb, _ptr(qa), _ptr(da), _ptr(dots), _ptr(terms)) > 0
