"""Python binding of libmoecache.so (the GB300 routed-expert FFN with a
quantized HBM expert cache).

Argument marshalling only: every entry point forwards to the C ABI declared
in include/moe_cache.h, with the same name.  Device buffers may be given as
torch CUDA tensors or raw device addresses; host buffers as numpy arrays.
Every step of the path runs in the library's CUDA kernels: there is no
Python or CPU fallback, and importing this module fails loudly when the
library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_lib = None

MOE_OK = 0
ERRORS = {-1: "MOE_ERR_ARG", -2: "MOE_ERR_OOM", -3: "MOE_ERR_CUDA", -4: "MOE_ERR_NOT_PINNED",
          -5: "MOE_ERR_TIMEOUT", -6: "MOE_ERR_CAPACITY", -7: "MOE_ERR_STATE", -8: "MOE_ERR_FAULT"}
KIND_GATE, KIND_UP, KIND_DOWN = 0, 1, 2
FMT_Q4_0, FMT_Q8_0, FMT_Q5_0, FMT_Q4_K, FMT_Q6_K, FMT_Q5_K = 0, 1, 2, 3, 4, 5


class MoeError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{ERRORS.get(code, code)}: {msg}")
        self.code = code


class moe_cfg(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "hidden", "ffn", "n_experts", "top_k", "n_layers", "slots_per_tensor", "max_tokens", "window_tokens",
        "max_swaps_per_step", "renorm_topk", "poll_timeout_ms", "device", "weight_format", "shared_experts")]


class moe_stats_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "steps", "hits", "misses", "admissions", "evictions", "upload_bytes", "cold_bytes", "clock",
        "lookahead_predicted", "lookahead_hits")]


# Every symbol include/moe_cache.h declares, with (restype, argtypes).
_vp, _i32, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "moe_layer_init": (_i32, [ctypes.POINTER(moe_cfg), _vp, ctypes.POINTER(_vp)]),
    "register_expert_tensor": (_i32, [_vp, _i32, _i32, _vp, _i32, _i32, _i32, _vp, _i32, ctypes.POINTER(_i32)]),
    "register_shared_expert": (_i32, [_vp, _i32, _i32, _vp, _i32, _i32]),
    "route_topk": (_i32, [_vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp]),
    "moe_ffn_forward": (_i32, [_vp, _i32, _vp, _i32, _vp, _vp, _vp, _vp]),
    "moe_ffn_forward_routed": (_i32, [_vp, _i32, _vp, _vp, _i32, _vp, _vp, _vp, _vp]),
    "moe_set_expert_shard": (_i32, [_vp, _i32, _i32]),
    "moe_ffn_forward_rows": (_i32, [_vp, _i32, _vp, _i32, _vp, _vp, _vp, _i32, _vp]),
    "cache_step": (_i32, [_vp, _i32]),
    "miss_drain": (_i32, [_vp, _vp, _sz, ctypes.POINTER(_sz)]),
    "moe_pool_borrow": (_i32, [_vp, _i32, ctypes.POINTER(_vp), ctypes.POINTER(_sz)]),
    "moe_pool_return": (_i32, [_vp]),
    "moe_set_lookahead": (_i32, [_vp, _i32]),
    "moe_set_router": (_i32, [_vp, _i32, _vp, _vp]),
    "moe_set_global_pool": (_i32, [_vp, _i32]),
    "moe_set_upload_overlap": (_i32, [_vp, _i32]),
    "moe_set_preheat": (_i32, [_vp, _i32]),
    "moe_pool_snapshot": (_i32, [_vp, _vp, _vp]),
    "moe_cache_reset": (_i32, [_vp, _i32]),
    "moe_cache_snapshot": (_i32, [_vp, _i32, _vp, _vp, _vp, _vp, _vp]),
    "moe_cache_layout": (_i32, [_vp, _i32, _vp, _vp, _vp, _vp]),
    "moe_stats": (_i32, [_vp, ctypes.POINTER(moe_stats_t)]),
    "moe_last_error": (ctypes.c_char_p, [_vp]),
    "moe_destroy": (None, [_vp]),
    "moe_debug_block_dots": (_i32, [_vp, _i32, _i32, _i32, _i32, _vp, _vp]),
    "moe_debug_read": (_i32, [_vp, _i32, _vp, _sz]),
    "moe_probe_host_read": (_i32, [_vp, _sz, _i32, ctypes.POINTER(ctypes.c_double),
                                   ctypes.POINTER(ctypes.c_double)]),
    "moe_debug_fail_upload": (_i32, [_vp, _i32]),
    "moe_debug_busy": (_i32, [_vp, _i32]),
    "moe_debug_timing": (_i32, [_vp, _i32]),
    "moe_debug_timing_read": (_i32, [_vp, _vp, _vp]),
    "moe_expert_ffn_noalloc": (_i32, [_vp, _i32, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _vp]),
    "moe_expert_ffn_noalloc_status": (_i32, [_vp]),
}


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libmoecache.so (building it first if it is missing)."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            if not build_if_missing:
                raise ImportError(f"libmoecache.so not built at {path}")
            _build.build()
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _dev(x) -> int | None:
    """Device address of a torch tensor (or an int address)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        if not x.is_cuda:
            raise ValueError("expected a CUDA tensor")
        if not x.is_contiguous():
            raise ValueError("expected a contiguous tensor")
        return x.data_ptr()
    raise TypeError(f"cannot take a device address of {type(x)}")


def _host(a: np.ndarray | None) -> int | None:
    if a is None:
        return None
    if not a.flags["C_CONTIGUOUS"]:
        raise ValueError("expected a C-contiguous array")
    return a.ctypes.data


def _stream(s) -> int | None:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream  # torch.cuda.Stream


def _check(ctx, rc):
    if rc != MOE_OK:
        msg = load().moe_last_error(ctx)
        raise MoeError(rc, msg.decode() if msg else "")
    return rc


def moe_layer_init(hidden, ffn, n_experts, top_k, n_layers, slots_per_tensor, max_tokens, window_tokens=64,
                   max_swaps_per_step=0, renorm_topk=1, poll_timeout_ms=10000, device=0, stream=None,
                   weight_format=FMT_Q4_0, shared_experts=0) -> int:
    cfg = moe_cfg(hidden, ffn, n_experts, top_k, n_layers, slots_per_tensor, max_tokens, window_tokens,
                  max_swaps_per_step, renorm_topk, poll_timeout_ms, device, weight_format, shared_experts)
    out = ctypes.c_void_p()
    _check(None, load().moe_layer_init(ctypes.byref(cfg), _stream(stream), ctypes.byref(out)))
    return out.value


def register_expert_tensor(ctx, layer, kind, host_q4: np.ndarray, rows, cols, capacity, seed_order=None,
                           n_seed=0) -> int:
    so = None if seed_order is None else np.ascontiguousarray(seed_order, np.int32)
    tid = ctypes.c_int()
    _check(ctx, load().register_expert_tensor(ctx, layer, kind, _host(host_q4), rows, cols, capacity, _host(so),
                                              n_seed, ctypes.byref(tid)))
    return tid.value


def register_shared_expert(ctx, layer, kind, host_w: np.ndarray, rows, cols):
    return _check(ctx, load().register_shared_expert(ctx, layer, kind, _host(host_w), rows, cols))


def route_topk(ctx, logits, n_tokens, n_experts, k, idx, w, stream=None):
    return _check(ctx, load().route_topk(ctx, _dev(logits), n_tokens, n_experts, k, _dev(idx), _dev(w),
                                         _stream(stream)))


def moe_ffn_forward(ctx, layer, x, n_tokens, idx, w, y, stream=None):
    return _check(ctx, load().moe_ffn_forward(ctx, layer, _dev(x), n_tokens, _dev(idx), _dev(w), _dev(y),
                                              _stream(stream)))


def moe_ffn_forward_routed(ctx, layer, x, logits, n_tokens, idx, w, y, stream=None):
    return _check(ctx, load().moe_ffn_forward_routed(ctx, layer, _dev(x), _dev(logits), n_tokens, _dev(idx), _dev(w),
                                                     _dev(y), _stream(stream)))


def moe_set_expert_shard(ctx, expert_base, n_route):
    return _check(ctx, load().moe_set_expert_shard(ctx, expert_base, n_route))


def moe_ffn_forward_rows(ctx, layer, x, n_rows, idx, w, y, step_tokens, stream=None):
    return _check(ctx, load().moe_ffn_forward_rows(ctx, layer, _dev(x), n_rows, _dev(idx), _dev(w), _dev(y),
                                                   step_tokens, _stream(stream)))


def cache_step(ctx, n_tokens):
    return _check(ctx, load().cache_step(ctx, n_tokens))


def miss_drain(ctx, cap: int = 1 << 20) -> np.ndarray:
    out = np.empty(cap, np.uint32)
    n = ctypes.c_size_t()
    _check(ctx, load().miss_drain(ctx, _host(out), cap, ctypes.byref(n)))
    return out[: n.value].copy()


def moe_pool_borrow(ctx, n_slots):
    ws = ctypes.c_void_p()
    nb = ctypes.c_size_t()
    _check(ctx, load().moe_pool_borrow(ctx, n_slots, ctypes.byref(ws), ctypes.byref(nb)))
    return ws.value, nb.value


def moe_pool_return(ctx):
    return _check(ctx, load().moe_pool_return(ctx))


def moe_set_lookahead(ctx, enable=True):
    return _check(ctx, load().moe_set_lookahead(ctx, 1 if enable else 0))


def moe_set_router(ctx, layer, w, b=None):
    """Router of a layer for decode lookahead: w fp32 [E][H], b fp32 [E] (host)."""
    w = np.ascontiguousarray(w, np.float32)
    bb = None if b is None else np.ascontiguousarray(b, np.float32)
    return _check(ctx, load().moe_set_router(ctx, layer, _host(w), _host(bb)))


def moe_set_upload_overlap(ctx, enable=True):
    return _check(ctx, load().moe_set_upload_overlap(ctx, 1 if enable else 0))


def moe_set_global_pool(ctx, enable=True):
    return _check(ctx, load().moe_set_global_pool(ctx, 1 if enable else 0))


def moe_set_preheat(ctx, enable=True):
    return _check(ctx, load().moe_set_preheat(ctx, 1 if enable else 0))


def moe_cache_reset(ctx, global_pool=False):
    return _check(ctx, load().moe_cache_reset(ctx, 1 if global_pool else 0))


def moe_pool_snapshot(ctx, n_slots):
    """Owner key (tensor << 12 | expert, or -1) and stamp of each of the
    n_slots = 3L x slots_per_tensor arena slots."""
    owner = np.empty(max(1, n_slots), np.int32)
    stamps = np.empty(max(1, n_slots), np.uint32)
    _check(ctx, load().moe_pool_snapshot(ctx, _host(owner), _host(stamps)))
    return dict(owner=owner[:n_slots], stamps=stamps[:n_slots])


def moe_cache_snapshot(ctx, tensor_id, n_experts, slots_per_tensor):
    tbl = np.empty(n_experts, np.uint64)
    slot_of = np.empty(n_experts, np.int32)
    last_seen = np.empty(n_experts, np.int32)
    owner = np.empty(max(1, slots_per_tensor), np.int32)
    stamps = np.empty(max(1, slots_per_tensor), np.uint32)
    _check(ctx, load().moe_cache_snapshot(ctx, tensor_id, _host(tbl), _host(slot_of), _host(last_seen),
                                          _host(owner), _host(stamps)))
    return dict(tbl=tbl, slot_of=slot_of, last_seen=last_seen, owner=owner[:slots_per_tensor],
                stamps=stamps[:slots_per_tensor])


def moe_cache_layout(ctx, tensor_id):
    pb, hb, sb = ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_uint64()
    nt = ctypes.c_int32()
    _check(ctx, load().moe_cache_layout(ctx, tensor_id, ctypes.byref(pb), ctypes.byref(hb), ctypes.byref(sb),
                                        ctypes.byref(nt)))
    return dict(pool_base=pb.value, host_base=hb.value, slot_bytes=sb.value, n_tensors=nt.value)


def moe_stats(ctx) -> dict:
    s = moe_stats_t()
    _check(ctx, load().moe_stats(ctx, ctypes.byref(s)))
    return {n: getattr(s, n) for n, _ in moe_stats_t._fields_}


def moe_last_error(ctx) -> str:
    m = load().moe_last_error(ctx)
    return m.decode() if m else ""


def moe_destroy(ctx):
    if ctx:
        load().moe_destroy(ctx)


def moe_debug_block_dots(ctx, tensor_id, expert, row0, n_rows, qa, out):
    return _check(ctx, load().moe_debug_block_dots(ctx, tensor_id, expert, row0, n_rows, _dev(qa), _dev(out)))


def moe_debug_read(ctx, what, out: np.ndarray):
    return _check(ctx, load().moe_debug_read(ctx, what, _host(out), out.nbytes))


def moe_probe_host_read(host_pinned_addr: int, nbytes: int, iters: int = 5, with_copy: bool = True):
    g = ctypes.c_double()
    c = ctypes.c_double()
    _check(None, load().moe_probe_host_read(host_pinned_addr, nbytes, iters, ctypes.byref(g),
                                            ctypes.byref(c) if with_copy else None))
    return g.value, (c.value if with_copy else None)


def moe_debug_fail_upload(ctx, nth):
    return _check(ctx, load().moe_debug_fail_upload(ctx, nth))


def moe_debug_busy(ctx, microseconds):
    return _check(ctx, load().moe_debug_busy(ctx, microseconds))


def moe_debug_timing(ctx, enable=True):
    return _check(ctx, load().moe_debug_timing(ctx, int(enable)))


def moe_debug_timing_read(ctx, n_layers):
    gu = np.zeros(n_layers, np.float64)
    dn = np.zeros(n_layers, np.float64)
    _check(ctx, load().moe_debug_timing_read(ctx, _host(gu), _host(dn)))
    return gu, dn


def moe_expert_ffn_noalloc(x, n_tokens, idx, w, tbl, hidden, ffn, n_experts, top_k, y, stream=None):
    """One layer without any device allocation (scratch in a fixed device array)."""
    return _check(None, load().moe_expert_ffn_noalloc(_dev(x), n_tokens, _dev(idx), _dev(w), _dev(tbl), hidden, ffn,
                                                      n_experts, top_k, _dev(y), _stream(stream)))


def moe_expert_ffn_noalloc_status(stream=None):
    """Device-side status of the last allocation-free call on this device
    (raises MoeError(MOE_ERR_FAULT) when its kernel reported an error)."""
    return _check(None, load().moe_expert_ffn_noalloc_status(_stream(stream)))
