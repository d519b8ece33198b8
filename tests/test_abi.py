"""The C-ABI library loads and exports every symbol include/*.h declares
(no compute calls: this runs without a GPU)."""
import ctypes
import glob
import os
import re

import pytest

import quantized_expert_cache_gb300 as qec

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                             src, flags=re.M):
            names.add(m.group(1))
    return names


def test_header_declares_the_six_calls():
    names = _declared_functions()
    for n in ("moe_layer_init", "register_expert_tensor", "route_topk", "moe_ffn_forward", "cache_step",
              "miss_drain"):
        assert n in names


def test_library_exports_every_declared_symbol():
    qec.build.build()
    lib = ctypes.CDLL(qec.lib_path())
    names = _declared_functions()
    assert names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # the binding covers the same set
    assert names == set(qec.SIGNATURES)


def test_init_rejects_bad_config_without_a_device():
    with pytest.raises(qec.MoeError) as ei:
        qec.moe_layer_init(hidden=100, ffn=64, n_experts=8, top_k=2, n_layers=1, slots_per_tensor=8, max_tokens=4)
    assert ei.value.code == -1
    assert "hidden" in qec.moe_last_error(None)
    with pytest.raises(qec.MoeError):
        qec.moe_layer_init(hidden=256, ffn=64, n_experts=5000, top_k=2, n_layers=1, slots_per_tensor=8, max_tokens=4)
    with pytest.raises(qec.MoeError):
        qec.moe_layer_init(hidden=256, ffn=64, n_experts=8, top_k=9, n_layers=1, slots_per_tensor=8, max_tokens=4)


def test_init_rejects_bad_formats_and_shared_experts_without_a_device():
    def bad(**kw):
        args = dict(hidden=256, ffn=256, n_experts=8, top_k=2, n_layers=1, slots_per_tensor=8, max_tokens=4)
        args.update(kw)
        with pytest.raises(qec.MoeError) as ei:
            qec.moe_layer_init(**args)
        assert ei.value.code == -1
        return qec.moe_last_error(None)

    assert "weight_format" in bad(weight_format=7)
    # Q4_K needs widths that are whole 256-weight super-blocks
    bad(weight_format=qec.FMT_Q4_K, hidden=256, ffn=320)
    bad(weight_format=qec.FMT_Q4_K, hidden=320, ffn=256)
    # a shared expert takes table column E, so E + 1 ids must fit 12 bits
    bad(shared_experts=1, n_experts=4096, top_k=2)
    bad(shared_experts=2)
