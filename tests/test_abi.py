"""The C-ABI library loads and exports every symbol include/*.h declares
(no compute calls: this runs without a GPU)."""
import ctypes
import glob
import os
import re

import pytest

import quantized_expert_cache_gb300 as qec


def _read(path):
    with open(path) as f:
        return f.read()


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = _read(h)
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


# entry points whose first argument is the context
_CTX_CALLS = [n for n, (_, args) in qec.SIGNATURES.items()
              if n not in ("moe_layer_init", "moe_last_error", "moe_destroy", "moe_probe_host_read",
                           "moe_expert_ffn_noalloc", "moe_expert_ffn_noalloc_status")]


@pytest.mark.parametrize("name", _CTX_CALLS)
def test_every_context_call_rejects_a_null_context(name):
    # the header's error behaviour: a null context is MOE_ERR_ARG, checked
    # before any other argument and before any CUDA call
    lib = qec.load()
    fn = getattr(lib, name)
    args = [None if t is ctypes.c_void_p or issubclass(t, ctypes._Pointer) else 0 for t in qec.SIGNATURES[name][1]]
    assert fn(*args) == -1
    assert qec.moe_last_error(None)


def test_destroy_of_a_null_context_is_a_no_op():
    qec.load().moe_destroy(None)


def test_noalloc_and_probe_reject_bad_arguments_without_a_device():
    lib = qec.load()
    p = ctypes.c_void_p(16)  # never dereferenced: every case below fails its size checks first

    def call(n_tokens=1, hidden=256, ffn=256, n_experts=8, top_k=2, ptr=p):
        return lib.moe_expert_ffn_noalloc(ptr, n_tokens, ptr, ptr, ptr, hidden, ffn, n_experts, top_k, ptr, None)

    assert call(n_tokens=-1) == -1
    assert call(hidden=100) == -1 and call(ffn=48) == -1
    assert call(n_experts=0) == -1 and call(n_experts=4097) == -1
    assert call(top_k=0) == -1 and call(top_k=9) == -1
    assert call(n_tokens=33) == -1          # more tokens than the single launch holds
    assert call(n_tokens=1, ptr=None) == -1  # a null pointer
    # above the 8 MiB array: refused before any device work, and the bytes the
    # message names follow the header's estimate T*k*(4H + F + F/4) + T*(H + H/4)
    # plus the small tables
    T, k, H, F, E = 32, 8, 8192, 8192, 64
    assert call(n_tokens=T, hidden=H, ffn=F, n_experts=E, top_k=k) == -6
    msg = qec.moe_last_error(None)
    need = int(re.search(r"needs (\d+) scratch bytes", msg).group(1))
    estimate = T * k * (4 * H + F + F // 4) + T * (H + H // 4)
    assert estimate <= need <= estimate + 64 * 1024, (need, estimate)
    assert call(n_tokens=0, ptr=None) == 0   # nothing to do: no pointer is read
    gbs = ctypes.c_double()
    assert lib.moe_probe_host_read(None, 1 << 20, 1, ctypes.byref(gbs), None) == -1


def _declarations_with_docs():
    """(name, the comment just before its declaration) for every function the
    header declares; the hooks at the end share their section's note."""
    src = _read(os.path.join(ROOT, "include", "moe_cache.h"))
    comments = [(m.end(), m.group(1)) for m in re.finditer(r"/\*(.*?)\*/", src, flags=re.S)]
    hooks_at = src.index("inspection and measurement hooks")
    out = []
    for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([A-Za-z_][A-Za-z0-9_]*)\s*\(",
                         src, flags=re.M):
        before = [c for end, c in comments if end <= m.start()]
        assert before, m.group(1)
        doc = before[-1]
        if m.start() > hooks_at:
            doc += " (no counterpart on the source pages)"
        out.append((m.group(1), doc))
    return out


def test_every_declaration_cites_its_passage_and_states_its_errors():
    docs = _declarations_with_docs()
    assert {n for n, _ in docs} == _declared_functions()
    pages = ("Zapdev-labs", "neurall/llama.cpp", "mihailescu2m/llama.cpp", "mx-llama.cpp", "no counterpart",
             "No counterpart")
    for name, doc in docs:
        assert any(p in doc for p in pages), name
        assert any(k in doc for k in ("Errors", "MOE_ERR_", "Never fails", "Returns nothing")), name


def test_header_is_plain_c_and_the_library_links_from_c(tmp_path):
    # the boundary is a C ABI: the header compiles as C99 with warnings as
    # errors, and a C program linked against the library calls it
    import shutil
    import subprocess

    if shutil.which("gcc") is None:
        pytest.skip("needs gcc")
    qec.build.build()
    lib = qec.lib_path()
    src = tmp_path / "use_abi.c"
    src.write_text(r"""
#include <stdio.h>
#include <string.h>
#include "moe_cache.h"
int main(void) {
    moe_cfg cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.hidden = 100; /* not a multiple of 32 */
    cfg.ffn = 64; cfg.n_experts = 8; cfg.top_k = 2; cfg.n_layers = 1;
    cfg.slots_per_tensor = 8; cfg.max_tokens = 4; cfg.window_tokens = 64; cfg.renorm_topk = 1;
    moe_ctx *ctx = NULL;
    int rc = moe_layer_init(&cfg, NULL, &ctx);
    printf("%d %s\n", rc, moe_last_error(NULL));
    moe_destroy(NULL);
    return rc == MOE_ERR_ARG && ctx == NULL ? 0 : 1;
}
""")
    exe = tmp_path / "use_abi"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I",
                    os.path.join(ROOT, "include"), str(src), "-o", str(exe), lib,
                    "-Wl,-rpath," + os.path.dirname(lib)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.startswith("-1 ") and "hidden" in out.stdout
