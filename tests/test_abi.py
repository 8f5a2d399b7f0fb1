"""The C-ABI library: it loads, exports every function include/kvm.h declares,
and rejects bad arguments on the host before touching the GPU.  No test here
launches a kernel."""
import ctypes
import os
import re

import pytest

import sparse_attention_decode_04_b300 as K
from sparse_attention_decode_04_b300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return K.lib()


def declared_functions():
    inc = os.path.join(ROOT, "include")
    src = "\n".join(open(os.path.join(inc, f)).read() for f in sorted(os.listdir(inc)) if f.endswith(".h"))
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(kvm_[a-z_0-9]+)\s*\(", src, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert {"kvm_create", "kvm_destroy", "kvm_index_append", "kvm_score_select", "kvm_materialize",
            "kvm_decode_attn", "kvm_materialize_attn", "kvm_device_status", "kvm_step_attn",
            "kvm_select_control", "kvm_quantize_pages", "kvm_index_append_fp8", "kvm_materialize_fp8",
            "kvm_materialize_host", "kvm_attention_mass", "kvm_index_append_layers"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"{n} is declared in kvm.h but not exported"


def test_library_is_built_for_sm_103a_and_has_no_torch_dependency(lib):
    data = open(K.LIB_PATH, "rb").read()
    assert b"sm_103a" in data or b"sm_103" in data
    assert b"libtorch" not in data and b"libc10" not in data


def _params(**kw):
    base = dict(h_q=40, h_kv=8, d=128, n_sink=4, n_recent=32, top_k=988, rope_theta=1e6, max_blocks=8192,
                max_sessions=1, max_queries=1)
    base.update(kw)
    return K.Params(*[base[f] for f, _ in K.Params._fields_])


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), 2), (dict(h_q=41), 2), (dict(h_q=72, h_kv=8), 2), (dict(top_k=-1), 3),
    (dict(n_sink=0, n_recent=0, top_k=0), 3), (dict(rope_theta=0.5), 1), (dict(max_blocks=0), 2),
    (dict(max_blocks=10 ** 7), 2), (dict(max_sessions=65), 2), (dict(max_queries=0), 2)])
def test_create_rejects_bad_params_on_the_host(lib, kw, code):
    h = ctypes.c_void_p()
    p = _params(**kw)
    st = lib.kvm_create(ctypes.byref(p), ctypes.byref(h))
    assert st == code, (st, lib.kvm_last_error())
    assert h.value is None
    assert len(lib.kvm_last_error()) > 0


def test_calls_reject_null_context(lib):
    n = (ctypes.c_int64 * 1)(32)
    assert lib.kvm_index_append(None, None, 1, None, 1, n, n, None, None) == 1
    assert lib.kvm_score_select(None, None, 1, None, n, 1, None, None, None, None) == 1
    assert lib.kvm_materialize(None, None, None, 1, None, n, 1, None, None, None, None, None) == 1
    assert lib.kvm_decode_attn(None, None, None, None, None, 1, None, None) == 1
    assert lib.kvm_materialize_attn(None, None, None, 1, None, n, 1, None, None, None, None, None, None, None) == 1
    assert lib.kvm_step_attn(None, None, 4, None, None, None, 1, None, None) == 1
    assert lib.kvm_quantize_pages(None, None, 1, None, 1, None, None, None) == 1
    assert lib.kvm_index_append_fp8(None, None, None, 1, None, 1, n, n, None, None) == 1
    assert lib.kvm_materialize_fp8(None, None, None, None, None, 1, None, n, 1, None, None, None, None, None) == 1
    assert lib.kvm_materialize_host(None, None, None, 1, None, n, 1, None, None, None, None, None) == 1
    assert lib.kvm_attention_mass(None, None, None, 1, None, n, 1, None, None) == 1
    assert lib.kvm_index_append_layers(None, 2, None, 1, None, 1, n, n, None, None) == 1
    out = ctypes.c_uint32(0)
    assert lib.kvm_device_status(None, ctypes.byref(out), 0, None) == 1
    assert lib.kvm_destroy(None) == 0
    assert lib.kvm_scratch_bytes(None) == 0
    assert lib.kvm_status_string(6) == b"KVM_ERR_DEVICE"


def test_product_and_oracle_share_no_code():
    pkg = os.path.join(ROOT, "sparse_attention_decode_04_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(from|import)\s+oracle|kvm_oracle|#include.*oracle", text, re.M), f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith(".py"):
            text = open(os.path.join(ROOT, "oracle", f)).read()
            assert "sparse_attention_decode_04_b300" not in text and "libkvm" not in text, f


def test_debug_build_exports_the_same_symbols_and_says_so(lib):
    """libkvm_debug.so (device-side index checks) is the same interface; kvm_debug_checks tells them apart."""
    path = B.build(debug=True)
    dbg = ctypes.CDLL(path)
    for n in declared_functions():
        assert hasattr(dbg, n), f"{n} is declared in kvm.h but not exported by the debug build"
    dbg.kvm_debug_checks.restype = ctypes.c_int32
    lib.kvm_debug_checks.restype = ctypes.c_int32
    assert dbg.kvm_debug_checks() == 1 and lib.kvm_debug_checks() == 0
