"""CPU checks of the C ABI: the library builds for sm_103a, loads, and exports every
function include/pic.h declares; host-only calls work without a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h")]


def declared_functions():
    names = set()
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w\s\*]*?\b(pic_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    from position_independent_kv_link_gb300 import _build, _lib
    if not os.path.exists(_lib.LIB_PATH):
        _build.build()
    return _lib.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("pic_model_create", "pic_store_create", "pic_compile", "pic_link", "pic_release_chunk",
              "pic_release_request", "pic_status_string", "pic_op_gemm", "pic_op_attention"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(lib._name)
    missing = [n for n in declared_functions() if not hasattr(raw, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    from position_independent_kv_link_gb300 import _lib
    assert set(declared_functions()) <= set(_lib.SIGNATURES)


def declared_arities():
    """name -> number of parameters, from the prototypes in include/*.h."""
    out = {}
    for h in HEADERS:
        src = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        for m in re.finditer(r"\b(pic_\w+)\s*\(([^;{}]*?)\)\s*;", src, flags=re.S):
            params = m.group(2).strip()
            out[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_arities_match_the_header():
    from position_independent_kv_link_gb300 import _lib
    ar = declared_arities()
    assert set(ar) == set(declared_functions())
    wrong = {n: (k, len(_lib.SIGNATURES[n][1])) for n, k in ar.items() if len(_lib.SIGNATURES[n][1]) != k}
    assert not wrong, wrong


def test_host_only_calls(lib):
    assert lib.pic_status_string(0) == b"PIC_OK"
    assert lib.pic_status_string(2) == b"PIC_ERR_OUT_OF_BLOCKS"
    assert b"sm_103a" in lib.pic_version()
    # invalid arguments are rejected before any CUDA call
    assert lib.pic_model_create(None, None, None) == 1
    assert lib.pic_release_chunk(None, 1) == 1
    assert lib.pic_op_gemm(0, None, None, None, 1, 1, 1, None) == 1
    assert lib.pic_compile_cached(None, None, None, 1, 0, None, None, None) == 1
    assert lib.pic_store_get_cache_stats(None, None) == 1
    assert lib.pic_store_evict(None, -1, None) == 1
    assert lib.pic_decode(None, None, None, 1, None, None, None, None, None) == 1


def test_build_targets_sm103a():
    from position_independent_kv_link_gb300 import _build
    assert "arch=compute_103a,code=sm_103a" in " ".join(_build.ARCH)
