"""Position-independent KV link (compile / LegoLink link) for GB300 (sm_103a).

The compute path is the CUDA library built from csrc/ (libpiclink.so); this package
is a thin binding over its C ABI (include/pic.h). Importing the package does not load
the library; creating a model or calling a kernel-level function does, and fails
loudly if it has not been built.
"""
from ._lib import LIB_PATH, PicError, load  # noqa: F401

__all__ = ["LIB_PATH", "PicError", "load", "PicModel", "PicStore", "gemm", "gemm_packed", "pack_weight", "attention",
           "attention_plan", "rope_table"]


def __getattr__(name):
    if name in ("PicModel", "PicStore", "gemm", "gemm_packed", "pack_weight", "attention", "attention_plan",
                "rope_table", "LinkResult", "DecodeResult"):
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
