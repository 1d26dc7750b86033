"""ctypes declarations of the C ABI in include/pic.h (argument marshalling only)."""
import ctypes as C
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libpiclink.so")

PIC_OK, PIC_ERR_INVALID_ARG, PIC_ERR_OUT_OF_BLOCKS, PIC_ERR_CUDA, PIC_ERR_DEVICE_TIMEOUT, PIC_ERR_CAPACITY, \
    PIC_ERR_UNSUPPORTED, PIC_ERR_RANGE = range(8)
PIC_F32, PIC_BF16 = 0, 1


class ModelConfig(C.Structure):
    _fields_ = [("n_layers", C.c_int32), ("d_model", C.c_int32), ("n_heads", C.c_int32),
                ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32), ("ffn_dim", C.c_int32),
                ("vocab", C.c_int32), ("rope_base", C.c_double), ("rms_eps", C.c_float),
                ("dtype", C.c_int32), ("block_size", C.c_int32)]


class Weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("lm_head", C.c_void_p), ("final_norm", C.c_void_p),
                ("attn_norm", C.POINTER(C.c_void_p)), ("mlp_norm", C.POINTER(C.c_void_p)),
                ("w_qkv", C.POINTER(C.c_void_p)), ("w_o", C.POINTER(C.c_void_p)),
                ("w_gate_up", C.POINTER(C.c_void_p)), ("w_down", C.POINTER(C.c_void_p))]


class StoreConfig(C.Structure):
    _fields_ = [("num_blocks", C.c_int32), ("max_rows", C.c_int32), ("max_requests", C.c_int32),
                ("max_positions", C.c_int32), ("max_logit_rows", C.c_int32)]


class LinkRequest(C.Structure):
    _fields_ = [("chunks", C.POINTER(C.c_int32)), ("n_chunks", C.c_int32),
                ("query", C.POINTER(C.c_int32)), ("query_len", C.c_int32)]


class RequestInfo(C.Structure):
    _fields_ = [("n_selected", C.c_int32), ("selected", C.POINTER(C.c_int32)), ("slots", C.POINTER(C.c_int32)),
                ("n_pages", C.c_int32), ("page_table", C.POINTER(C.c_int32)), ("page_pos", C.POINTER(C.c_int32)),
                ("page_len", C.POINTER(C.c_int32)), ("n_private", C.c_int32),
                ("private_blocks", C.POINTER(C.c_int32))]


PROF_CLASSES = 6


class CacheStats(C.Structure):
    _fields_ = [("hits", C.c_int64), ("misses", C.c_int64), ("evictions", C.c_int64),
                ("cached_chunks", C.c_int32), ("unreferenced_chunks", C.c_int32),
                ("unreferenced_blocks", C.c_int32), ("blocks_in_use", C.c_int32), ("block_bytes", C.c_int64)]


class Profile(C.Structure):
    _fields_ = [("launches", C.c_int64 * PROF_CLASSES), ("ms", C.c_double * PROF_CLASSES),
                ("bytes", C.c_double * PROF_CLASSES), ("flops", C.c_double * PROF_CLASSES),
                ("total_launches", C.c_int64)]


P = C.c_void_p
I32 = C.c_int32
PI32 = C.POINTER(C.c_int32)

# name -> (restype, argtypes)
SIGNATURES = {
    "pic_status_string": (C.c_char_p, [I32]),
    "pic_last_error": (C.c_char_p, []),
    "pic_version": (C.c_char_p, []),
    "pic_model_create": (I32, [C.POINTER(ModelConfig), C.POINTER(Weights), C.POINTER(P)]),
    "pic_model_destroy": (I32, [P]),
    "pic_store_create": (I32, [P, C.POINTER(StoreConfig), P, P, C.POINTER(P)]),
    "pic_store_destroy": (I32, [P]),
    "pic_store_free_blocks": (I32, [P]),
    "pic_compile": (I32, [P, C.POINTER(PI32), PI32, I32, I32, P, PI32]),
    "pic_compile_cached": (I32, [P, C.POINTER(PI32), PI32, I32, I32, P, PI32, PI32]),
    "pic_store_get_cache_stats": (I32, [P, C.POINTER(CacheStats)]),
    "pic_store_evict": (I32, [P, I32, PI32]),
    "pic_chunk_import": (I32, [P, PI32, I32, P, P, P, PI32]),
    "pic_link": (I32, [P, C.POINTER(LinkRequest), I32, I32, I32, P, P, P, PI32]),
    "pic_link_dynamic": (I32, [P, C.POINTER(LinkRequest), I32, I32, I32, P, P, P, P, PI32]),
    "pic_decode": (I32, [P, PI32, PI32, I32, P, P, P, PI32, PI32]),
    "pic_request_get_info": (I32, [P, I32, C.POINTER(RequestInfo)]),
    "pic_chunk_get_blocks": (I32, [P, I32, PI32, C.POINTER(PI32)]),
    "pic_release_chunk": (I32, [P, I32]),
    "pic_release_request": (I32, [P, I32]),
    "pic_sync": (I32, [P, P]),
    "pic_debug_raise_device_flag": (I32, [I32]),
    "pic_profile_begin": (I32, [P]),
    "pic_profile_end": (I32, [P, C.POINTER(Profile)]),
    "pic_store_launch_count": (C.c_int64, [P]),
    "pic_op_gemm": (I32, [I32, P, P, P, I32, I32, I32, P]),
    "pic_op_pack_weight": (I32, [P, P, I32, I32, P]),
    "pic_op_gemm_packed": (I32, [P, P, P, I32, I32, I32, P]),
    "pic_op_attention_scratch_bytes": (C.c_size_t, [I32, I32, I32, I32, I32]),
    "pic_op_attention": (I32, [I32, I32, I32, I32, I32, P, PI32, P, P, PI32, PI32, PI32, I32, I32, P, I32, P, P,
                               C.c_size_t, P]),
    "pic_op_rope_table": (I32, [I32, I32, C.c_double, P, P]),
    "pic_op_attention_noalloc_max_scratch": (C.c_size_t, []),
    "pic_op_attention_plan": (I32, [I32, I32, I32, I32, I32, PI32, PI32, PI32, PI32, I32, PI32, I32, PI32, I32, PI32]),
    "pic_op_attention_noalloc": (I32, [I32, I32, I32, I32, I32, P, PI32, P, P, PI32, PI32, PI32, I32, I32, P, I32, P,
                                       P]),
}

_LIB = None


class PicError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{status_name(status)}: {msg}")
        self.status = status


def status_name(s):
    names = ["PIC_OK", "PIC_ERR_INVALID_ARG", "PIC_ERR_OUT_OF_BLOCKS", "PIC_ERR_CUDA", "PIC_ERR_DEVICE_TIMEOUT",
             "PIC_ERR_CAPACITY", "PIC_ERR_UNSUPPORTED", "PIC_ERR_RANGE"]
    return names[s] if 0 <= s < len(names) else f"status {s}"


def load(path: str = LIB_PATH) -> C.CDLL:
    """Loads the built library; raises if it is missing (there is no fallback path)."""
    global _LIB
    if _LIB is not None and path == LIB_PATH:
        return _LIB
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    if path == LIB_PATH:
        _LIB = lib
    return lib


def check(status: int):
    if status != PIC_OK:
        raise PicError(status, load().pic_last_error().decode())
