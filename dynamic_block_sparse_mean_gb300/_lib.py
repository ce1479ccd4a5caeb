"""ctypes view of libbsa.so: the structs and prototypes of include/bsa.h.

Loading is lazy and loud: the first call that needs the library raises if the
shared object is missing or cannot be loaded.  There is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
# BSA_BOUNDS_CHECK=1 selects the bounds-checked build (libbsa_bounds.so, built by
# build(bounds_check=True)): same ABI, every table index range-checked on the device.
BOUNDS_CHECK = os.environ.get("BSA_BOUNDS_CHECK", "0") == "1"
LIB_PATH = os.path.join(PKG, "libbsa_bounds.so" if BOUNDS_CHECK else "libbsa.so")

BSA_OK = 0
STATUS_NAMES = {
    0: "BSA_OK", 1: "BSA_ERR_INVALID_ARG", 2: "BSA_ERR_UNSUPPORTED", 3: "BSA_ERR_WORKSPACE",
    4: "BSA_ERR_LAUNCH", 16: "BSA_ERR_INDEX_RANGE", 17: "BSA_ERR_INDEX_ORDER",
    18: "BSA_ERR_COUNT", 19: "BSA_ERR_TIMEOUT", 20: "BSA_ERR_CACHE",
}
BSA_BF16, BSA_FP32 = 0, 1
NUM_BUCKETS = 7
MAX_K = 256
MAX_GLOBAL = 32

c_i32p = ctypes.POINTER(ctypes.c_int32)
c_f32p = ctypes.POINTER(ctypes.c_float)


class Shape(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int32),
                ("max_seqlen", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block", ctypes.c_int32), ("max_blocks", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("cu_seqlens", ctypes.c_void_p)]


class RouteParams(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("k_max", ctypes.c_int32), ("k_min", ctypes.c_int32),
                ("tau_delta", ctypes.c_float), ("force_sink", ctypes.c_int32),
                ("window", ctypes.c_int32), ("num_global", ctypes.c_int32),
                ("global_blocks", ctypes.c_void_p), ("screen", ctypes.c_int32)]


class DecodeShape(ctypes.Structure):
    _fields_ = [("num_reqs", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("max_pages_per_req", ctypes.c_int32),
                ("num_phys_pages", ctypes.c_int32), ("top_k", ctypes.c_int32)]


class KVCache(ctypes.Structure):
    _fields_ = [("k_cache", ctypes.c_void_p), ("v_cache", ctypes.c_void_p),
                ("page_summ", ctypes.c_void_p), ("page_sum", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("prefix_lens", ctypes.c_void_p),
                ("max_pages_per_req", ctypes.c_int32), ("num_phys_pages", ctypes.c_int32),
                ("max_context_blocks", ctypes.c_int32)]


V = ctypes.c_void_p
SZ = ctypes.c_size_t
I32 = ctypes.c_int32
F32 = ctypes.c_float
PROTOTYPES = {
    "bsa_version": (I32, []),
    "bsa_bounds_checked": (I32, []),
    "bsa_status_string": (ctypes.c_char_p, [I32]),
    "bsa_block_summaries": (I32, [ctypes.POINTER(Shape), V, V, V]),
    "bsa_route_workspace_size": (SZ, [ctypes.POINTER(Shape), ctypes.POINTER(RouteParams)]),
    "bsa_route": (I32, [ctypes.POINTER(Shape), ctypes.POINTER(RouteParams), V, V, V, V, V, V, V,
                        SZ, V]),
    "bsa_worklist_workspace_size": (SZ, [ctypes.POINTER(Shape), I32]),
    "bsa_build_worklist": (I32, [ctypes.POINTER(Shape), I32, V, V, V, V, V, V, V, V, SZ, V]),
    "bsa_build_worklist_noalloc": (I32, [ctypes.POINTER(Shape), I32, V, V, V, V, V, V, V, V]),
    "bsa_attention_fwd": (I32, [ctypes.POINTER(Shape), V, V, V, V, V, V, V, F32, V, V, V, V]),
    "bsa_attention_bwd_workspace_size": (SZ, [ctypes.POINTER(Shape)]),
    "bsa_attention_bwd": (I32, [ctypes.POINTER(Shape), V, V, V, V, V, V, V, V, V, V, F32, V, V, V,
                                V, V, SZ, V]),
    "bsa_causal_worklist_capacity": (SZ, [ctypes.POINTER(Shape)]),
    "bsa_build_causal_worklist": (I32, [ctypes.POINTER(Shape), V, V, V, V, V, SZ, V]),
    "bsa_coverage": (I32, [ctypes.POINTER(Shape), V, V, V, V]),
    "bsa_recall_tiles_per_seq": (I32, [ctypes.POINTER(Shape)]),
    "bsa_token_recall": (I32, [ctypes.POINTER(Shape), I32, V, V, V, V, I32, V, I32, V, V, V]),
    "bsa_selftest_wait_timeout": (I32, [V, V]),
    "bsa_chunk_append": (I32, [ctypes.POINTER(Shape), ctypes.POINTER(KVCache), V, V, V, V]),
    "bsa_route_chunk_workspace_size": (SZ, [ctypes.POINTER(Shape), ctypes.POINTER(KVCache),
                                            ctypes.POINTER(RouteParams)]),
    "bsa_route_chunk": (I32, [ctypes.POINTER(Shape), ctypes.POINTER(KVCache),
                              ctypes.POINTER(RouteParams), V, V, V, V, V, V, SZ, V]),
    "bsa_build_worklist_chunk": (I32, [ctypes.POINTER(Shape), ctypes.POINTER(KVCache), I32, V, V,
                                       V, V, V, V, V, V, SZ, V]),
    "bsa_attention_chunk": (I32, [ctypes.POINTER(Shape), ctypes.POINTER(KVCache), V, V, V, V, V,
                                  F32, V, V, V, V]),
    "bsa_page_summaries": (I32, [ctypes.POINTER(DecodeShape), V, V, V, V, V]),
    "bsa_page_summaries_append": (I32, [ctypes.POINTER(DecodeShape), V, V, V, V, V, V]),
    "bsa_decode_workspace_size": (SZ, [ctypes.POINTER(DecodeShape)]),
    "bsa_decode_paged": (I32, [ctypes.POINTER(DecodeShape), V, V, V, V, V, V, F32, V, V, V, V, V,
                               V, SZ, V]),
}

_lib = None


def lib():
    """The loaded library (loaded once).  Raises if libbsa.so is absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built; run `python -m dynamic_block_sparse_mean_gb300.build` "
                "(or __graft_entry__.build()) on a machine with nvcc")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in PROTOTYPES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


class BsaError(RuntimeError):
    def __init__(self, call: str, code: int):
        self.code = code
        super().__init__(f"{call} failed: {STATUS_NAMES.get(code, code)}")


def check(call: str, code: int) -> None:
    if code != BSA_OK:
        raise BsaError(call, code)
