"""ctypes declarations of libinjectscale.so (see include/injectscale.h)."""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_double, c_int, c_int32, c_int64, c_uint32, c_void_p

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libinjectscale.so")

IS_OK = 0
STATUS_NAMES = {0: "IS_OK", 1: "IS_ERR_INVALID_ARG", 2: "IS_ERR_OOM", 3: "IS_ERR_CAPACITY",
                4: "IS_ERR_OUT_OF_RANGE", 5: "IS_ERR_CUDA", 6: "IS_ERR_TIMEOUT", 7: "IS_ERR_DEVICE",
                8: "IS_ERR_UNSUPPORTED"}
IS_F32, IS_BF16, IS_F16, IS_FP8_E4M3 = 0, 1, 2, 3
IS_ST_FACT_RANGE, IS_ST_FACT_USER, IS_ST_BLOCK_TABLE, IS_ST_BLOCK_ID = 0x01, 0x02, 0x04, 0x08
IS_ST_USER_RANGE, IS_ST_POSITION, IS_ST_COUNT, IS_ST_TIMEOUT = 0x10, 0x20, 0x40, 0x80
IS_STAGE_SIMILARITY, IS_STAGE_TOPK, IS_STAGE_PLAN, IS_STAGE_INJECT = 0, 1, 2, 3
IS_MAX_K, IS_MAX_QUERIES, IS_MAX_REQUESTS, IS_EMB_TILE = 1024, 1024, 4096, 128
IS_NOALLOC_MAX_REQUESTS, IS_NOALLOC_MAX_FACTS = 256, 256
IS_MAX_CAPTURE_FACTS = 65536
IS_MAX_LAYERS_PER_CALL = 128
IS_RETRIEVAL_AUTO, IS_RETRIEVAL_PER_QUERY, IS_RETRIEVAL_BATCHED = 0, 1, 2
IS_KV_DEVICE, IS_KV_HOST = 0, 1


class StoreConfig(ctypes.Structure):
    _fields_ = [("num_layers", c_int32), ("num_kv_heads", c_int32), ("head_dim", c_int32),
                ("emb_dim", c_int32), ("kv_dtype", c_int32), ("emb_dtype", c_int32),
                ("max_facts", c_int64), ("max_tokens", c_int64), ("max_users", c_int32),
                ("max_queries", c_int32), ("max_k", c_int32), ("max_requests", c_int32),
                ("max_facts_per_user", c_int64), ("kv_placement", c_int32), ("reserved", c_int32)]


class RopeParams(ctypes.Structure):
    _fields_ = [("theta", c_double), ("style", c_int32), ("scaling", c_int32),
                ("factor", c_double), ("low_freq_factor", c_double),
                ("high_freq_factor", c_double), ("original_max_pos", c_int32)]


class CacheDesc(ctypes.Structure):
    _fields_ = [("block_size", c_int32), ("num_blocks", c_int32), ("dtype", c_int32),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


class StoreInfo(ctypes.Structure):
    _fields_ = [("n_facts", c_int64), ("n_tokens", c_int64), ("n_tiles", c_int32),
                ("max_user_tiles", c_int32), ("max_user_facts", c_int64), ("kv_bytes", c_int64),
                ("emb_bytes", c_int64), ("scratch_bytes", c_int64), ("num_sms", c_int32),
                ("kv_placement", c_int32)]


# name -> argtypes (restype is is_status_t unless listed in _RESTYPES)
SIGNATURES = {
    "is_store_create": [POINTER(StoreConfig), c_int, c_void_p, POINTER(c_void_p)],
    "is_store_destroy": [c_void_p],
    "is_store_add_facts": [c_void_p, c_int32, c_int32, POINTER(c_int32), c_void_p, c_void_p,
                           c_void_p, POINTER(c_int64), c_void_p],
    "is_store_info": [c_void_p, POINTER(StoreInfo)],
    "is_store_capture_begin": [c_void_p, c_int32, c_int32, POINTER(c_int32), POINTER(c_int32), c_void_p,
                               c_void_p],
    "is_store_capture_layer": [c_void_p, c_int32, c_void_p, c_void_p, c_void_p],
    "is_store_capture_end": [c_void_p, POINTER(c_int64), c_void_p],
    "is_store_capture_abort": [c_void_p],
    "is_retrieve_topk": [c_void_p, c_int32, c_void_p, c_void_p, c_int32, c_void_p, c_void_p,
                         c_void_p],
    "is_inject": [c_void_p, c_int32, c_void_p, c_void_p, c_int32, c_void_p, c_void_p,
                  POINTER(RopeParams), c_void_p, c_int32, POINTER(CacheDesc), c_void_p, c_void_p,
                  c_void_p, c_void_p],
    "is_inject_layer": [c_void_p, c_int32, c_int32, c_void_p, c_void_p, c_int32, c_void_p, c_void_p,
                        POINTER(RopeParams), c_void_p, c_int32, POINTER(CacheDesc), c_void_p,
                        c_void_p, c_void_p, c_void_p],
    "is_inject_layers": [c_void_p, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_int32, c_void_p,
                         c_void_p, POINTER(RopeParams), c_void_p, c_int32, POINTER(CacheDesc), c_void_p,
                         c_void_p, c_void_p, c_void_p],
    "is_retrieve_and_inject": [c_void_p, c_int32, c_void_p, c_void_p, c_int32, c_void_p,
                               POINTER(RopeParams), c_void_p, c_int32, POINTER(CacheDesc),
                               c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, c_void_p],
    "is_retrieve_and_inject_host": [c_void_p, c_int32, c_void_p, c_void_p, c_int32, c_void_p,
                                    POINTER(RopeParams), c_void_p, c_int32, POINTER(CacheDesc),
                                    c_void_p, c_void_p, c_void_p, c_void_p, c_void_p],
    "is_host_call_prepare": [c_void_p, c_int32, c_void_p, c_void_p, c_int32, c_void_p,
                             POINTER(RopeParams), c_void_p, c_int32, POINTER(CacheDesc),
                             c_void_p, c_void_p, c_void_p, c_void_p, c_void_p, POINTER(c_void_p)],
    "is_host_call_run": [c_void_p],
    "is_host_call_destroy": [c_void_p],
    "is_inject_noalloc": [c_void_p, c_int64, c_void_p, c_void_p, c_int64, c_int32, c_int32, c_int32,
                          c_int32, c_int32, c_int32, c_void_p, c_void_p, c_int32, c_void_p,
                          POINTER(RopeParams), c_void_p, c_int32, POINTER(CacheDesc), c_void_p,
                          c_void_p, c_void_p, c_void_p, c_void_p],
    "is_get_status": [c_void_p, c_void_p, POINTER(c_uint32)],
    "is_last_error_message": [],
    "is_status_string": [c_int],
    "is_rope_frequencies": [POINTER(RopeParams), c_int32, POINTER(c_double)],
    "is_set_retrieval_mode": [c_void_p, c_int32],
    "is_set_wait_budget": [c_void_p, c_int64],
    "is_set_timing": [c_void_p, c_int32],
    "is_get_timing": [c_void_p, c_int32, POINTER(c_double), POINTER(c_int64)],
    "is_reset_timing": [c_void_p],
}
_RESTYPES = {"is_last_error_message": c_char_p, "is_status_string": c_char_p}

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libinjectscale.so; raises if it has not been built (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with kv_cache_injection_gb300.build.build() "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    for name, argtypes in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = argtypes
        fn.restype = _RESTYPES.get(name, c_int)
    _lib = lib
    return lib
