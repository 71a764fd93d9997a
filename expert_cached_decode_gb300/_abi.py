"""ctypes view of the C ABI in include/moe_gb300.h (argument marshalling only).

Every function here forwards to the shared library built from ``csrc/``;
there is no Python or CPU implementation of any step.  Loading fails loudly
when the library has not been built.
"""

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmoe_gb300.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_OOM", -3: "MOE_ERR_CUDA",
                -4: "MOE_ERR_HOST_PIN", -5: "MOE_ERR_TIMEOUT", -6: "MOE_ERR_STATE",
                -7: "MOE_ERR_UNIMPLEMENTED"}

ENTRY_POINTS = ("moe_layer_create", "moe_cache_configure", "moe_route_topk", "moe_forward",
                "moe_sync", "moe_cache_stats", "moe_cache_export", "moe_layer_destroy",
                "moe_route_topk_noalloc", "moe_set_miss_mode", "moe_debug_inject_failure",
                "moe_debug_set_wait_limit", "moe_last_error", "moe_pack_experts", "moe_forward_ahead",
                "moe_kv_create", "moe_kv_write", "moe_kv_read_blocks", "moe_kv_stats", "moe_kv_destroy")

MOE_MISS_HOST_COPY = 0
MOE_MISS_DEVICE_PULL = 1
MOE_INJECT_MISS_COPY = 1
MOE_INJECT_HOLD_ROUTER = 2
MOE_INJECT_HOST_REGISTER = 3
MOE_INJECT_DEVICE_ALLOC = 4


class MoeLayerDesc(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("f", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("n_layers", ctypes.c_int32), ("group", ctypes.c_int32),
                ("router_w", ctypes.c_void_p), ("router_b", ctypes.c_void_p),
                ("shared_q", ctypes.c_void_p), ("host_pool", ctypes.c_void_p),
                ("host_pool_entries", ctypes.c_int64), ("shared_weight", ctypes.c_float),
                ("host_pool_layout", ctypes.c_int32)]


MOE_POOL_CANONICAL = 0
MOE_POOL_DEVICE = 1


class MoeKvDesc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("cell_bytes", ctypes.c_int32), ("n_cells", ctypes.c_int64),
                ("resident_cells", ctypes.c_int64), ("block_cells", ctypes.c_int32),
                ("host_cells", ctypes.c_void_p)]


class MoeStats(ctypes.Structure):
    _fields_ = [("layer_calls", ctypes.c_int64), ("token_hits", ctypes.c_int64),
                ("token_misses", ctypes.c_int64), ("distinct_hits", ctypes.c_int64),
                ("distinct_misses", ctypes.c_int64), ("evictions", ctypes.c_int64),
                ("miss_bytes", ctypes.c_int64)]

    def as_dict(self):
        return {k: int(getattr(self, k)) for k, _ in self._fields_}


class MoeTrace(ctypes.Structure):
    _fields_ = [("idx", ctypes.c_void_p), ("w", ctypes.c_void_p), ("slot", ctypes.c_void_p),
                ("miss_expert", ctypes.c_void_p), ("miss_slot", ctypes.c_void_p),
                ("evicted_key", ctypes.c_void_p), ("n_miss", ctypes.c_int32),
                ("n_distinct", ctypes.c_int32), ("token_hits", ctypes.c_int64),
                ("token_misses", ctypes.c_int64)]


_lib = None


def load():
    """Load the CUDA library (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                           "(run __graft_entry__.build())")
    L = ctypes.CDLL(LIB_PATH)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    L.moe_layer_create.argtypes = [ctypes.POINTER(MoeLayerDesc), ctypes.POINTER(vp)]
    L.moe_cache_configure.argtypes = [vp, i64, vp, i64]
    L.moe_route_topk.argtypes = [vp, i32, vp, i32, vp, vp, vp]
    L.moe_forward.argtypes = [vp, i32, vp, i32, vp, vp, ctypes.POINTER(MoeTrace)]
    L.moe_sync.argtypes = [vp]
    L.moe_cache_stats.argtypes = [vp, ctypes.POINTER(MoeStats), vp]
    L.moe_cache_export.argtypes = [vp, vp, vp]
    L.moe_layer_destroy.argtypes = [vp]
    L.moe_layer_destroy.restype = None
    L.moe_route_topk_noalloc.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp]
    L.moe_set_miss_mode.argtypes = [vp, i32]
    L.moe_debug_inject_failure.argtypes = [i32, i64]
    L.moe_debug_set_wait_limit.argtypes = [vp, i64]
    L.moe_pack_experts.argtypes = [vp, vp, i64, i32, i32, vp]
    L.moe_forward_ahead.argtypes = [vp, i32, vp, i32, vp, vp, ctypes.POINTER(MoeTrace), i32, vp]
    L.moe_kv_create.argtypes = [ctypes.POINTER(MoeKvDesc), ctypes.POINTER(vp)]
    L.moe_kv_write.argtypes = [vp, i32, i64, i64, vp, vp]
    L.moe_kv_read_blocks.argtypes = [vp, i32, vp, i32, vp, vp]
    L.moe_kv_stats.argtypes = [vp, ctypes.POINTER(i64), ctypes.POINTER(i64)]
    L.moe_kv_destroy.argtypes = [vp]
    L.moe_kv_destroy.restype = None
    L.moe_last_error.argtypes = []
    L.moe_last_error.restype = ctypes.c_char_p
    for name in ("moe_layer_create", "moe_cache_configure", "moe_route_topk", "moe_forward",
                 "moe_sync", "moe_cache_stats", "moe_cache_export", "moe_route_topk_noalloc",
                 "moe_set_miss_mode", "moe_debug_inject_failure", "moe_debug_set_wait_limit",
                 "moe_pack_experts", "moe_forward_ahead", "moe_kv_create", "moe_kv_write",
                 "moe_kv_read_blocks", "moe_kv_stats"):
        getattr(L, name).restype = ctypes.c_int
    _lib = L
    return L


class MoeError(RuntimeError):
    def __init__(self, status, where):
        msg = load().moe_last_error().decode(errors="replace")
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def check(status, where):
    if status != MOE_OK:
        raise MoeError(status, where)
