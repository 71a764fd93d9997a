"""Python binding of the C ABI with the same entry-point names.

PyTorch supplies device memory and streams only; every step of the path runs
in the CUDA library.  Tensors are passed by ``data_ptr()`` and streams by
their ``cuda_stream`` handle.
"""

import ctypes

import numpy as np
import torch

from . import _abi
from ._abi import MoeKvDesc, MoeLayerDesc, MoeStats, MoeTrace, check


def _ptr(a):
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        if not a.is_contiguous():
            raise ValueError("tensor must be contiguous")
        return ctypes.c_void_p(a.data_ptr())
    if isinstance(a, np.ndarray):
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("array must be C-contiguous")
        return ctypes.c_void_p(a.ctypes.data)
    raise TypeError(f"unsupported buffer type {type(a)}")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class MoELayer:
    """One context of the library: a stack of n_layers MoE layers of one shape.

    router_w: [L, E, d] bf16 (torch bf16 tensor or uint16 array, host or device)
    router_b: [L, E] fp32 or None
    shared_q: [L, B_x] uint8 canonical packed shared experts
    host_pool: [P, B_x] uint8 canonical packed experts in host memory; keep it
               alive as long as the layer (pinned torch tensors avoid a
               registration)
    """

    def __init__(self, d, f, n_experts, top_k, n_layers, router_w, router_b, shared_q, host_pool,
                 host_pool_entries=0, shared_weight=1.0, group=32, host_pool_layout=0):
        self._lib = _abi.load()
        self._keep = (router_w, router_b, shared_q, host_pool)
        desc = MoeLayerDesc(d=d, f=f, n_experts=n_experts, top_k=top_k, n_layers=n_layers, group=group,
                            router_w=_ptr(router_w), router_b=_ptr(router_b), shared_q=_ptr(shared_q),
                            host_pool=_ptr(host_pool), host_pool_entries=host_pool_entries,
                            shared_weight=shared_weight, host_pool_layout=host_pool_layout)
        ctx = ctypes.c_void_p()
        check(self._lib.moe_layer_create(ctypes.byref(desc), ctypes.byref(ctx)), "moe_layer_create")
        self.ctx = ctx
        self.d, self.f, self.E, self.k, self.L = d, f, n_experts, top_k, n_layers
        self.capacity = 0

    # --- entry points ---------------------------------------------------------
    def moe_cache_configure(self, capacity, preload_keys=None):
        keys = None
        n = 0
        if preload_keys is not None:
            keys = np.ascontiguousarray(np.asarray(preload_keys, dtype=np.int32))
            n = keys.size
        check(self._lib.moe_cache_configure(self.ctx, int(capacity), _ptr(keys), n), "moe_cache_configure")
        self.capacity = int(capacity)

    def moe_route_topk(self, layer, x, idx, w, stream=None):
        T = x.shape[0]
        check(self._lib.moe_route_topk(self.ctx, layer, _ptr(x), T, _ptr(idx), _ptr(w), _stream(stream)),
              "moe_route_topk")

    def moe_forward(self, layer, x, y, stream=None, trace=False):
        """y[T, d] (fp32, device) <- layer-call on x[T, d] (bf16, device).
        With trace=True returns a dict of host arrays (synchronises)."""
        call = lambda tr: self._lib.moe_forward(self.ctx, layer, _ptr(x), x.shape[0], _ptr(y), _stream(stream), tr)
        return self._run(call, x.shape[0], trace, "moe_forward")

    def moe_forward_ahead(self, layer, x, y, next_layer=0, next_x=None, stream=None, trace=False):
        """moe_forward of (layer, x) that also routes the layer-call
        (next_layer, next_x), runs its cache step and copies its misses;
        that call must be the next forward on this layer (same x tensor)."""
        call = lambda tr: self._lib.moe_forward_ahead(self.ctx, layer, _ptr(x), x.shape[0], _ptr(y), _stream(stream),
                                                      tr, int(next_layer), _ptr(next_x))
        return self._run(call, x.shape[0], trace, "moe_forward_ahead")

    def _run(self, call, T, trace, where):
        if not trace:
            check(call(None), where)
            return None
        n = T * self.k
        bufs = {"idx": np.zeros(n, np.int32), "w": np.zeros(n, np.float32), "slot": np.zeros(n, np.int32),
                "miss_expert": np.zeros(n, np.int32), "miss_slot": np.zeros(n, np.int32),
                "evicted_key": np.zeros(n, np.int32)}
        tr = MoeTrace(**{k: _ptr(v) for k, v in bufs.items()})
        check(call(ctypes.byref(tr)), where)
        m = tr.n_miss
        return {"idx": bufs["idx"].reshape(T, self.k), "w": bufs["w"].reshape(T, self.k),
                "slot": bufs["slot"].reshape(T, self.k), "miss_expert": bufs["miss_expert"][:m].copy(),
                "miss_slot": bufs["miss_slot"][:m].copy(), "evicted_key": bufs["evicted_key"][:m].copy(),
                "n_distinct": int(tr.n_distinct), "token_hits": int(tr.token_hits),
                "token_misses": int(tr.token_misses)}

    def moe_set_miss_mode(self, mode):
        """mode: _abi.MOE_MISS_DEVICE_PULL (GPU reads the host pool itself) or
        _abi.MOE_MISS_HOST_COPY (host issues the miss copies)."""
        check(self._lib.moe_set_miss_mode(self.ctx, int(mode)), "moe_set_miss_mode")

    def moe_sync(self):
        check(self._lib.moe_sync(self.ctx), "moe_sync")

    def moe_debug_set_wait_limit(self, ns):
        """Test hook: limit (ns) of every bounded device wait of this context."""
        check(self._lib.moe_debug_set_wait_limit(self.ctx, int(ns)), "moe_debug_set_wait_limit")

    def moe_cache_stats(self, per_layer=False):
        tot = MoeStats()
        pl = (MoeStats * self.L)() if per_layer else None
        check(self._lib.moe_cache_stats(self.ctx, ctypes.byref(tot), pl), "moe_cache_stats")
        if per_layer:
            return tot.as_dict(), [s.as_dict() for s in pl]
        return tot.as_dict()

    def moe_cache_export(self):
        owner = np.zeros(self.capacity, np.int32)
        stamp = np.zeros(self.capacity, np.int64)
        check(self._lib.moe_cache_export(self.ctx, _ptr(owner), _ptr(stamp)), "moe_cache_export")
        return owner, stamp

    def moe_layer_destroy(self):
        if self.ctx is not None and self.ctx.value:
            self._lib.moe_layer_destroy(self.ctx)
        self.ctx = None

    close = moe_layer_destroy

    def __del__(self):
        try:
            self.moe_layer_destroy()
        except Exception:
            pass


def moe_route_topk_noalloc(x, router_w, router_b, top_k, idx, w, stream=None):
    """Binding of the allocation-free router entry point: x[T, d] bf16,
    router_w[E, d] bf16, router_b[E] fp32 or None (all device tensors);
    writes idx[T, k] int32 and w[T, k] fp32 (device)."""
    L = _abi.load()
    T, d = x.shape
    E = router_w.shape[0]
    check(L.moe_route_topk_noalloc(_ptr(x), _ptr(router_w), _ptr(router_b), T, d, E, top_k, _ptr(idx), _ptr(w),
                                   _stream(stream)), "moe_route_topk_noalloc")


def moe_pack_experts(src, dst, n, d, f, stream=None):
    """Binding of moe_pack_experts: n experts of shape (d, f), canonical
    packed bytes in `src` -> device block layout in `dst`.  Both are uint8
    tensors on the GPU or in page-locked host memory, B_x * n bytes each.
    Asynchronous on `stream`."""
    L = _abi.load()
    check(L.moe_pack_experts(_ptr(src), _ptr(dst), int(n), int(d), int(f), _stream(stream)), "moe_pack_experts")


class KVWindow:
    """Binding of the KV-streaming window (moe_kv_*): per layer the first
    resident_cells cells in VRAM, the rest in `host_cells` (a page-locked
    uint8 tensor or array of n_layers * (n_cells - resident_cells) *
    cell_bytes bytes that must outlive the window)."""

    def __init__(self, n_layers, n_cells, resident_cells, cell_bytes, block_cells, host_cells):
        self._lib = _abi.load()
        self._keep = host_cells
        desc = MoeKvDesc(n_layers=n_layers, cell_bytes=cell_bytes, n_cells=n_cells, resident_cells=resident_cells,
                         block_cells=block_cells, host_cells=_ptr(host_cells))
        kv = ctypes.c_void_p()
        check(self._lib.moe_kv_create(ctypes.byref(desc), ctypes.byref(kv)), "moe_kv_create")
        self.kv = kv
        self.n_layers, self.n_cells, self.resident_cells = n_layers, n_cells, resident_cells
        self.cell_bytes, self.block_cells = cell_bytes, block_cells

    def moe_kv_write(self, layer, first_cell, src, stream=None):
        """Cells [first_cell, first_cell + len(src)) of `layer` from src [n, cell_bytes] uint8 (device or pinned)."""
        check(self._lib.moe_kv_write(self.kv, int(layer), int(first_cell), int(src.shape[0]), _ptr(src),
                                     _stream(stream)), "moe_kv_write")

    def moe_kv_read_blocks(self, layer, block_ids, dst, stream=None):
        """dst[i] <- block block_ids[i] (device int32 ids; dst [n, block_cells * cell_bytes] uint8, device)."""
        check(self._lib.moe_kv_read_blocks(self.kv, int(layer), _ptr(block_ids), int(block_ids.shape[0]), _ptr(dst),
                                           _stream(stream)), "moe_kv_read_blocks")

    def moe_kv_stats(self):
        """(block reads, block reads served from VRAM) since create; synchronises."""
        r, h = ctypes.c_int64(), ctypes.c_int64()
        check(self._lib.moe_kv_stats(self.kv, ctypes.byref(r), ctypes.byref(h)), "moe_kv_stats")
        return int(r.value), int(h.value)

    def moe_kv_destroy(self):
        if self.kv is not None and self.kv.value:
            self._lib.moe_kv_destroy(self.kv)
        self.kv = None

    close = moe_kv_destroy

    def __del__(self):
        try:
            self.moe_kv_destroy()
        except Exception:
            pass
