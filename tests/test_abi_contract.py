"""The C ABI's argument checks and error reporting (include/moe_gb300.h):
every call below is rejected before any CUDA work, so this runs without a
GPU.  Status codes, the message of moe_last_error and the untouched output
pointer are checked."""

import ctypes

import pytest

from expert_cached_decode_gb300 import _abi

INVALID, UNIMPL = -1, -7


@pytest.fixture(scope="module")
def lib():
    import os
    from expert_cached_decode_gb300 import LIB_PATH, build_library
    if not os.path.exists(LIB_PATH):
        build_library()
    return _abi.load()


def _desc(**over):
    buf = ctypes.create_string_buffer(64)
    d = dict(d=2048, f=768, n_experts=512, top_k=10, n_layers=1, group=32,
             router_w=ctypes.addressof(buf), router_b=None, shared_q=ctypes.addressof(buf),
             host_pool=ctypes.addressof(buf), host_pool_entries=0, shared_weight=1.0)
    d.update(over)
    desc = _abi.MoeLayerDesc(**d)
    desc._keep = buf
    return desc


@pytest.mark.parametrize("over,status,words", [
    (dict(group=16), UNIMPL, "group"),
    (dict(d=100), UNIMPL, "multiple of 256"),
    (dict(f=96), UNIMPL, "multiple of 64"),
    (dict(f=2048), UNIMPL, "multiple of 64"),
    (dict(top_k=1), UNIMPL, "top_k"),
    (dict(top_k=17), UNIMPL, "top_k"),
    (dict(n_experts=2048), UNIMPL, "n_experts"),
    (dict(n_experts=10), UNIMPL, "n_experts"),
    (dict(n_layers=0), INVALID, "n_layers"),
    (dict(router_w=None), INVALID, "required"),
    (dict(shared_q=None), INVALID, "required"),
    (dict(host_pool=None), INVALID, "required"),
    (dict(host_pool_entries=-1), INVALID, "host_pool_entries"),
])
def test_create_rejects_bad_descriptors(lib, over, status, words):
    out = ctypes.c_void_p(12345)
    st = lib.moe_layer_create(ctypes.byref(_desc(**over)), ctypes.byref(out))
    assert st == status
    assert out.value is None            # *out is cleared before any check that can fail
    assert words in lib.moe_last_error().decode()


def test_create_rejects_null(lib):
    out = ctypes.c_void_p()
    assert lib.moe_layer_create(None, ctypes.byref(out)) == INVALID
    assert lib.moe_layer_create(ctypes.byref(_desc()), None) == INVALID
    assert "NULL" in lib.moe_last_error().decode()


def test_calls_on_a_null_context(lib):
    x = ctypes.create_string_buffer(4096)
    stats = _abi.MoeStats()
    assert lib.moe_cache_configure(None, 512, None, 0) == INVALID
    assert lib.moe_route_topk(None, 0, ctypes.addressof(x), 1, ctypes.addressof(x), ctypes.addressof(x), None) == INVALID
    assert lib.moe_forward(None, 0, ctypes.addressof(x), 1, ctypes.addressof(x), None, None) == INVALID
    assert lib.moe_sync(None) == INVALID
    assert lib.moe_cache_stats(None, ctypes.byref(stats), None) == INVALID
    assert lib.moe_cache_export(None, ctypes.addressof(x), ctypes.addressof(x)) == INVALID
    assert lib.moe_set_miss_mode(None, _abi.MOE_MISS_DEVICE_PULL) == INVALID
    assert "NULL" in lib.moe_last_error().decode()
    lib.moe_layer_destroy(None)         # a no-op


@pytest.mark.parametrize("T,d,E,k,misalign,words", [
    (0, 2048, 512, 10, 0, "static scratch"),
    (17, 2048, 512, 10, 0, "static scratch"),
    (1, 2048, 512, 1, 0, "top_k"),
    (1, 2048, 2048, 10, 0, "top_k"),
    (1, 100, 512, 10, 0, "multiple of 256"),
    (1, 2048, 512, 10, 8, "16-byte aligned"),
])
def test_noalloc_router_rejects_bad_arguments(lib, T, d, E, k, misalign, words):
    buf = ctypes.create_string_buffer(4096 + 32)
    base = (ctypes.addressof(buf) + 15) // 16 * 16
    st = lib.moe_route_topk_noalloc(base + misalign, base, None, T, d, E, k, base, base, None)
    assert st == INVALID
    assert words in lib.moe_last_error().decode()


def test_noalloc_router_rejects_null_pointers(lib):
    buf = ctypes.create_string_buffer(64)
    a = ctypes.addressof(buf)
    for args in ((None, a, a, a), (a, None, a, a), (a, a, None, a), (a, a, a, None)):
        x, wr, idx, w = args
        assert lib.moe_route_topk_noalloc(x, wr, None, 1, 2048, 512, 10, idx, w, None) == INVALID


def test_create_without_a_device_fails_cleanly(lib):
    # on a machine without a usable GPU the first CUDA call fails: the status
    # is MOE_ERR_CUDA, the partial context is released, *out stays NULL
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    out = ctypes.c_void_p(12345)
    st = lib.moe_layer_create(ctypes.byref(_desc()), ctypes.byref(out))
    assert st == -3
    assert out.value is None
    assert "cuda" in lib.moe_last_error().decode().lower()


def test_failure_injection_hook_arguments(lib):
    assert lib.moe_debug_inject_failure(7, 1) == INVALID
    assert lib.moe_debug_inject_failure(_abi.MOE_INJECT_MISS_COPY, 0) == INVALID
    assert "unknown kind" in lib.moe_last_error().decode()
    assert lib.moe_debug_inject_failure(_abi.MOE_INJECT_MISS_COPY, 3) == 0
    assert lib.moe_debug_inject_failure(0, 0) == 0        # disarm
