"""Failure detection without a GPU fault.

* Host-side injection: the issue of a miss copy fails in the host-copy miss
  mode (moe_forward returns MOE_ERR_CUDA with the cache state unchanged, and
  the retried call leaves exactly the state of a layer that never failed);
  the host pool's registration fails at create (MOE_ERR_HOST_PIN, nothing
  left registered); a device allocation fails at create (MOE_ERR_OOM, no
  memory left allocated) or at configure (MOE_ERR_OOM, the previous cache
  unchanged and usable).
* Bounded device waits: one CTA holds back its router logits (words that
  nothing else writes), every CTA's wait for them runs out after a short
  limit, the kernel returns, moe_sync reports MOE_ERR_TIMEOUT and the context
  works again (after reconfiguring, for a cache that can miss).
"""

import dataclasses

import numpy as np
import pytest
import torch

from moe_inputs import Synth, WORKLOADS, BIAS_LAMBDA
from expert_cached_decode_gb300 import _abi
from expert_cached_decode_gb300._abi import MoeError, MOE_MISS_HOST_COPY, MOE_INJECT_MISS_COPY
from gpu_helpers import make_layer, to_device_bf16

pytestmark = pytest.mark.gpu

OVER = dict(d=256, f=128, n_experts=32, top_k=4, n_layers=6, tokens=5, capacity=40, calls=4)


def _layer(s):
    layer = make_layer(s, pool_entries=96)
    layer.moe_set_miss_mode(MOE_MISS_HOST_COPY)
    layer.moe_cache_configure(s.wl.capacity)      # empty: the first call misses on every expert
    return layer


def test_failed_miss_copy_leaves_the_cache_unchanged():
    wl = dataclasses.replace(WORKLOADS[3], **OVER)
    s = Synth(wl, bias_lambda=BIAS_LAMBDA)
    lib = _abi.load()
    x = to_device_bf16(s.tokens_many(0, [0], T=wl.tokens)[0])
    y = torch.empty((wl.tokens, wl.d), dtype=torch.float32, device="cuda")
    layer = _layer(s)
    try:
        owner0, stamp0 = layer.moe_cache_export()
        stats0 = layer.moe_cache_stats()
        assert lib.moe_debug_inject_failure(MOE_INJECT_MISS_COPY, 2) == 0
        with pytest.raises(MoeError) as ei:
            layer.moe_forward(0, x, y)
        assert ei.value.status == -3 and "injected" in str(ei.value)
        owner1, stamp1 = layer.moe_cache_export()
        assert np.array_equal(owner0, owner1) and np.array_equal(stamp0, stamp1)
        assert layer.moe_cache_stats() == stats0
        # nothing armed now: the same call succeeds
        layer.moe_forward(0, x, y)
        layer.moe_sync()
        owner2, stamp2 = layer.moe_cache_export()
        y2 = y.cpu().numpy().copy()
    finally:
        lib.moe_debug_inject_failure(0, 0)
        layer.close()
    ref = _layer(s)
    try:
        ref.moe_forward(0, x, y)
        ref.moe_sync()
        owner_r, stamp_r = ref.moe_cache_export()
        assert np.array_equal(owner2, owner_r) and np.array_equal(stamp2, stamp_r)
        assert np.array_equal(y2, y.cpu().numpy())
        assert ref.moe_cache_stats()["layer_calls"] == 1
    finally:
        ref.close()


# ---- bounded device waits that run out (no GPU fault: a flag nobody sets) --

def _resident_tiny():
    from moe_inputs import synth
    s = synth(1)
    layer = make_layer(s)
    layer.moe_cache_configure(s.wl.capacity, np.arange(s.wl.keys))
    return s, layer


def _oracle_check(s, layer, xb):
    from moe_inputs import bf16_bits_to_f64
    from oracle.routing import route
    from gpu_helpers import ExpertMemo, oracle_y, assert_close_rms
    y = torch.empty((xb.shape[0], s.wl.d), dtype=torch.float32, device="cuda")
    tr = layer.moe_forward(0, to_device_bf16(xb), y, trace=True)
    _, wr64, b = s.router(0)
    idx, w, _ = route(bf16_bits_to_f64(xb), wr64, b, s.wl.top_k)
    assert np.array_equal(tr["idx"], idx)
    assert_close_rms(y.cpu().numpy(), oracle_y(ExpertMemo(s, s.wl.keys), 0, xb, idx, w))


@pytest.mark.parametrize("T", [1, 4])
def test_router_wait_runs_out_and_the_context_recovers(T):
    # CTA 0 holds back its router logits: every CTA's wait for them runs out
    # after 20 ms, the kernel returns, moe_sync reports MOE_ERR_TIMEOUT, and
    # the next call is correct again (T = 1: the one-token selection, whose
    # CTAs hand the producer its units right after selecting)
    lib = _abi.load()
    s, layer = _resident_tiny()
    try:
        layer.moe_debug_set_wait_limit(20_000_000)
        xb = s.tokens_many(0, [3], T=T)[0]
        y = torch.empty((T, s.wl.d), dtype=torch.float32, device="cuda")
        assert lib.moe_debug_inject_failure(_abi.MOE_INJECT_HOLD_ROUTER, 1) == 0
        layer.moe_forward(0, to_device_bf16(xb), y)      # asynchronous: no error yet
        with pytest.raises(MoeError) as ei:
            layer.moe_sync()
        assert ei.value.status == -5                     # MOE_ERR_TIMEOUT
        layer.moe_sync()                                 # the error was reported once
        _oracle_check(s, layer, xb)
    finally:
        lib.moe_debug_inject_failure(0, 0)
        layer.close()


def test_router_wait_runs_out_with_a_cache_that_misses():
    # the same on the miss-capable path (CTA 0 manages the cache): after the
    # timeout the cache must be configured again, then calls are correct
    lib = _abi.load()
    wl = dataclasses.replace(WORKLOADS[3], **OVER)
    s = Synth(wl, bias_lambda=BIAS_LAMBDA)
    layer = make_layer(s, pool_entries=96)
    try:
        layer.moe_cache_configure(wl.capacity)
        layer.moe_debug_set_wait_limit(20_000_000)
        x = to_device_bf16(s.tokens_many(0, [0], T=wl.tokens)[0])
        y = torch.empty((wl.tokens, wl.d), dtype=torch.float32, device="cuda")
        assert lib.moe_debug_inject_failure(_abi.MOE_INJECT_HOLD_ROUTER, 1) == 0
        layer.moe_forward(0, x, y)
        with pytest.raises(MoeError) as ei:
            layer.moe_sync()
        assert ei.value.status == -5
        with pytest.raises(MoeError) as ei:
            layer.moe_forward(0, x, y)
        assert ei.value.status == -6                     # MOE_ERR_STATE until configured
        layer.moe_cache_configure(wl.capacity)
        layer.moe_forward(0, x, y)
        layer.moe_sync()
        y1 = y.cpu().numpy().copy()
        owner1, stamp1 = layer.moe_cache_export()
    finally:
        lib.moe_debug_inject_failure(0, 0)
        layer.close()
    ref = make_layer(s, pool_entries=96)
    try:
        ref.moe_cache_configure(wl.capacity)
        ref.moe_forward(0, x, y)
        ref.moe_sync()
        owner_r, stamp_r = ref.moe_cache_export()
        assert np.array_equal(owner1, owner_r) and np.array_equal(stamp1, stamp_r)
        assert np.array_equal(y1, y.cpu().numpy())
    finally:
        ref.close()


# ---- failed registration and allocations (host-side injection) ------------

def _desc_args(s, pool):
    wl = s.wl
    wr = np.stack([s.router(l)[0] for l in range(wl.n_layers)])
    b = np.stack([s.router(l)[2] for l in range(wl.n_layers)])
    shared = np.stack([s.shared_packed(l) for l in range(wl.n_layers)])
    return (wl.d, wl.f, wl.n_experts, wl.top_k, wl.n_layers, wr, b, shared, pool)


def test_failed_host_pool_registration():
    from expert_cached_decode_gb300.layer import MoELayer
    from moe_inputs import synth
    lib = _abi.load()
    s = synth(1)
    pool = np.stack([s.expert_packed(e) for e in range(s.wl.keys)])     # pageable: registered at create
    args = _desc_args(s, pool)
    try:
        assert lib.moe_debug_inject_failure(_abi.MOE_INJECT_HOST_REGISTER, 1) == 0
        with pytest.raises(MoeError) as ei:
            MoELayer(*args)
        assert ei.value.status == -4                     # MOE_ERR_HOST_PIN
        layer = MoELayer(*args)                          # nothing was left registered
        layer.moe_cache_configure(s.wl.capacity, np.arange(s.wl.keys))
        _oracle_check(s, layer, s.tokens(0, 0))
        layer.close()
    finally:
        lib.moe_debug_inject_failure(0, 0)


def test_failed_device_allocation_at_create_leaves_nothing():
    from expert_cached_decode_gb300.layer import MoELayer
    from moe_inputs import synth
    lib = _abi.load()
    s = synth(2)
    pool = torch.from_numpy(np.stack([s.expert_packed(e) for e in range(4)])).pin_memory()
    args = _desc_args(s, pool)
    MoELayer(*args, host_pool_entries=4).close()         # warm: module loading, first allocations
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    try:
        for nth in (1, 3, 6, 9):
            assert lib.moe_debug_inject_failure(_abi.MOE_INJECT_DEVICE_ALLOC, nth) == 0
            with pytest.raises(MoeError) as ei:
                MoELayer(*args, host_pool_entries=4)
            assert ei.value.status == -2                 # MOE_ERR_OOM
            torch.cuda.synchronize()
            assert abs(torch.cuda.mem_get_info()[0] - free0) < (2 << 20), f"allocation {nth}"
    finally:
        lib.moe_debug_inject_failure(0, 0)


def test_failed_device_allocation_at_configure_keeps_the_cache():
    lib = _abi.load()
    wl = dataclasses.replace(WORKLOADS[3], **OVER)
    s = Synth(wl, bias_lambda=BIAS_LAMBDA)
    xs = [to_device_bf16(s.tokens_many(0, [c], T=wl.tokens)[0]) for c in range(2)]
    y = torch.empty((wl.tokens, wl.d), dtype=torch.float32, device="cuda")
    layer = make_layer(s, pool_entries=96)
    try:
        layer.moe_cache_configure(wl.capacity)
        layer.moe_forward(0, xs[0], y)
        layer.moe_sync()
        owner0, stamp0 = layer.moe_cache_export()
        stats0 = layer.moe_cache_stats()
        for nth in (1, 2, 4):
            assert lib.moe_debug_inject_failure(_abi.MOE_INJECT_DEVICE_ALLOC, nth) == 0
            with pytest.raises(MoeError) as ei:
                layer.moe_cache_configure(wl.capacity + 8)
            assert ei.value.status == -2
            owner1, stamp1 = layer.moe_cache_export()
            assert np.array_equal(owner0, owner1) and np.array_equal(stamp0, stamp1)
            assert layer.moe_cache_stats() == stats0
        layer.moe_forward(0, xs[1], y)                    # the old cache goes on
        layer.moe_sync()
        y1 = y.cpu().numpy().copy()
        owner1, stamp1 = layer.moe_cache_export()
    finally:
        lib.moe_debug_inject_failure(0, 0)
        layer.close()
    ref = make_layer(s, pool_entries=96)
    try:
        ref.moe_cache_configure(wl.capacity)
        for c in range(2):
            ref.moe_forward(0, xs[c], y)
        ref.moe_sync()
        owner_r, stamp_r = ref.moe_cache_export()
        assert np.array_equal(owner1, owner_r) and np.array_equal(stamp1, stamp_r)
        assert np.array_equal(y1, y.cpu().numpy())
    finally:
        ref.close()
