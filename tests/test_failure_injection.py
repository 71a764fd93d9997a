"""Host-side failure injection (no GPU fault): the issue of a miss copy fails
in the host-copy miss mode.  moe_forward must return MOE_ERR_CUDA with the
cache state (owners, stamps, counters) unchanged, and the same layer-call
must then succeed and leave exactly the state of a layer that never failed."""

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
