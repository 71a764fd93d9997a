"""GPU parity of the decode path (T <= 16) against the CPU oracle, through
the C ABI: routing indices and cache slots bit-exact, routing weights within
1e-5, outputs within 2e-3 * rms."""

import numpy as np
import pytest
import torch

from moe_inputs import synth, bf16_bits_to_f64, Synth
from moe_inputs.configs import Workload
from oracle.routing import route

from gpu_helpers import make_layer, to_device_bf16, ExpertMemo, oracle_y, assert_close_rms, W_TOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny():
    s = synth(1)
    layer = make_layer(s)
    layer.moe_cache_configure(s.wl.capacity, np.arange(s.wl.keys))
    yield s, layer, ExpertMemo(s, s.wl.keys)
    layer.close()


@pytest.fixture(scope="module")
def decode():
    s = synth(2)
    layer = make_layer(s)
    layer.moe_cache_configure(s.wl.capacity, np.arange(s.wl.keys))
    yield s, layer, ExpertMemo(s, s.wl.keys)
    layer.close()


def _check_call(s, layer, memo, xb, layer_idx=0):
    wl = s.wl
    T = xb.shape[0]
    x = to_device_bf16(xb)
    y = torch.empty((T, wl.d), dtype=torch.float32, device="cuda")
    tr = layer.moe_forward(layer_idx, x, y, trace=True)
    _, wr64, b = s.router(layer_idx)
    idx, w, _ = route(bf16_bits_to_f64(xb), wr64, b, wl.top_k)
    assert np.array_equal(tr["idx"], idx)
    assert np.abs(tr["w"] - w).max() <= W_TOL
    want = oracle_y(memo, layer_idx, xb, idx, w)
    rel = assert_close_rms(y.cpu().numpy(), want)
    return tr, y, rel


@pytest.mark.parametrize("T", [1, 2, 4, 7, 8, 9, 16])
def test_tiny_layer_parity(tiny, T):
    s, layer, memo = tiny
    xb = s.tokens_many(0, [100 + T], T=T)[0]
    tr, _, _ = _check_call(s, layer, memo, xb)
    # all 16 experts preloaded into slots 0..15 in key order
    assert np.array_equal(tr["slot"], tr["idx"])
    assert tr["token_hits"] == T * s.wl.top_k and tr["token_misses"] == 0


def test_tiny_config_exact_workload(tiny):
    s, layer, memo = tiny
    xb = s.tokens(0, 0)              # the tiny workload's 4 tokens
    _check_call(s, layer, memo, xb)


def test_route_topk_only(tiny):
    s, layer, memo = tiny
    wl = s.wl
    xb = s.tokens_many(0, [7], T=16)[0]
    idx = torch.empty((16, wl.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((16, wl.top_k), dtype=torch.float32, device="cuda")
    layer.moe_route_topk(0, to_device_bf16(xb), idx, w)
    torch.cuda.synchronize()
    _, wr64, b = s.router(0)
    ri, rw, _ = route(bf16_bits_to_f64(xb), wr64, b, wl.top_k)
    assert np.array_equal(idx.cpu().numpy(), ri)
    assert np.abs(w.cpu().numpy() - rw).max() <= W_TOL


def test_decode_layer_parity_full_size(decode):
    s, layer, memo = decode
    for b in (0, 1, 2, 9_999):
        xb = s.tokens(0, b)
        tr, _, _ = _check_call(s, layer, memo, xb)
        assert np.array_equal(tr["slot"], tr["idx"])     # key e preloaded into slot e


def test_decode_stamps_follow_calls(decode):
    s, layer, memo = decode
    tr, _, _ = _check_call(s, layer, memo, s.tokens(0, 5))
    owner, stamp = layer.moe_cache_export()
    assert np.array_equal(owner, np.arange(512))
    # the call's ten experts carry the latest logical clock
    assert np.all(stamp[tr["idx"][0]] == stamp.max()) and stamp.max() >= 0


@pytest.mark.parametrize("T", [5, 16])
def test_verify_batch_equals_single_calls(decode, T):
    s, layer, memo = decode
    wl = s.wl
    xb = s.tokens_many(0, [500 + T], T=T)[0]
    tr, yb, _ = _check_call(s, layer, memo, xb)
    ys = []
    for t in range(T):
        x1 = to_device_bf16(xb[t:t + 1])
        y1 = torch.empty((1, wl.d), dtype=torch.float32, device="cuda")
        layer.moe_forward(0, x1, y1)
        ys.append(y1)
    torch.cuda.synchronize()
    ys = torch.cat(ys).cpu().numpy()
    ybn = yb.cpu().numpy()
    rms = np.sqrt((ybn.astype(np.float64) ** 2).mean())
    assert np.abs(ys - ybn).max() <= 2e-3 * rms
    print(f"T={T}: batch vs singles bitwise equal: {np.array_equal(ys, ybn)}")


def test_decode_many_calls_sampled(decode):
    # consecutive calls reuse per-call scratch; check a sample of a longer run
    s, layer, memo = decode
    wl = s.wl
    before = layer.moe_cache_stats()
    xs = s.tokens_many(0, list(range(64)), T=1)
    xd = to_device_bf16(xs.reshape(64, wl.d))
    y = torch.empty((64, wl.d), dtype=torch.float32, device="cuda")
    for i in range(64):
        layer.moe_forward(0, xd[i:i + 1], y[i:i + 1])
    layer.moe_sync()
    _, wr64, b = s.router(0)
    yn = y.cpu().numpy()
    for i in (0, 17, 63):
        idx, w, _ = route(bf16_bits_to_f64(xs[i]), wr64, b, wl.top_k)
        assert_close_rms(yn[i:i + 1], oracle_y(memo, 0, xs[i], idx, w))
    st = layer.moe_cache_stats()
    assert st["token_misses"] == 0
    assert st["layer_calls"] - before["layer_calls"] == 64
    assert st["token_hits"] - before["token_hits"] == 64 * wl.top_k
    assert st["distinct_hits"] - before["distinct_hits"] == 64 * wl.top_k


@pytest.mark.parametrize("d,f", [(256, 64), (256, 192), (256, 320), (512, 128), (768, 64), (1280, 128)])
def test_shapes_slices_and_down_stages(d, f):
    # f/32 slices per expert from 2 to 10; d/32 row blocks of the down part
    # from 8 (half a stage) over 24 (a stage and a half) to 40 (two and a half
    # stages); one and two token tiles
    import dataclasses
    from moe_inputs import WORKLOADS, BIAS_LAMBDA
    wl = dataclasses.replace(WORKLOADS[1], d=d, f=f)
    s = Synth(wl, bias_lambda=BIAS_LAMBDA)
    layer = make_layer(s)
    try:
        layer.moe_cache_configure(wl.capacity, np.arange(wl.keys))
        memo = ExpertMemo(s, wl.keys)
        for T in (1, 5, 9, 16):
            xb = s.tokens_many(0, [900 + T], T=T)[0]
            _check_call(s, layer, memo, xb)
    finally:
        layer.close()


@pytest.mark.parametrize("T", [1, 5, 16])
def test_decode_is_deterministic(decode, T):
    # the same call twice gives bitwise the same y (fixed-order combine)
    s, layer, memo = decode
    xb = s.tokens_many(0, [700 + T], T=T)[0]
    x = to_device_bf16(xb)
    y1 = torch.empty((T, s.wl.d), dtype=torch.float32, device="cuda")
    y2 = torch.empty_like(y1)
    layer.moe_forward(0, x, y1)
    layer.moe_forward(0, to_device_bf16(s.tokens_many(0, [1], T=T)[0]), y2)   # another call between
    layer.moe_forward(0, x, y2)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
