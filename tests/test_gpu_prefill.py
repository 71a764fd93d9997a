"""GPU parity of the prefill path (T > 16): tensor-core router logits,
counting sort by expert and the tcgen05 grouped GEMMs with in-loader
dequant, against the CPU oracle (routing bit-exact on every token, outputs
within 2e-3 * rms)."""

import dataclasses

import numpy as np
import pytest
import torch

from moe_inputs import Synth, WORKLOADS, bf16_bits_to_f64
from oracle.routing import route

from gpu_helpers import make_layer, to_device_bf16, ExpertMemo, oracle_y, assert_close_rms, W_TOL

pytestmark = pytest.mark.gpu


def _layer(wl):
    s = Synth(wl)
    layer = make_layer(s)
    layer.moe_cache_configure(wl.keys, np.arange(wl.keys))
    return s, layer


@pytest.fixture(scope="module")
def tiny():
    wl = dataclasses.replace(WORKLOADS[1], tokens=300)
    s, layer = _layer(wl)
    yield s, layer, ExpertMemo(s, wl.keys)
    layer.close()


@pytest.fixture(scope="module")
def chunk():
    wl = WORKLOADS[5]
    s, layer = _layer(wl)
    yield s, layer, ExpertMemo(s, wl.keys)
    layer.close()


def _prefill(s, layer, xb):
    T = xb.shape[0]
    x = to_device_bf16(xb)
    y = torch.empty((T, s.wl.d), dtype=torch.float32, device="cuda")
    tr = layer.moe_forward(0, x, y, trace=True)
    _, wr64, b = s.router(0)
    idx, w, _ = route(bf16_bits_to_f64(xb), wr64, b, s.wl.top_k)
    return tr, y.cpu().numpy(), idx, w


@pytest.mark.parametrize("T", [17, 64, 257, 300])
def test_tiny_prefill_parity(tiny, T):
    s, layer, memo = tiny
    xb = s.tokens_many(0, [1000 + T], T=T)[0]
    tr, y, idx, w = _prefill(s, layer, xb)
    assert np.array_equal(tr["idx"], idx)
    assert np.abs(tr["w"] - w).max() <= W_TOL
    assert_close_rms(y, oracle_y(memo, 0, xb, idx, w))


def test_prefill_route_topk_matches_oracle(tiny):
    s, layer, memo = tiny
    wl = s.wl
    xb = s.tokens_many(0, [77], T=300)[0]
    idx = torch.empty((300, wl.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((300, wl.top_k), dtype=torch.float32, device="cuda")
    layer.moe_route_topk(0, to_device_bf16(xb), idx, w)
    torch.cuda.synchronize()
    _, wr64, b = s.router(0)
    ri, rw, _ = route(bf16_bits_to_f64(xb), wr64, b, wl.top_k)
    assert np.array_equal(idx.cpu().numpy(), ri)
    assert np.abs(w.cpu().numpy() - rw).max() <= W_TOL


def test_prefill_equals_decode_path(tiny):
    # the same 17 tokens through the prefill path and as one-token decode calls
    s, layer, memo = tiny
    wl = s.wl
    xb = s.tokens_many(0, [4242], T=17)[0]
    tr, yp, idx, w = _prefill(s, layer, xb)
    ys = []
    for t in range(17):
        y1 = torch.empty((1, wl.d), dtype=torch.float32, device="cuda")
        layer.moe_forward(0, to_device_bf16(xb[t:t + 1]), y1)
        ys.append(y1)
    yd = torch.cat(ys).cpu().numpy()
    rms = np.sqrt((yd.astype(np.float64) ** 2).mean())
    assert np.abs(yp - yd).max() <= 2e-3 * rms


@pytest.mark.parametrize("T", [4096, 12288])
def test_chunk_prefill_full_size(chunk, T):
    s, layer, memo = chunk
    xb = s.tokens_many(0, [T], T=T)[0]
    tr, y, idx, w = _prefill(s, layer, xb)
    assert np.array_equal(tr["idx"], idx)
    assert np.abs(tr["w"] - w).max() <= W_TOL
    # outputs on a sample of tokens (the oracle evaluates them one by one)
    rng = np.random.default_rng(T)
    sample = np.sort(rng.choice(T, 12, replace=False))
    sample[0], sample[-1] = 0, T - 1
    for t in sample:
        want = oracle_y(memo, 0, xb[t:t + 1], idx[t:t + 1], w[t:t + 1])
        assert_close_rms(y[t:t + 1], want, what=f"y[{t}]")
    assert np.all(np.isfinite(y))
    # every expert got ~T*k/E tokens; the counting sort covered all picks
    counts = np.bincount(idx.ravel(), minlength=512)
    assert counts.sum() == T * 10
