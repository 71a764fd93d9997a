"""Pins of the multi-layer stack driver (routing + cache over a call stream)."""

import numpy as np

from moe_inputs import Synth
from moe_inputs.configs import Workload
from oracle.stack import StackOracle
from oracle.routing import route
from oracle.ffn import layer_forward
from oracle.packed import unpack_expert
from moe_inputs import bf16_bits_to_f64


def _small_stack(zipf=1.1, C=12):
    wl = Workload(90, "small-stack", d=64, f=64, n_experts=16, top_k=3, n_layers=4, tokens=3,
                  calls=40, capacity=C, preload_all=False, zipf_s=zipf, warm_passes=1)
    return StackOracle(Synth(wl))


def test_stack_invariants_over_passes():
    so = _small_stack()
    wl = so.wl
    so.prepare(range(wl.calls))
    th = tm = 0
    for p in range(2):
        for b in range(wl.calls):
            call = p * wl.calls + b
            for layer in range(wl.n_layers):
                idx, w, r = so.layer_call(call, b, layer)
                # hits + misses = k per token per layer; 10+1 structure scaled down
                assert r.token_hits + r.token_misses == wl.tokens * wl.top_k
                assert np.all(r.keys // wl.n_experts == layer)
                assert np.allclose(w.sum(1), 1, atol=1e-12)
                th += r.token_hits
                tm += r.token_misses
            so.cache.check_invariants()
    assert 0 < th and 0 < tm


def test_stack_routes_equal_per_token_route():
    so = _small_stack()
    wl = so.wl
    so.prepare(range(3))
    for layer in range(wl.n_layers):
        _, wr, b = so.s.router(layer)
        for bt in range(3):
            x = bf16_bits_to_f64(so.x_bits[(bt, layer)])
            idx, w, _ = route(x, wr, b, wl.top_k)
            i2, w2 = so.routes[(bt, layer)]
            assert np.array_equal(idx, i2)
            assert np.allclose(w, w2, rtol=0, atol=1e-15)


def test_zipf_bias_raises_hit_rate():
    rates = []
    for zipf in (0.0, 2.0):
        so = _small_stack(zipf=zipf, C=20)
        wl = so.wl
        so.prepare(range(wl.calls))
        h = n = 0
        for p in range(2):
            for b in range(wl.calls):
                for layer in range(wl.n_layers):
                    _, _, r = so.layer_call(p * wl.calls + b, b, layer)
                    if p == 1:
                        h += r.token_hits
                        n += r.token_hits + r.token_misses
        rates.append(h / n)
    assert rates[1] > rates[0]


def test_ffn_uses_pool_aliasing():
    wl = Workload(91, "alias", d=64, f=64, n_experts=8, top_k=2, n_layers=2, tokens=2, calls=2,
                  capacity=8, preload_all=False)
    so = StackOracle(Synth(wl), pool_entries=5)
    so.prepare(range(2))
    idx, w = so.routes[(1, 1)]
    e = int(idx[0, 0])
    assert so.pool_index(so.key(1, e)) == (8 + e) % 5
    y = so.ffn(1, 1)
    x = bf16_bits_to_f64(so.x_bits[(1, 1)])
    W = lambda ee: unpack_expert(so.s.expert_packed((8 + ee) % 5), wl.d, wl.f)
    want = layer_forward(x, idx, w, W, unpack_expert(so.s.shared_packed(1), wl.d, wl.f))
    assert np.allclose(y, want, rtol=1e-13, atol=1e-14)
