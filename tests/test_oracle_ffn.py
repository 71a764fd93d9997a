"""Pins of the oracle expert FFN and combine."""

import math

import numpy as np

from moe_inputs import synth, bf16_bits_to_f64
from oracle.packed import unpack_expert
from oracle.ffn import silu, expert_forward, layer_forward
from oracle.routing import route


def test_silu_closed_forms():
    assert silu(0.0) == 0.0
    assert abs(silu(1.0) - 1.0 / (1.0 + math.exp(-1.0))) < 1e-16
    assert abs(silu(40.0) - 40.0) < 1e-12
    assert abs(silu(-40.0)) < 1e-15
    assert silu(-1000.0) == 0.0                      # no overflow to nan
    z = np.linspace(-5, 5, 101)
    assert np.allclose(silu(z) - silu(-z), z, atol=1e-14)   # silu(z) - silu(-z) = z


def _codes_and_scales(packed, d, f):
    """Group-wise view straight from the bytes (independent of unpack_expert)."""
    b = packed.tobytes()
    n = 3 * d * f
    ints = []
    off = 0
    for rows, cols in ((f, d), (f, d), (d, f)):
        ng = rows * cols // 32
        grp = []
        for gi in range(ng):
            v = int.from_bytes(b[off + 12 * gi: off + 12 * gi + 12], "little")
            grp.append([((v >> (3 * i)) & 7) - 4 for i in range(32)])
        ints.append((rows, cols, grp))
        off += ng * 12
    sc = np.frombuffer(b[n * 3 // 8:], dtype=np.float16).astype(np.float64)
    scales = []
    so = 0
    for rows, cols, _ in ints:
        ng = rows * cols // 32
        scales.append(sc[so:so + ng])
        so += ng
    return ints, scales


def _gemv_groupwise(grp, sc, rows, cols, v):
    """Loop form: out_j = sum_g s[j,g] * sum_i q[j,g,i] * v[32 g + i]."""
    gpr = cols // 32
    out = []
    for j in range(rows):
        acc = 0.0
        for g in range(gpr):
            q = grp[j * gpr + g]
            part = 0.0
            for i in range(32):
                part += q[i] * v[32 * g + i]
            acc += sc[j * gpr + g] * part
        out.append(acc)
    return np.array(out)


def test_expert_forward_equals_groupwise_loops():
    # dequant-GEMV equals a dense matmul on the dequantised weights (brute force)
    s = synth(1)
    wl = s.wl
    packed = s.expert_packed(2)
    W = unpack_expert(packed, wl.d, wl.f)
    x = bf16_bits_to_f64(s.tokens(0, 0))[:2]
    ref = expert_forward(W, x)
    ints, scales = _codes_and_scales(packed, wl.d, wl.f)
    for t in range(2):
        g = _gemv_groupwise(ints[0][2], scales[0], wl.f, wl.d, x[t])
        u = _gemv_groupwise(ints[1][2], scales[1], wl.f, wl.d, x[t])
        h = [gi / (1.0 + math.exp(-gi)) * ui for gi, ui in zip(g, u)]
        o = _gemv_groupwise(ints[2][2], scales[2], wl.d, wl.f, h)
        assert np.allclose(o, ref[t], rtol=1e-12, atol=1e-13)


def test_one_hot_input_uses_one_column():
    s = synth(1)
    wl = s.wl
    wg, wu, wd = unpack_expert(s.expert_packed(0), wl.d, wl.f)
    j = 77
    x = np.zeros((1, wl.d))
    x[0, j] = 2.0
    got = expert_forward((wg, wu, wd), x)[0]
    g, u = 2.0 * wg[:, j], 2.0 * wu[:, j]
    want = sum(wd[:, i] * (g[i] / (1 + math.exp(-g[i])) * u[i]) for i in range(wl.f))
    assert np.allclose(got, want, rtol=1e-13, atol=1e-14)


def _tiny_layer():
    s = synth(1)
    wl = s.wl
    x = bf16_bits_to_f64(s.tokens(0, 0))
    _, wr, b = s.router(0)
    idx, w, _ = route(x, wr, b, wl.top_k)
    experts = [unpack_expert(s.expert_packed(e), wl.d, wl.f) for e in range(wl.n_experts)]
    shared = unpack_expert(s.shared_packed(0), wl.d, wl.f)
    return s, wl, x, idx, w, experts, shared


def test_identical_experts_make_output_routing_free():
    s, wl, x, idx, w, experts, shared = _tiny_layer()
    same = experts[5]
    y1 = layer_forward(x, idx, w, lambda e: same, shared)
    rng = np.random.default_rng(0)
    idx2 = np.sort(np.array([rng.choice(wl.n_experts, wl.top_k, replace=False) for _ in range(x.shape[0])]), 1)
    w2 = rng.dirichlet(np.ones(wl.top_k), size=x.shape[0])
    y2 = layer_forward(x, idx2, w2, lambda e: same, shared)
    want = expert_forward(same, x) + expert_forward(shared, x)
    assert np.allclose(y1, want, rtol=1e-12, atol=1e-12)
    assert np.allclose(y2, want, rtol=1e-12, atol=1e-12)


def test_zero_routed_weights_leave_shared_expert():
    s, wl, x, idx, w, experts, shared = _tiny_layer()
    zero = tuple(np.zeros_like(m) for m in experts[0])
    y = layer_forward(x, idx, w, lambda e: zero, shared)
    assert np.array_equal(y, expert_forward(shared, x))


def test_combine_is_weighted_sum_per_token():
    s, wl, x, idx, w, experts, shared = _tiny_layer()
    y = layer_forward(x, idx, w, lambda e: experts[e], shared)
    for t in range(x.shape[0]):
        want = expert_forward(shared, x[t:t + 1])[0]
        for i in range(wl.top_k):
            want = want + w[t, i] * expert_forward(experts[idx[t, i]], x[t:t + 1])[0]
        assert np.allclose(y[t], want, rtol=1e-12, atol=1e-13)


def test_k_token_batch_equals_single_token_calls():
    # a verify batch shares one fetch of each expert and gives each token the
    # result it would get alone (page 2, §2.3)
    s, wl, x, idx, w, experts, shared = _tiny_layer()
    yb = layer_forward(x, idx, w, lambda e: experts[e], shared)
    for t in range(x.shape[0]):
        ys = layer_forward(x[t:t + 1], idx[t:t + 1], w[t:t + 1], lambda e: experts[e], shared)
        assert np.allclose(ys[0], yb[t], rtol=1e-13, atol=1e-14)
