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
from oracle.ffn import layer_forward
from oracle.packed import unpack_expert

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


SWEEP = WORKLOADS[5].sweep        # 4,096 / 6,144 / 8,192 / 12,288 / 16,384 tokens


def _oracle_many(s, chunks):
    """Oracle outputs of several chunks of one layer, every expert unpacked
    once for all of them (fp64 matrices are not kept: 37.7 MB each)."""
    wl = s.wl
    xs = np.concatenate([c[0] for c in chunks])
    idx = np.concatenate([c[1] for c in chunks])
    w = np.concatenate([c[2] for c in chunks])
    shared = unpack_expert(s.shared_packed(0), wl.d, wl.f)
    y = layer_forward(bf16_bits_to_f64(xs), idx, w, lambda e: unpack_expert(s.expert_packed(e), wl.d, wl.f), shared)
    out, o = [], 0
    for c in chunks:
        out.append(y[o:o + c[0].shape[0]])
        o += c[0].shape[0]
    return out


@pytest.fixture(scope="module")
def sweep_runs(chunk):
    """Every chunk size of the sweep through the GPU, then the oracle."""
    s, layer, _ = chunk
    runs = {}
    for T in SWEEP:
        xb = s.tokens_many(0, [T], T=T)[0]
        tr, y, idx, w = _prefill(s, layer, xb)
        runs[T] = dict(xb=xb, tr=tr, y=y, idx=idx, w=w)
    want = _oracle_many(s, [(runs[T]["xb"], runs[T]["idx"], runs[T]["w"]) for T in SWEEP])
    for T, wy in zip(SWEEP, want):
        runs[T]["want"] = wy
    return runs


@pytest.mark.parametrize("T", SWEEP)
def test_chunk_prefill_full_size(sweep_runs, T):
    # every output of the chunk against the oracle (no sampling)
    r = sweep_runs[T]
    assert np.array_equal(r["tr"]["idx"], r["idx"])
    assert np.abs(r["tr"]["w"] - r["w"]).max() <= W_TOL
    assert_close_rms(r["y"], r["want"], what=f"y[{T} tokens]")
    counts = np.bincount(r["idx"].ravel(), minlength=512)
    assert counts.sum() == T * 10


def test_chunk_prefill_is_deterministic(chunk, sweep_runs):
    # the same 12,288-token chunk twice: bitwise the same outputs
    s, layer, _ = chunk
    r = sweep_runs[12288]
    _, y2, _, _ = _prefill(s, layer, r["xb"])
    assert np.array_equal(r["y"].view(np.uint32), y2.view(np.uint32))


def test_chunk_prefill_skewed_routing():
    # A steep Zipf router bias (s = 1.5, scale 1): a few experts take almost
    # every token (several 256-token tiles each) while most take none.
    wl = dataclasses.replace(WORKLOADS[5], zipf_s=1.5, tokens=4096)
    s = Synth(wl, bias_lambda=1.0)
    layer = make_layer(s)
    layer.moe_cache_configure(wl.keys, np.arange(wl.keys))
    xb = s.tokens_many(0, [7], T=4096)[0]
    tr, y, idx, w = _prefill(s, layer, xb)
    layer.close()
    counts = np.bincount(idx.ravel(), minlength=512)
    assert (counts == 0).sum() > 100 and counts.max() > 3 * 256
    assert np.array_equal(tr["idx"], idx)
    assert np.abs(tr["w"] - w).max() <= W_TOL
    assert tr["n_distinct"] == int((counts > 0).sum())
    want = layer_forward(bf16_bits_to_f64(xb), idx, w, lambda e: unpack_expert(s.expert_packed(e), wl.d, wl.f),
                         unpack_expert(s.shared_packed(0), wl.d, wl.f))
    assert_close_rms(y, want, what="y (skewed routing)")
