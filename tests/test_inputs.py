"""Pins of the seeded input generator (rounding, value ranges, conditioning)."""

import numpy as np
import pytest
import torch

from moe_inputs import (WORKLOADS, MARGIN_DELTA, synth, bf16_bits_from_f64, bf16_bits_to_f64,
                        fp16_from_f64, expert_nbytes, expert_sections)
from moe_inputs.configs import Workload


def test_bf16_rounding_matches_torch_on_fp32_values():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(200_000) * np.exp(rng.uniform(-20, 20, 200_000))).astype(np.float32)
    ours = bf16_bits_from_f64(x.astype(np.float64))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_rounding_ties_to_even():
    # 1 + 2^-8 lies halfway between 1 and 1 + 2^-7: ties go to the even mantissa (1.0)
    # 1 + 3*2^-8 lies halfway between 1 + 2^-7 and 1 + 2^-6: goes to 1 + 2^-6
    x = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 1 + 2.0 ** -8 + 2.0 ** -40])
    got = bf16_bits_to_f64(bf16_bits_from_f64(x))
    assert got.tolist() == [1.0, 1 + 2.0 ** -6, -1.0, 1 + 2.0 ** -7]


def test_fp16_rounding_matches_numpy_and_torch():
    rng = np.random.default_rng(2)
    x = rng.uniform(0.004, 0.021, 100_000).astype(np.float32)
    ours = fp16_from_f64(x.astype(np.float64))
    assert np.array_equal(ours.view(np.uint16), x.astype(np.float16).view(np.uint16))
    tref = torch.from_numpy(x).to(torch.float16).numpy()
    assert np.array_equal(ours.view(np.uint16), tref.view(np.uint16))
    # tie: 1 + 2^-11 is halfway between 1 and 1 + 2^-10 -> 1.0
    assert float(fp16_from_f64(np.array([1 + 2.0 ** -11]))[0]) == 1.0


def test_workloads_match_the_pages_structure():
    # 512 routed experts, top-10 (+1 shared) per token per layer; 48 layers;
    # 24,576 (layer, expert) identities; 8,445 cache slots on one RTX 4090
    # (page "一张 RTX 4090 跑千亿模型", §先看结果 and §如何做到：三层存储;
    #  page "从一张到四张 RTX 4090", §先看结果: 48 layers split 4 x 12).
    for c in (2, 3, 4, 5):
        w = WORKLOADS[c]
        assert (w.n_experts, w.top_k, w.d, w.f) == (512, 10, 2048, 768)
    for c in (3, 4):
        assert WORKLOADS[c].n_layers * WORKLOADS[c].n_experts == 24_576
        assert WORKLOADS[c].capacity == 8_445
    # 12,288-token prefill chunk is the single-GPU sweet spot (page 1, §加个草稿层)
    assert WORKLOADS[5].tokens == 12_288
    assert 240 == 12_288 * 10 // 512


def test_expert_size_is_2064384_bytes():
    assert expert_nbytes(2048, 768) == 2_064_384
    assert expert_nbytes(256, 128) == 43_008
    sec = expert_sections(2048, 768)
    assert sec["wg_q"] == (0, 589_824) and sec["wd_s"][0] + sec["wd_s"][1] == 2_064_384


def test_expert_draw_ranges_and_uniform_codes():
    s = synth(1)
    wl = s.wl
    p = s.expert_packed(3)
    assert p.dtype == np.uint8 and p.size == expert_nbytes(wl.d, wl.f)
    n = 3 * wl.d * wl.f
    codes = np.unpackbits(p[: n * 3 // 8]).reshape(-1)
    # uniform random bits <=> uniform 3-bit codes
    assert abs(codes.mean() - 0.5) < 0.01
    sc = p[n * 3 // 8:].view(np.float16).astype(np.float64)
    assert sc.min() >= 0.005 - 1e-5 and sc.max() <= 0.02 + 1e-5
    assert abs(sc.mean() - 0.0125) < 2e-4
    assert not np.array_equal(s.expert_packed(4), p)
    assert np.array_equal(s.expert_packed(3), p)      # reproducible, order-free


def test_router_draws():
    s = synth(2)
    bits, w64, b = s.router(0)
    assert bits.shape == (512, 2048)
    assert abs(w64.std() - 0.02) < 2e-4
    assert np.all(b == 0)
    s3 = synth(3)
    b3 = s3.router_bias(5)
    ranks = np.rint(np.exp(-b3.astype(np.float64) / (s3.bias_lambda * 1.1))).astype(int)
    assert sorted(ranks.tolist()) == list(range(1, 513))


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_token_margin_conditioning(cfg):
    s = synth(cfg)
    wl = s.wl
    stats = {}
    xs = s.tokens_many(0, list(range(40)), T=wl.tokens if cfg != 2 else 4, stats=stats)
    x64 = bf16_bits_to_f64(xs.reshape(-1, wl.d))
    _, wr64, b = s.router(0)
    l = x64 @ wr64.T + b.astype(np.float64)
    srt = np.sort(l, axis=1)[:, ::-1]
    gap = srt[:, wl.top_k - 1] - srt[:, wl.top_k]
    assert np.all(gap >= MARGIN_DELTA)
    assert abs(x64.std() - 1.0) < 0.02
    assert stats["tokens"] == x64.shape[0]


def test_margin_screen_agrees_with_fp64_on_large_batches():
    wl = Workload(99, "t", d=128, f=64, n_experts=64, top_k=4, n_layers=1, tokens=200, calls=1,
                  capacity=64, preload_all=True)
    from moe_inputs import Synth
    s = Synth(wl)
    xs = s._draw_x(np.random.default_rng(5), 4000)
    _, wr64, b = s.router(0)
    fast = s._small_gap(xs, wr64, b)
    exact = s._small_gap(xs, wr64, b, exact=True)
    assert np.array_equal(fast, exact)


def test_token_draws_are_prefix_consistent():
    # the verify-width sweep slices the widest draw: the first T rows of a
    # T=7 draw equal the T-token draw (margin redraws are per token)
    from moe_inputs import Synth, WORKLOADS, BIAS_LAMBDA
    s = Synth(WORKLOADS[3], bias_lambda=BIAS_LAMBDA)
    wide = s.tokens_many(2, [0, 5, 17], T=7)
    for T in (1, 4):
        assert np.array_equal(wide[:, :T], s.tokens_many(2, [0, 5, 17], T=T))
