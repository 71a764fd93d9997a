"""Shared set-up of the GPU parity tests: build a library context from the
seeded inputs and compare its outputs with the CPU oracle."""

import numpy as np
import torch

from moe_inputs import Synth, bf16_bits_to_f64
from oracle.packed import unpack_expert
from oracle.ffn import layer_forward

TOL = 2e-3          # max|y - y*| <= TOL * rms(y*), per call tensor
W_TOL = 1e-5        # routing weights


def make_pool(s: Synth, entries):
    pool = torch.empty((entries, s.B), dtype=torch.uint8, pin_memory=True)
    view = pool.numpy()
    for p in range(entries):
        s.expert_packed(p, out=view[p])
    return pool


def make_layer(s: Synth, pool_entries=None, layers=None, pool_layout=0):
    """pool_layout 1: the canonical pool is re-laid out on the GPU
    (moe_pack_experts) into a second pinned buffer that the layer uses."""
    from expert_cached_decode_gb300.layer import MoELayer, moe_pack_experts
    wl = s.wl
    L = wl.n_layers
    P = wl.keys if pool_entries is None else pool_entries
    wr = np.stack([s.router(l)[0] for l in range(L)])
    b = np.stack([s.router(l)[2] for l in range(L)])
    shared = np.stack([s.shared_packed(l) for l in range(L)])
    pool = make_pool(s, P)
    if pool_layout == 1:
        packed = torch.empty_like(pool).pin_memory()
        moe_pack_experts(pool, packed, P, wl.d, wl.f)
        torch.cuda.synchronize()
        pool = packed
    layer = MoELayer(wl.d, wl.f, wl.n_experts, wl.top_k, L, wr, b, shared, pool,
                     host_pool_entries=0 if P == wl.keys else P, host_pool_layout=pool_layout)
    layer._pool = pool
    layer._shared_np = shared
    return layer


def to_device_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


class ExpertMemo:
    """fp64 expert matrices, unpacked once."""

    def __init__(self, s: Synth, P):
        self.s, self.P, self.memo = s, P, {}

    def routed(self, layer, e):
        p = (layer * self.s.wl.n_experts + e) % self.P
        if p not in self.memo:
            self.memo[p] = unpack_expert(self.s.expert_packed(p), self.s.wl.d, self.s.wl.f)
        return self.memo[p]

    def shared(self, layer):
        key = ("shared", layer)
        if key not in self.memo:
            self.memo[key] = unpack_expert(self.s.shared_packed(layer), self.s.wl.d, self.s.wl.f)
        return self.memo[key]


def oracle_y(memo: ExpertMemo, layer, x_bits, idx, w):
    x64 = bf16_bits_to_f64(x_bits)
    return layer_forward(x64, idx, w, lambda e: memo.routed(layer, e), memo.shared(layer))


def assert_close_rms(got, want, tol=TOL, what="y"):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - want).max()
    rms = np.sqrt((want ** 2).mean())
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert err <= tol * rms, f"{what}: max|err| {err:.3e} > {tol} * rms {rms:.3e}"
    return err / rms
