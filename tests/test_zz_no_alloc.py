"""The allocation-free router entry point (moe_route_topk_noalloc) against
the context-based one (moe_route_topk), through the C ABI.

moe_route_topk_noalloc serves callers that cannot call cudaMalloc (their
device memory is reserved up front by their own allocator, or an allocation's
possible device-wide synchronisation is not acceptable on their path).  Its
scratch is a fixed array inside the library, shared by every call, so this
file runs two calls in a row and checks that the second does not see the
first one's leftovers.  It is collected last so that a run stopping at the
first failure has already run every other test.
"""

import numpy as np
import pytest
import torch

from moe_inputs import synth, bf16_bits_to_f64
from oracle.routing import route

pytestmark = pytest.mark.gpu


def _setup(cfg):
    from expert_cached_decode_gb300.layer import MoELayer
    s = synth(cfg)
    wl = s.wl
    wr, _, b = s.router(0)
    shared = np.stack([s.shared_packed(0)])
    pool = torch.from_numpy(np.stack([s.expert_packed(e) for e in range(min(wl.keys, 4))])).pin_memory()
    layer = MoELayer(wl.d, wl.f, wl.n_experts, wl.top_k, 1, wr.reshape(1, wl.n_experts, wl.d), b.reshape(1, -1),
                     shared, pool, host_pool_entries=pool.shape[0])
    layer._pool = pool
    wr_dev = torch.from_numpy(wr.view(np.int16)).view(torch.bfloat16).cuda()
    b_dev = torch.from_numpy(b).cuda()
    return s, layer, wr_dev, b_dev


@pytest.mark.parametrize("cfg,T1,T2", [(1, 4, 16), (2, 1, 5)])
def test_noalloc_route_matches_context_route(cfg, T1, T2):
    from expert_cached_decode_gb300.layer import moe_route_topk_noalloc
    s, layer, wr_dev, b_dev = _setup(cfg)
    k = s.wl.top_k
    for call, T in enumerate((T1, T2)):
        xb = s.tokens_many(0, [900 + call], T=T)[0]
        x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
        idx_ref = torch.empty((T, k), dtype=torch.int32, device="cuda")
        w_ref = torch.empty((T, k), dtype=torch.float32, device="cuda")
        layer.moe_route_topk(0, x, idx_ref, w_ref)
        idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        w = torch.full((T, k), -1.0, dtype=torch.float32, device="cuda")
        moe_route_topk_noalloc(x, wr_dev, b_dev, k, idx, w)
        torch.cuda.synchronize()
        assert torch.equal(idx, idx_ref), f"call {call}"
        assert (w - w_ref).abs().max().item() <= 1e-5, f"call {call}"
        # and against the fp64 oracle, which shares no code with either path
        _, wr64, b64 = s.router(0)
        oi, ow, _ = route(bf16_bits_to_f64(xb), wr64, b64, k)
        assert np.array_equal(idx.cpu().numpy(), oi), f"call {call}"
        assert np.abs(w.cpu().numpy() - ow).max() <= 1e-5, f"call {call}"
    layer.close()


def test_noalloc_route_allocates_nothing():
    # After a first call (which may load the library's module and with it
    # the fixed scratch array), further calls change neither the device's
    # free memory nor torch's allocation count.
    from expert_cached_decode_gb300.layer import moe_route_topk_noalloc
    s = synth(2)
    wl = s.wl
    wr, _, b = s.router(0)
    wr_dev = torch.from_numpy(wr.view(np.int16)).view(torch.bfloat16).cuda()
    b_dev = torch.from_numpy(b).cuda()
    xb = s.tokens_many(0, [57], T=4)[0]
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    idx = torch.empty((4, wl.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((4, wl.top_k), dtype=torch.float32, device="cuda")
    moe_route_topk_noalloc(x, wr_dev, b_dev, wl.top_k, idx, w)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    n0 = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    for _ in range(3):
        moe_route_topk_noalloc(x, wr_dev, b_dev, wl.top_k, idx, w)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0
    assert torch.cuda.memory_stats().get("allocation.all.allocated", 0) == n0


def test_noalloc_route_without_bias_and_size_limits():
    from expert_cached_decode_gb300.layer import moe_route_topk_noalloc
    from expert_cached_decode_gb300._abi import MoeError
    s, layer, wr_dev, b_dev = _setup(2)
    k = s.wl.top_k
    xb = s.tokens_many(0, [31], T=3)[0]
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).cuda()
    idx0 = torch.empty((3, k), dtype=torch.int32, device="cuda")
    w0 = torch.empty((3, k), dtype=torch.float32, device="cuda")
    moe_route_topk_noalloc(x, wr_dev, None, k, idx0, w0)          # zero bias (cfg 2 has none)
    idx1 = torch.empty_like(idx0)
    w1 = torch.empty_like(w0)
    moe_route_topk_noalloc(x, wr_dev, b_dev, k, idx1, w1)
    torch.cuda.synchronize()
    assert torch.equal(idx0, idx1) and torch.equal(w0, w1)
    big = torch.zeros((17, s.wl.d), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(MoeError, match="static scratch"):
        moe_route_topk_noalloc(big, wr_dev, b_dev, k, torch.empty((17, k), dtype=torch.int32, device="cuda"),
                               torch.empty((17, k), dtype=torch.float32, device="cuda"))
    layer.close()
