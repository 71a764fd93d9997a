"""Expert selection on crafted logits, through the C ABI.

The router matrix is zero, so each layer's logits are exactly its bias row,
and the bias rows are chosen to drive the selection's branches: the largest
logits crowded into a few of the 32 lanes that hold entry e at lane e % 32
(more candidates than the threshold pass ranks, and a middle case that needs
two ranking passes), exact ties (broken towards the lower id), and plain
distinct values.  The decode kernel (fused routing), the routing kernel and
the allocation-free router must all pick the oracle's experts bit-exactly,
with weights within 1e-5 and outputs within 2e-3 * rms.
"""

import numpy as np
import pytest
import torch

from moe_inputs import synth
from oracle.routing import route

from gpu_helpers import make_pool, to_device_bf16, ExpertMemo, oracle_y, assert_close_rms, W_TOL

pytestmark = pytest.mark.gpu

E, K = 512, 10


def _bias_rows():
    rng = np.random.default_rng(7)
    ids = np.arange(E)
    lane, i = ids % 32, ids // 32
    rows = []
    # lanes 0-3 hold the 64 largest logits
    r = rng.normal(0.0, 0.5, E)
    r[lane < 4] = 10.0 + i[lane < 4] * 4 + lane[lane < 4] * 0.25
    rows.append(r)
    # lanes 0-1 hold the 32 largest logits
    r = rng.normal(0.0, 0.5, E)
    r[lane < 2] = 5.0 + i[lane < 2] * 0.5 + lane[lane < 2] * 0.125
    rows.append(r)
    # ties: a few levels, the top level shared by 14 experts
    r = np.round(rng.uniform(0.0, 2.0, E) * 2) / 2
    r[rng.choice(E, 14, replace=False)] = 3.0
    rows.append(r)
    # distinct values
    rows.append(rng.normal(0.0, 1.0, E))
    return np.stack(rows).astype(np.float32)


@pytest.fixture(scope="module")
def crafted():
    from expert_cached_decode_gb300.layer import MoELayer
    s = synth(2)
    wl = s.wl
    b = _bias_rows()
    L = b.shape[0]
    wr = np.zeros((L, E, wl.d), dtype=np.uint16)
    shared = np.stack([s.shared_packed(l) for l in range(L)])
    P = 4
    pool = make_pool(s, P)
    layer = MoELayer(wl.d, wl.f, E, K, L, wr, b, shared, pool, host_pool_entries=P)
    layer._pool = pool
    layer.moe_cache_configure(L * E, np.arange(L * E))
    yield s, layer, b, ExpertMemo(s, P)
    layer.close()


def _oracle_route(s, xb, b_row):
    wr64 = np.zeros((E, s.wl.d))
    return route(np.zeros((xb.shape[0], s.wl.d)), wr64, b_row.astype(np.float64), K)[:2]


@pytest.mark.parametrize("T", [1, 3])
@pytest.mark.parametrize("l", [0, 1, 2, 3])
def test_fused_decode_selection(crafted, l, T):
    s, layer, b, memo = crafted
    xb = s.tokens_many(0, [300 + T], T=T)[0]
    x = to_device_bf16(xb)
    y = torch.empty((T, s.wl.d), dtype=torch.float32, device="cuda")
    tr = layer.moe_forward(l, x, y, trace=True)
    idx, w = _oracle_route(s, xb, b[l])
    assert np.array_equal(tr["idx"], idx)
    assert np.abs(tr["w"] - w).max() <= W_TOL
    assert np.array_equal(tr["slot"], l * E + idx)
    assert_close_rms(y.cpu().numpy(), oracle_y(memo, l, xb, idx, w))


@pytest.mark.parametrize("l", [0, 1, 2, 3])
def test_routing_kernel_selection(crafted, l):
    from expert_cached_decode_gb300.layer import moe_route_topk_noalloc
    s, layer, b, _ = crafted
    T = 5
    xb = s.tokens_many(0, [400], T=T)[0]
    x = to_device_bf16(xb)
    idx_want, w_want = _oracle_route(s, xb, b[l])
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    layer.moe_route_topk(l, x, idx, w)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), idx_want)
    assert np.abs(w.cpu().numpy() - w_want).max() <= W_TOL
    wr_dev = torch.zeros((E, s.wl.d), dtype=torch.bfloat16, device="cuda")
    b_dev = torch.from_numpy(b[l]).cuda()
    idx.fill_(-1)
    moe_route_topk_noalloc(x, wr_dev, b_dev, K, idx, w)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), idx_want)
    assert np.abs(w.cpu().numpy() - w_want).max() <= W_TOL
