"""GPU parity of the KV-streaming window against its oracle: block reads
bit-exact, read and hit counters exact (tiny layers, the split inside a
write, both degenerate windows, an id out of range, and sampled blocks of a
full-size 131,072-cell layer)."""

import numpy as np
import pytest
import torch

from moe_inputs.kv import KV_BLOCK_CELLS, KV_CELL_BYTES, KV_CONTEXT_CELLS, KV_RESIDENT_CELLS, kv_block_ids, kv_cells
from oracle import kv as okv

pytestmark = pytest.mark.gpu


def _window(n_layers, n, resident, cb, bc):
    from expert_cached_decode_gb300.layer import KVWindow
    host = torch.zeros(max(1, n_layers * (n - resident) * cb), dtype=torch.uint8, pin_memory=True)
    return KVWindow(n_layers, n, resident, cb, bc, host if resident < n else None), host


def _read(kv, layer, ids, bc, cb):
    d_ids = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).cuda()
    dst = torch.zeros((len(ids), bc * cb), dtype=torch.uint8, device="cuda")
    kv.moe_kv_read_blocks(layer, d_ids, dst)
    torch.cuda.synchronize()
    return dst.cpu().numpy()


@pytest.mark.parametrize("n,resident,bc", [(512, 192, 32), (512, 0, 32), (512, 512, 32), (96, 32, 16)])
def test_block_reads_match_the_oracle(n, resident, bc):
    cb, L = KV_CELL_BYTES, 2
    kv, host = _window(L, n, resident, cb, bc)
    try:
        cells = [kv_cells(5, l, n, cb) for l in range(L)]
        for l in range(L):
            kv.moe_kv_write(l, 0, torch.from_numpy(cells[l]).cuda())
        torch.cuda.synchronize()
        reads = hits = 0
        for l in range(L):
            ids = kv_block_ids(5, l, n // bc, 3 * (n // bc) + 7)
            win, hst = okv.split_layer(cells[l], resident)
            got = _read(kv, l, ids, bc, cb)
            assert np.array_equal(got, okv.read_blocks(win, hst, resident, bc, ids)), f"layer {l}"
            r, h = okv.block_hits(ids, resident, bc)
            reads, hits = reads + r, hits + h
        assert kv.moe_kv_stats() == (reads, hits)
        # the host buffer holds exactly the cells beyond the window, layer after layer
        if resident < n:
            hv = host.numpy().reshape(L, n - resident, cb)
            for l in range(L):
                assert np.array_equal(hv[l], cells[l][resident:])
    finally:
        kv.close()


def test_a_write_across_the_split_updates_both_sides():
    n, resident, bc, cb = 256, 96, 16, 64
    kv, _ = _window(1, n, resident, cb, bc)
    try:
        cells = kv_cells(6, 0, n, cb)
        kv.moe_kv_write(0, 0, torch.from_numpy(cells).cuda())
        new = kv_cells(7, 0, 20, cb)
        kv.moe_kv_write(0, resident - 7, torch.from_numpy(new).cuda())   # cells 89 .. 108
        cells[resident - 7:resident + 13] = new
        ids = np.arange(n // bc, dtype=np.int32)
        win, hst = okv.split_layer(cells, resident)
        assert np.array_equal(_read(kv, 0, ids, bc, cb), okv.read_blocks(win, hst, resident, bc, ids))
    finally:
        kv.close()


def test_an_id_out_of_range_is_reported_and_reads_nothing():
    from expert_cached_decode_gb300 import MoeError
    n, resident, bc, cb = 128, 64, 16, 32
    kv, _ = _window(1, n, resident, cb, bc)
    try:
        cells = kv_cells(8, 0, n, cb)
        kv.moe_kv_write(0, 0, torch.from_numpy(cells).cuda())
        ids = np.array([1, n // bc, 5, -1, 2], dtype=np.int32)
        got = _read(kv, 0, ids, bc, cb)
        win, hst = okv.split_layer(cells, resident)
        for i in (0, 2, 4):
            assert np.array_equal(got[i], okv.read_blocks(win, hst, resident, bc, ids[i:i + 1])[0])
        assert not got[1].any() and not got[3].any()
        with pytest.raises(MoeError) as ei:
            kv.moe_kv_stats()
        assert ei.value.status == -1
        assert kv.moe_kv_stats() == (3, 2)   # reported once; the valid reads counted
    finally:
        kv.close()


def test_full_size_layer_sampled_blocks():
    n, resident, bc, cb = KV_CONTEXT_CELLS, KV_RESIDENT_CELLS, KV_BLOCK_CELLS, KV_CELL_BYTES
    kv, _ = _window(1, n, resident, cb, bc)
    try:
        cells = kv_cells(9, 0, n, cb)
        kv.moe_kv_write(0, 0, torch.from_numpy(cells).cuda())
        nb = n // bc
        ids = np.arange(nb, dtype=np.int32)   # the bench's dense read
        got = _read(kv, 0, ids, bc, cb)
        win, hst = okv.split_layer(cells, resident)
        sample = np.concatenate([np.arange(0, nb, 97), [resident // bc - 1, resident // bc, nb - 1]])
        assert np.array_equal(got[sample], okv.read_blocks(win, hst, resident, bc, ids[sample]))
        assert np.array_equal(got.reshape(n, cb), cells)   # and every block, as the logical array
        assert kv.moe_kv_stats() == (nb, resident // bc)
    finally:
        kv.close()
