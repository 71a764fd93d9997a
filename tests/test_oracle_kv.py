"""Pins of the KV-streaming window oracle (no GPU).

The window is a split of one logical array of cells: block reads must give
back the logical array's cells whatever side of the split they live on, and
the hit count is the number of reads below the split.  The sizes the pages
print (tests/golden/kv_window.txt) pin the reading of the layout."""

import os

import numpy as np
import pytest

from moe_inputs.kv import (KV_BLOCK_CELLS, KV_CELL_BYTES, KV_CONTEXT_CELLS, KV_RESIDENT_CELLS, kv_block_ids,
                           kv_cells)
from oracle import kv as okv

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kv_window.txt")


def _golden():
    vals = {}
    for ln in open(GOLDEN):
        ln = ln.strip()
        if ln and not ln.startswith("#"):
            k, v = ln.split()
            vals[k] = float(v)
    return vals


def test_sizes_reproduce_the_pages_host_footprint():
    g = _golden()
    assert KV_CELL_BYTES == g["cell_bytes_int8"]
    assert KV_CONTEXT_CELLS == g["context_cells"]
    assert KV_RESIDENT_CELLS == g["resident_cells"]
    per_layer = okv.host_bytes(1, KV_CONTEXT_CELLS, KV_RESIDENT_CELLS, KV_CELL_BYTES)
    assert per_layer == 98304 * 1056
    # a whole number of QSA layers gives the printed 1.55 GiB, to its two decimals
    layers = [n for n in range(1, 49) if round(okv.host_bytes(n, KV_CONTEXT_CELLS, KV_RESIDENT_CELLS,
                                                              KV_CELL_BYTES) / 2**30, 2) == g["host_gib"]]
    assert layers == [16]
    # both printed cell sizes are multiples of 16 bytes, the window's copy unit
    assert g["cell_bytes_int8"] % 16 == 0 and g["cell_bytes_q4_0"] % 16 == 0


@pytest.mark.parametrize("n,resident,bc", [(64, 32, 8), (64, 0, 8), (64, 64, 8), (96, 48, 16), (40, 8, 8)])
def test_reading_every_block_in_order_gives_back_the_layer(n, resident, bc):
    cells = kv_cells(0, 3, n, cell_bytes=32)
    window, host = okv.split_layer(cells, resident)
    assert window.shape[0] == resident and host.shape[0] == n - resident
    ids = np.arange(n // bc, dtype=np.int32)
    out = okv.read_blocks(window, host, resident, bc, ids)
    assert np.array_equal(out.reshape(n, 32), cells)
    assert okv.block_hits(ids, resident, bc) == (n // bc, resident // bc)


def test_random_block_reads_match_the_logical_array():
    n, resident, bc, cb = 128, 48, 16, 48
    cells = kv_cells(1, 0, n, cell_bytes=cb)
    window, host = okv.split_layer(cells, resident)
    ids = kv_block_ids(1, 0, n // bc, 40)
    out = okv.read_blocks(window, host, resident, bc, ids)
    for i, b in enumerate(ids):
        assert np.array_equal(out[i], cells[b * bc:(b + 1) * bc].reshape(-1))
    reads, hits = okv.block_hits(ids, resident, bc)
    assert reads == 40
    assert hits == sum(1 for b in ids if b < resident // bc)


def test_hits_at_the_split_boundary():
    bc, resident = 8, 32
    # block 3 ends at cell 32 (the last resident one); block 4 starts at 32
    assert okv.block_hits([3], resident, bc) == (1, 1)
    assert okv.block_hits([4], resident, bc) == (1, 0)
    assert okv.block_hits([0, 4, 3, 4], resident, bc) == (4, 2)


def test_the_stated_window_hits_a_quarter_of_a_dense_read():
    ids = np.arange(KV_CONTEXT_CELLS // KV_BLOCK_CELLS)
    reads, hits = okv.block_hits(ids, KV_RESIDENT_CELLS, KV_BLOCK_CELLS)
    assert hits * 4 == reads
