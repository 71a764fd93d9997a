"""Oracle of the KV-streaming window (test infrastructure only: imported by
tests/, the smoke check and bench.py's CPU baseline, never by the library).

What the window computes, from the page "单卡5090跑125B 大模型": §2.1 (the
engine keeps 32,768 of each QSA layer's 131,072 KV cells in VRAM and the
rest of the K/V, 1.55 GiB, in page-locked host memory), §2.2 (the resident
cells are the first 32,768 of the layer; the rest is streamed from host
memory) and §7.2 (the engine counts the share of block reads served from
VRAM, about 98.8% there):

  * a layer's cells 0 .. n-1 are split at R = resident cells: cell c < R is
    held in VRAM, cell c >= R in host memory at position c - R;
  * a block read of block b returns cells [b*bc, (b+1)*bc) in order;
  * a block read hits VRAM when all its cells are below R (R is a multiple
    of bc, so a block is wholly on one side).

Plain numpy indexing, one block at a time.
"""

import numpy as np


def split_layer(cells, resident):
    """cells [n, cell_bytes] -> (window [R, cell_bytes], host [n - R, cell_bytes])."""
    return cells[:resident].copy(), cells[resident:].copy()


def read_blocks(window, host, resident, block_cells, block_ids):
    """Block reads of one layer: [len(block_ids), block_cells * cell_bytes] uint8."""
    cell_bytes = window.shape[1] if window.shape[0] else host.shape[1]
    out = np.empty((len(block_ids), block_cells * cell_bytes), dtype=np.uint8)
    for i, b in enumerate(block_ids):
        rows = []
        for c in range(int(b) * block_cells, (int(b) + 1) * block_cells):
            rows.append(window[c] if c < resident else host[c - resident])
        out[i] = np.concatenate(rows)
    return out


def block_hits(block_ids, resident, block_cells):
    """(block reads, block reads that hit VRAM)."""
    ids = np.asarray(block_ids, dtype=np.int64)
    return int(ids.size), int(np.count_nonzero((ids + 1) * block_cells <= resident))


def host_bytes(n_layers, n_cells, resident, cell_bytes):
    """Bytes of the host (pinned) part of the store over n_layers layers."""
    return n_layers * (n_cells - resident) * cell_bytes
