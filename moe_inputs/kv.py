"""Seeded inputs of the KV-streaming window (no window arithmetic here).

The pages size the window and the cell but not the cells' contents or which
blocks a step reads, so both are drawn:
  * cells: uniformly random bytes (an int8 K/V cell with its scales is
    opaque to the window: it only moves bytes);
  * block reads of one step: every block of the context once (a dense
    attention read), or a seeded list of block ids (with repeats) for the
    parity tests.

Sizes from the pages (page "单卡5090跑125B 大模型", §2.1-§2.2): 1,056 bytes
per int8 cell, 131,072 cells per QSA layer, the first 32,768 of them in VRAM.
The block size is this build's choice (the pages read KV "block by block"
without giving one).
"""

import numpy as np

KV_CELL_BYTES = 1056        # int8 K/V cell (q4_0 would be 576)
KV_CONTEXT_CELLS = 131072   # cells per QSA layer
KV_RESIDENT_CELLS = 32768   # the first cells of a layer kept in VRAM
KV_BLOCK_CELLS = 32         # cells per block read (a reading: the pages give none)

KIND_KV_CELLS = 21
KIND_KV_BLOCKS = 22


def _rng(seed, *key):
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(seed, spawn_key=tuple(int(k) for k in key))))


def kv_cells(seed, layer, n_cells, cell_bytes=KV_CELL_BYTES):
    """Cells 0 .. n_cells-1 of one layer, [n_cells, cell_bytes] uint8."""
    return _rng(seed, KIND_KV_CELLS, layer).integers(0, 256, size=(n_cells, cell_bytes), dtype=np.uint8)


def kv_block_ids(seed, step, n_blocks_total, n):
    """n block ids drawn uniformly from [0, n_blocks_total) (repeats allowed), int32."""
    return _rng(seed, KIND_KV_BLOCKS, step).integers(0, n_blocks_total, size=n, dtype=np.int32)
