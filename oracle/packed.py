"""Canonical packed expert -> fp64 weights.

Format (the workload definition's; the pages only say the experts are 3-bit
class block-quantised, P1 §先看结果 "IQ3_XXS", and ~1.7 MB each,
P1 §如何做到：三层存储):
  sections in order: Wg codes [f][d/32][12 B], Wu codes [f][d/32][12 B],
  Wd codes [d][f/32][12 B], Wg scales [f][d/32] fp16, Wu scales, Wd scales.
  In a 12-byte group, weight i (0..31 along the input dimension) is the 3-bit
  field u at bits [3i, 3i+3) of the 96-bit little-endian integer; q = u - 4.
  The dequantised weight is W = q * s exactly (fp64), s the group's fp16 scale.

Pins: a hand-written golden group (tests/golden/packed_group.txt) and an
independent pure-Python bit packer on random codes.
"""

import numpy as np

GROUP = 32


def _sections(d, f):
    gq = f * (d // GROUP) * 12
    dq = d * (f // GROUP) * 12
    gs = f * (d // GROUP) * 2
    ds = d * (f // GROUP) * 2
    o = np.cumsum([0, gq, gq, dq, gs, gs, ds])
    return o


def unpack_codes(group_bytes):
    """[..., 12] uint8 groups -> [..., 32] int codes q in [-4, 3].

    The 96 bits are laid out least-significant first (byte 0 bit 0 is bit 0);
    field i is bits 3i, 3i+1, 3i+2 with bit 3i the least significant.
    """
    g = np.asarray(group_bytes, dtype=np.uint8)
    bits = np.unpackbits(g, axis=-1, bitorder="little")          # [..., 96]
    bits = bits.reshape(g.shape[:-1] + (32, 3)).astype(np.int64)
    u = bits[..., 0] + 2 * bits[..., 1] + 4 * bits[..., 2]
    return u - 4


def _matrix(codes_bytes, scale_bytes, rows, cols):
    q = unpack_codes(np.frombuffer(codes_bytes, dtype=np.uint8).reshape(rows, cols // GROUP, 12))
    s = np.frombuffer(scale_bytes, dtype=np.float16).reshape(rows, cols // GROUP).astype(np.float64)
    return (q.astype(np.float64) * s[:, :, None]).reshape(rows, cols)


def unpack_expert(packed, d, f):
    """Canonical packed expert bytes -> (Wg [f,d], Wu [f,d], Wd [d,f]) in fp64."""
    b = np.asarray(packed, dtype=np.uint8).tobytes()
    o = _sections(d, f)
    assert len(b) == o[-1], "packed expert has the wrong size"
    wg = _matrix(b[o[0]:o[1]], b[o[3]:o[4]], f, d)
    wu = _matrix(b[o[1]:o[2]], b[o[4]:o[5]], f, d)
    wd = _matrix(b[o[2]:o[3]], b[o[5]:o[6]], d, f)
    return wg, wu, wd
