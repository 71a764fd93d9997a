"""Pins of the oracle's unpacking of the canonical 3-bit expert format."""

import os

import numpy as np

from oracle.packed import unpack_codes, unpack_expert
from moe_inputs import expert_sections

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "packed_group.txt")


def _golden():
    out = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        name, hx, qs = (p.strip() for p in line.split("|"))
        out.append((name, bytes.fromhex(hx), [int(v) for v in qs.split(",")]))
    return out


def test_golden_groups():
    g = _golden()
    assert len(g) == 5
    for name, b, q in g:
        got = unpack_codes(np.frombuffer(b, dtype=np.uint8))
        assert got.tolist() == q, name


def _pack_group_bitwise(codes):
    """Independent packer: one integer, field i at bit 3i, little-endian bytes."""
    v = 0
    for i, q in enumerate(codes):
        u = int(q) + 4
        assert 0 <= u <= 7
        v |= u << (3 * i)
    return v.to_bytes(12, "little")


def test_random_groups_round_trip_against_bit_packer():
    rng = np.random.default_rng(7)
    q = rng.integers(-4, 4, size=(300, 32))
    packed = np.frombuffer(b"".join(_pack_group_bitwise(r) for r in q), dtype=np.uint8).reshape(300, 12)
    assert np.array_equal(unpack_codes(packed), q)


def test_unpack_expert_sections_and_scales():
    d, f = 64, 32
    sec = expert_sections(d, f)
    buf = bytearray(sec["wd_s"][0] + sec["wd_s"][1])

    def fill(name, code):
        o, n = sec[name]
        grp = _pack_group_bitwise([code] * 32)
        buf[o:o + n] = grp * (n // 12)

    fill("wg_q", 1)      # q = 1
    fill("wu_q", -2)
    fill("wd_q", 3)
    rng = np.random.default_rng(3)
    scales = {}
    for name, rows, cols in (("wg_s", f, d), ("wu_s", f, d), ("wd_s", d, f)):
        s = rng.uniform(0.005, 0.02, (rows, cols // 32)).astype(np.float16)
        o, n = sec[name]
        buf[o:o + n] = s.tobytes()
        scales[name] = s.astype(np.float64)
    wg, wu, wd = unpack_expert(np.frombuffer(bytes(buf), np.uint8), d, f)
    assert wg.shape == (f, d) and wd.shape == (d, f)
    assert np.array_equal(wg, np.repeat(scales["wg_s"], 32, axis=1) * 1.0)
    assert np.array_equal(wu, np.repeat(scales["wu_s"], 32, axis=1) * -2.0)
    assert np.array_equal(wd, np.repeat(scales["wd_s"], 32, axis=1) * 3.0)


def test_group_scale_applies_per_row_and_group():
    # row r, group g of Wg gets scale (r+1) * 2^-8 * (g+1); codes ramp
    d, f = 64, 32
    sec = expert_sections(d, f)
    buf = bytearray(sec["wd_s"][0] + sec["wd_s"][1])
    ramp = [i % 8 - 4 for i in range(32)]
    o, n = sec["wg_q"]
    buf[o:o + n] = _pack_group_bitwise(ramp) * (n // 12)
    s = np.array([[(r + 1) * (g + 1) / 256 for g in range(d // 32)] for r in range(f)], dtype=np.float16)
    o, n = sec["wg_s"]
    buf[o:o + n] = s.tobytes()
    wg, _, _ = unpack_expert(np.frombuffer(bytes(buf), np.uint8), d, f)
    for r in (0, 5, 31):
        for k in (0, 7, 33, 63):
            assert wg[r, k] == ramp[k % 32] * float(s[r, k // 32])
