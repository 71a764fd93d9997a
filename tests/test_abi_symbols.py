"""The C-ABI library loads and exports every entry point include/*.h declares
(no compute calls: this runs without a GPU)."""

import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[\w\s\*]+?\b(moe_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib_path():
    from expert_cached_decode_gb300 import LIB_PATH, build_library
    if not os.path.exists(LIB_PATH):
        build_library()
    return LIB_PATH


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("moe_layer_create", "moe_cache_configure", "moe_route_topk", "moe_forward"):
        assert n in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    names = _declared()
    assert names
    for n in sorted(names):
        assert hasattr(lib, n), f"{n} not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    assert names <= exported


def test_binding_names_match_header():
    from expert_cached_decode_gb300 import ENTRY_POINTS
    assert set(ENTRY_POINTS) == _declared()


def test_null_arguments_are_rejected_without_a_gpu(lib_path):
    from expert_cached_decode_gb300 import _abi
    L = _abi.load()
    assert L.moe_layer_create(None, None) == -1
    assert b"NULL" in L.moe_last_error()
    assert L.moe_forward(None, 0, None, 1, None, None, None) == -1
    L.moe_layer_destroy(None)
    # the pool re-layout checks its arguments before touching the GPU
    buf = ctypes.create_string_buffer(64)
    assert L.moe_pack_experts(None, buf, 1, 256, 64, None) == -1
    assert L.moe_pack_experts(buf, buf, -1, 256, 64, None) == -1
    assert L.moe_pack_experts(buf, buf, 1, 200, 64, None) == -1
    assert L.moe_pack_experts(buf, buf, 1, 256, 96, None) == -1
    assert L.moe_pack_experts(buf, buf, 0, 256, 64, None) == 0


def test_kv_window_arguments_are_rejected_without_a_gpu(lib_path):
    from expert_cached_decode_gb300 import _abi
    L = _abi.load()
    assert L.moe_kv_create(None, None) == -1
    out = ctypes.c_void_p()
    host = ctypes.create_string_buffer(4096 + 16)
    base = ctypes.addressof(host) + (-ctypes.addressof(host)) % 16

    def desc(**kw):
        d = dict(n_layers=1, cell_bytes=64, n_cells=64, resident_cells=32, block_cells=8, host_cells=base)
        d.update(kw)
        return _abi.MoeKvDesc(**d)

    for bad in (dict(n_layers=0), dict(cell_bytes=40), dict(block_cells=0), dict(n_cells=60),
                dict(resident_cells=36), dict(resident_cells=72), dict(host_cells=None), dict(host_cells=base + 8)):
        assert L.moe_kv_create(ctypes.byref(desc(**bad)), ctypes.byref(out)) == -1, bad
        assert out.value is None
    assert L.moe_kv_read_blocks(None, 0, None, 1, None, None) == -1
    assert L.moe_kv_write(None, 0, 0, 1, None, None) == -1
    assert L.moe_kv_stats(None, None, None) == -1
    L.moe_kv_destroy(None)
