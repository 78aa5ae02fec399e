"""The C-ABI library builds, loads and exports every symbol include/mok.h
declares; host-side argument checks reject bad input without touching a GPU."""
import ctypes
import os
import re

import pytest

from combine_router_top_expert_gb300 import build, mok

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mok.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mok_[a-z_0-9]+)\s*\(", src)))


def test_library_builds_and_exports_every_declared_symbol():
    build.build()
    L = mok.lib()
    decl = declared_functions()
    assert len(decl) >= 15
    for name in decl:
        assert hasattr(L, name), name
    assert sorted(decl) == sorted(mok.EXPORTS)


def test_sizes_and_host_validation():
    L = mok.lib()
    assert mok.version().startswith("mok-gb300")
    assert mok.route_workspace_size(64, 128, 8, 2) > 256
    assert mok.route_workspace_size(64, 128, 8, 9) == 0            # k > E
    assert mok.packed_weights_size(8, 128, 64, mok.BF16) == 1024 * ((8 * 128 * 128 * 2 + 1023) // 1024) * 2 // 2 + \
        1024 * ((8 * 128 * 64 * 2 + 1023) // 1024)
    assert mok.packed_weights_size(8, 100, 64, mok.BF16) == 0       # H % 128
    assert mok.packed_weights_size(8, 128, 64, mok.MXFP8) == 0      # I % 128 for MXFP8
    p = mok.make_problem(64, 128, 64, 8, 2)
    assert mok.workspace_size(p) > 0
    assert mok.saved_size(p) > 0
    assert mok.padded_rows_max(64, 8, 2) == 64 * 2 + 8 * 128
    bad = mok.make_problem(64, 128, 64, 8, 0)
    assert mok.workspace_size(bad) == 0
    # invalid arguments are rejected before any CUDA call
    rc = L.mok_moe_forward(ctypes.byref(bad), None, None, None)
    assert rc == mok.ERR_INVALID
    rc = L.mok_route_layout(None, None, None, 64, 128, 8, 9, None, None, None, None, None, None, None, 0, None)
    assert rc == mok.ERR_INVALID
    rc = L.mok_pack_weights(8, 100, 64, 0, None, None, None, None, 0, None)
    assert rc == mok.ERR_INVALID
    rc = L.mok_quantize_rows(None, 64, 100, None, None, None)       # H % 128
    assert rc == mok.ERR_INVALID
    rc = L.mok_quantize_rows(None, 64, 128, None, None, None)       # null buffers
    assert rc == mok.ERR_INVALID
    pm = mok.make_problem(64, 128, 128, 8, 2, mok.MXFP8)
    rc = L.mok_dispatch_quantized(ctypes.byref(p), None, None, None, None, None, None)   # BF16 problem
    assert rc == mok.ERR_INVALID
    rc = L.mok_dispatch_quantized(ctypes.byref(pm), None, None, None, None, None, None)  # no routing
    assert rc == mok.ERR_INVALID
    assert L.mok_status_string(3) == b"device wait timed out"


def test_product_path_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "combine_router_top_expert_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "mok_oracle" not in text, f
