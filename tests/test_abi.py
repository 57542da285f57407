"""The C-ABI library loads and exports every entry point of include/moe.h;
size helpers and host-side argument validation (no GPU needed: every call
here returns before anything touches a device)."""
import ctypes
import os
import re

import pytest

import quantized_routed_expert_router_gb300 as moe
from helpers import q8_row_bytes

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return re.findall(r"^\s*(?:moe_status|int|size_t|const char \*)\s*(moe_\w+)\(", src, re.M)


def test_library_exports_every_declared_symbol():
    names = header_functions()
    assert len(names) >= 12
    L = moe.lib()
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    assert sorted(names) == sorted(moe.EXPORTS)


def test_size_helpers():
    for n in (32, 96, 256, 512, 2048, 2880, 4096, 7168):
        assert moe.moe_act_block(n) == (256 if n % 256 == 0 else 32)
        assert moe.moe_q8_row_bytes(n) == q8_row_bytes(n)
        assert moe.moe_q8_row_bytes(n) % 16 == 0
    assert moe.moe_act_block(100) == 0 and moe.moe_q8_row_bytes(100) == 0
    # packed bytes equal the GGUF bytes (MXFP4: plus padding of a short last record)
    assert moe.moe_packed_bytes(moe.Q4_K, 512, 2048) == 512 * 8 * 144
    assert moe.moe_packed_bytes(moe.Q2_K, 64, 7168) == 64 * 28 * 84
    assert moe.moe_packed_bytes(moe.Q8_0, 32, 2048) == 32 * 64 * 34
    assert moe.moe_packed_bytes(moe.MXFP4, 32, 2048) == 32 * 64 * 17
    assert moe.moe_packed_bytes(moe.MXFP4, 32, 2880) == 32 * 88 * 17 + 2 * 512 + 256
    assert moe.moe_packed_bytes(moe.Q4_K, 33, 2048) == 0          # rows % 32
    assert moe.moe_packed_bytes(moe.Q4_K, 32, 2880) == 0          # K-quants need 256 columns
    assert moe.moe_packed_bytes(moe.F32, 32, 256) == 0


def test_argument_errors_return_before_launch():
    L = moe.lib()
    INVALID, UNSUP, WS = 1, 2, 3
    s = ctypes.c_void_p(0)
    assert L.moe_pack_weights(None, moe.Q4_K, 32, 256, None, s) == INVALID
    assert L.moe_pack_weights(1 << 20, moe.F32, 32, 256, 1 << 20, s) == UNSUP
    assert L.moe_quantize_q8K(None, 1, 100, None, s) == UNSUP
    assert L.moe_quantize_q8K(None, 1, 256, None, s) == INVALID
    assert L.moe_quantize_q8K(None, 0, 256, None, s) == 0          # T = 0: no-op
    args = [None, None, 1, 512, None, moe.F32, 16, None, 2, 0, 1, None, None, None, None, 0, s]
    assert L.moe_route(*args) == INVALID                            # NULL router
    bad_k = list(args); bad_k[8] = 17
    assert L.moe_route(*bad_k) == INVALID                            # k > E
    bad_g = list(args); bad_g[9] = 7
    assert L.moe_route(*bad_g) == INVALID
    bad_t = list(args); bad_t[5] = moe.Q4_K
    assert L.moe_route(*bad_t) == UNSUP
    ok_ptrs = list(args)
    ok_ptrs[0] = ok_ptrs[4] = ok_ptrs[11] = ok_ptrs[12] = 1 << 20
    assert L.moe_route(*ok_ptrs) == WS                               # missing workspace
    assert L.moe_expert_ffn(None, 1, None, None, 2, None, None, None, None, 0, s) == INVALID
    pool = moe._Pool(moe.Q4_K, 2048, 500, 8, 1 << 20)                 # I not a multiple of 32
    assert L.moe_expert_ffn(1 << 20, 1, 1 << 20, 1 << 20, 2, ctypes.byref(pool), None, 1 << 20, None, 0, s) == INVALID
    pool = moe._Pool(moe.Q4_K, 2048, 544, 8, 1 << 20)                 # Q4_K needs 256-multiples
    assert L.moe_expert_ffn(1 << 20, 1, 1 << 20, 1 << 20, 2, ctypes.byref(pool), None, 1 << 20, None, 0, s) == UNSUP
    pool = moe._Pool(moe.Q4_K, 2048, 512, 8, 1 << 20)
    assert L.moe_expert_ffn(1 << 20, 1, 1 << 20, 1 << 20, 2, ctypes.byref(pool), None, 1 << 20, None, 0, s) == WS
    assert L.moe_expert_ffn(1 << 20, 0, 1 << 20, 1 << 20, 2, ctypes.byref(pool), None, 1 << 20, None, 0, s) == 0
    assert L.moe_debug_row_dots(None, moe.Q4_K, 32, 256, 0, None, None, s) == INVALID
    assert moe.status_str(3).startswith("workspace")
