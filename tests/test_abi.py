"""The C-ABI library loads and exports every entry point of include/moe.h;
size helpers and host-side argument validation (no GPU needed: every call
here returns before anything touches a device).

The validation tests pass stand-in addresses (1 << 20) for device buffers.
They run only where no GPU is visible, so a validation regression can never
launch a kernel on those addresses; tests/test_gpu_rejections.py repeats the
checks with real device buffers on a GPU."""
import ctypes
import os
import re

import pytest

import quantized_routed_expert_router_gb300 as moe
from helpers import q8_row_bytes

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _gpu_visible():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:  # pragma: no cover
        return False


# stand-in device addresses are passed only where nothing can be launched
host_only = pytest.mark.skipif(_gpu_visible(), reason="stand-in device addresses: host-only check")


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
    # Q6_K: a 4-byte {d, 0, 0} entry per row and block instead of the 2-byte d;
    # Q3_K: 112 bytes per row and block instead of 110
    assert moe.moe_packed_bytes(moe.Q6_K, 64, 2048) == 64 * 8 * 212
    assert moe.moe_packed_bytes(moe.Q3_K, 64, 2048) == 64 * 8 * 112
    assert moe.moe_packed_bytes(moe.Q6_K, 32, 2880) == 0 and moe.moe_packed_bytes(moe.Q3_K, 32, 2880) == 0
    for code in (7, -1):
        assert moe.moe_packed_bytes(code, 32, 2048) == 0


@host_only
def test_argument_errors_return_before_launch():
    L = moe.lib()
    INVALID, UNSUP, WS = 1, 2, 3
    s = ctypes.c_void_p(0)
    assert L.moe_pack_weights(None, moe.Q4_K, 32, 256, None, s) == INVALID
    assert L.moe_pack_weights(1 << 20, moe.F32, 32, 256, 1 << 20, s) == UNSUP
    assert L.moe_quantize_q8K(None, 1, 100, None, s) == UNSUP
    assert L.moe_quantize_q8K(None, 1, 256, None, s) == INVALID
    assert L.moe_quantize_q8K(None, 0, 256, None, s) == 0          # T = 0: no-op
    args = [None, None, 1, 512, None, moe.F32, 16, None, 2, 0, 1, None, None, None, None, None, None, 0, s]
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
    assert L.moe_expert_ffn(None, 1, None, None, 2, None, None, None, None, None, 0, s) == INVALID
    pool = moe._Pool(moe.Q4_K, 2048, 500, 8, 1 << 20)                 # I not a multiple of 32
    assert L.moe_expert_ffn(1 << 20, 1, 1 << 20, 1 << 20, 2, ctypes.byref(pool), None, None, 1 << 20, None, 0, s) == INVALID
    pool = moe._Pool(moe.Q4_K, 2048, 544, 8, 1 << 20)                 # Q4_K needs 256-multiples
    assert L.moe_expert_ffn(1 << 20, 1, 1 << 20, 1 << 20, 2, ctypes.byref(pool), None, None, 1 << 20, None, 0, s) == UNSUP
    for code in (7, -1):                                               # codes the library does not know
        assert L.moe_pack_weights(1 << 20, code, 32, 2048, 1 << 20, s) == UNSUP
        pool = moe._Pool(code, 2048, 512, 8, 1 << 20)
        assert L.moe_expert_ffn(1 << 20, 1, 1 << 20, 1 << 20, 2, ctypes.byref(pool), None, None, 1 << 20, None, 0,
                                s) == INVALID
    for code in (moe.Q6_K, moe.Q3_K):                                  # 256-column formats
        pool = moe._Pool(code, 2048, 544, 8, 1 << 20)
        assert L.moe_expert_ffn(1 << 20, 1, 1 << 20, 1 << 20, 2, ctypes.byref(pool), None, None, 1 << 20, None, 0,
                                s) == UNSUP
    pool = moe._Pool(moe.Q4_K, 2048, 512, 8, 1 << 20)
    assert L.moe_expert_ffn(1 << 20, 1, 1 << 20, 1 << 20, 2, ctypes.byref(pool), None, None, 1 << 20, None, 0, s) == WS
    assert L.moe_expert_ffn(1 << 20, 0, 1 << 20, 1 << 20, 2, ctypes.byref(pool), None, None, 1 << 20, None, 0, s) == 0
    assert L.moe_debug_row_dots(None, moe.Q4_K, 32, 256, 0, None, None, s) == INVALID
    assert moe.status_str(3).startswith("workspace")


@host_only
def test_layer_call_sizes_and_argument_errors():
    """The layer call's workspace follows its batch-size dispatch, and its
    argument and workspace checks return before anything is launched."""
    L = moe.lib()
    INVALID, UNSUP, WS = 1, 2, 3
    s = ctypes.c_void_p(0)
    pool = moe._Pool(moe.Q4_K, 2048, 512, 256, 1 << 20)
    shared = moe._Pool(moe.Q4_K, 2048, 512, 1, 1 << 21)
    wsz = {T: L.moe_layer_workspace_bytes(T, 8, ctypes.byref(pool), ctypes.byref(shared)) for T in (1, 4, 5, 16)}
    assert all(v > 0 for v in wsz.values())
    assert wsz[1] < wsz[4]                       # one persistent launch: tagged words per pair
    assert wsz[5] < wsz[16]                      # separate kernels: their own workspaces
    assert L.moe_layer_workspace_bytes(0, 8, ctypes.byref(pool), None) == 0
    P = 1 << 20

    def call(T=1, k=8, pool_=pool, shared_=shared, rtype=moe.F32, ws=None, ws_bytes=0, hidden=P):
        return L.moe_layer_forward(hidden, T, P, rtype, None, k, 0, 1, ctypes.byref(pool_),
                                   ctypes.byref(shared_) if shared_ is not None else None, None, P,
                                   None, None, None, None, ws, ws_bytes, 0, s)

    assert call(T=17) == INVALID                  # above the token limit
    assert call(k=300) == INVALID                 # k > E
    assert call(rtype=moe.Q4_K) == UNSUP          # routers are F32 or Q8_0
    assert call(hidden=None) == INVALID
    assert call(hidden=P + 4) == INVALID          # hidden must be 16-byte aligned
    assert call(T=0) == 0                         # no tokens: nothing to do
    for T in (1, 4, 16):                          # both dispatch paths check the workspace first
        assert call(T=T) == WS
        assert call(T=T, ws=P, ws_bytes=wsz[T] - 1) == WS
    odd = moe._Pool(moe.Q4_K, 2048, 512, 1, 1 << 21)
    odd_shared_h = moe._Pool(moe.Q4_K, 1024, 512, 1, 1 << 21)
    assert call(shared_=odd_shared_h) == INVALID  # the shared expert must match H
    assert call(shared_=odd) == WS
    mx_shared = moe._Pool(moe.MXFP4, 2048, 512, 1, 1 << 21)
    assert call(shared_=mx_shared) == UNSUP       # shared: the routed format or Q8_0
    q8_shared = moe._Pool(moe.Q8_0, 2048, 512, 1, 1 << 21)
    assert call(shared_=q8_shared) == WS


@host_only
def test_documented_alignment_errors():
    """Buffers the header marks 16-byte aligned are refused before any launch
    when they are not."""
    L = moe.lib()
    INVALID = 1
    s = ctypes.c_void_p(0)
    P = 1 << 20
    assert L.moe_quantize_q8K(P + 4, 1, 256, P, s) == INVALID          # x
    assert L.moe_quantize_q8K(P, 1, 256, P + 8, s) == INVALID          # xq
    args = [P, None, 1, 512, P, moe.F32, 16, None, 2, 0, 1, P, P, None, None, None, P, 1 << 16, s]
    bad_h = list(args); bad_h[0] = P + 4
    assert L.moe_route(*bad_h) == INVALID                               # hidden, F32 router
    bad_w = list(args); bad_w[4] = P + 4
    assert L.moe_route(*bad_w) == INVALID                               # router rows
    pool = moe._Pool(moe.Q4_K, 2048, 512, 8, P)
    ffn = [P, 1, P, P, 2, ctypes.byref(pool), None, None, P, None, 0, s]
    bad_y = list(ffn); bad_y[8] = P + 4
    assert L.moe_expert_ffn(*bad_y) == INVALID                          # y
    bad_x = list(ffn); bad_x[0] = P + 8
    assert L.moe_expert_ffn(*bad_x) == INVALID                          # xq


def test_fused_gate_up_entry_points_into_one_buffer():
    """A fused gate_up matrix packed as one buffer: the pool's up pointer is the
    gate pointer plus the packed bytes of I rows (host-side table only)."""
    import torch
    H, I = 2048, 512
    for qt in (moe.Q4_K, moe.Q2_K, moe.Q8_0, moe.MXFP4):
        half = moe.moe_packed_bytes(qt, I, H)
        assert half > 0 and half % 16 == 0
        assert moe.moe_packed_bytes(qt, 2 * I, H) == 2 * half      # 32-row tiles stack
        gu = torch.zeros(2 * half, dtype=torch.uint8)
        down = torch.zeros(moe.moe_packed_bytes(qt, H, I), dtype=torch.uint8)
        pool = moe.ExpertPool(qt, H, I, [dict(gate_up=gu, down=down), None], device="cpu")
        t = pool.table.tolist()
        assert t[0][:3] == [gu.data_ptr(), gu.data_ptr() + half, down.data_ptr()]
        assert t[1] == [0] * 6
    with pytest.raises(ValueError):
        moe.ExpertPool(moe.Q4_K, H, I, [dict(gate_up=torch.zeros(10, dtype=torch.uint8), down=down)],
                       device="cpu")
    with pytest.raises(ValueError):
        moe.ExpertPool(moe.Q4_K, H, I, [dict(gate_up=gu, gate=gu, down=down)], device="cpu")
