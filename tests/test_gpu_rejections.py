"""Argument and workspace checks on a GPU, with real device buffers: every
rejected call returns its status before anything is enqueued, so the
outputs keep the values they had (NaN here) and the device status stays
clear.  The host-only twin of these checks is tests/test_abi.py."""
import ctypes

import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("quantized_routed_expert_router_gb300")
from quantized_routed_expert_router_gb300.device_layer import DeviceLayer  # noqa: E402

INVALID, UNSUP, WS = 1, 2, 3


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def test_rejected_calls_touch_nothing():
    cfg = synth.shrink(synth.CONFIGS["a3b"], H=512, I=256, E=8, k=2, shared_I=256)
    dl = DeviceLayer(synth.make_layer(cfg, 0, T=2), "cuda")
    L = moe.lib()
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    y = torch.full_like(dl.y, float("nan"))
    pool, shared = ctypes.byref(dl.pool.c), ctypes.byref(dl.shared.c)
    ffn_ws = L.moe_ffn_workspace_bytes(2, cfg.k, pool, shared)
    # FFN: workspace one byte short, unaligned y, out-of-range k
    assert L.moe_expert_ffn(_p(dl.xq), 2, _p(dl.ids), _p(dl.w), cfg.k, pool, shared, None, _p(y), _p(dl.ws_ffn),
                            ffn_ws - 1, s) == WS
    y_off = ctypes.c_void_p(y.data_ptr() + 4)
    assert L.moe_expert_ffn(_p(dl.xq), 2, _p(dl.ids), _p(dl.w), cfg.k, pool, shared, None, y_off, _p(dl.ws_ffn),
                            ffn_ws, s) == INVALID
    assert L.moe_expert_ffn(_p(dl.xq), 2, _p(dl.ids), _p(dl.w), 0, pool, shared, None, _p(y), _p(dl.ws_ffn),
                            ffn_ws, s) == INVALID
    # layer call: workspace one byte short (both dispatch paths)
    for T in (2, 8):
        need = L.moe_layer_workspace_bytes(T, cfg.k, pool, shared)
        ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
        x = torch.zeros((T, cfg.H), dtype=torch.float32, device="cuda")
        yT = torch.full((T, cfg.H), float("nan"), device="cuda")
        assert L.moe_layer_forward(_p(x), T, _p(dl.router), moe.F32, None, cfg.k, 0, 1, pool, shared, None, _p(yT),
                                   None, None, None, None, _p(ws), need - 1, 0, s) == WS
        assert bool(torch.isnan(yT).all())
        assert int(ws.count_nonzero()) == 0
    # route: k larger than E
    ids = torch.full((2, cfg.k), -7, dtype=torch.int32, device="cuda")
    assert L.moe_route(_p(dl.x), None, 2, cfg.H, _p(dl.router), moe.F32, cfg.E, None, cfg.E + 1, 0, 1, _p(ids),
                       _p(dl.w), None, None, None, _p(dl.ws_route), dl.ws_route.numel(), s) == INVALID
    torch.cuda.synchronize()
    assert bool(torch.isnan(y).all())
    assert int((ids == -7).sum()) == ids.numel()
    assert moe.moe_read_device_status(dl.ws_ffn) == 0
