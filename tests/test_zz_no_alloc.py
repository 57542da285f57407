"""moe_expert_ffn_noalloc: the FFN for callers that cannot allocate device
memory (fixed start-up memory plans, plugin hosts without an allocator,
paths where cudaMalloc/cudaFree may not run).  It must give the same results
as moe_expert_ffn with a caller workspace, call after call, although every
call reuses one fixed scratch array in the library.  This file is collected
last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from helpers import assert_y_close

moe = pytest.importorskip("quantized_routed_expert_router_gb300")
from quantized_routed_expert_router_gb300.device_layer import DeviceLayer  # noqa: E402

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_entry_point_twice_in_a_row():
    cfg = synth.shrink(synth.CONFIGS["a3b"], H=1024, I=512, E=16, k=4, shared_I=256)
    layers = [DeviceLayer(synth.make_layer(cfg, l, T=3), "cuda") for l in (0, 1)]
    refs = []
    for dl in layers:
        dl.quantize()
        dl.route()
        dl.ffn()
        refs.append(dl.y.cpu().numpy().astype(np.float64))
    # two calls in a row on different inputs: the second must not see the
    # first call's leftovers in the shared scratch
    for dl, ref in zip(layers, refs):
        y = torch.full_like(dl.y, float("nan"))
        moe.moe_expert_ffn_noalloc(dl.xq, dl.T, dl.ids, dl.w, dl.k, dl.pool, dl.shared, y)
        torch.cuda.synchronize()
        assert_y_close(y.cpu().numpy(), ref, "noalloc vs workspace")
    # and the same input again
    dl, ref = layers[0], refs[0]
    y = torch.full_like(dl.y, float("nan"))
    moe.moe_expert_ffn_noalloc(dl.xq, dl.T, dl.ids, dl.w, dl.k, dl.pool, dl.shared, y)
    torch.cuda.synchronize()
    assert_y_close(y.cpu().numpy(), ref, "noalloc repeat")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """Real (small) device buffers: the call must refuse the shape before it
    enqueues anything, so y keeps its NaNs."""
    L = moe.lib()
    T, k, H, I, E = 16, 32, 4096, 4096, 256
    dev = "cuda"
    xq = torch.zeros(T * moe.moe_q8_row_bytes(H), dtype=torch.uint8, device=dev)
    ids = torch.zeros((T, k), dtype=torch.int32, device=dev)
    w = torch.zeros((T, k), dtype=torch.float32, device=dev)
    y = torch.full((T, H), float("nan"), device=dev)
    table = torch.zeros((E, 6), dtype=torch.int64, device=dev)   # every expert "not mine"
    pool = moe._Pool(moe.Q4_K, H, I, E, table.data_ptr())
    # T=16, k=32, I=4096: the h scratch alone is 8 MiB > 2 MiB
    rc = L.moe_expert_ffn_noalloc(xq.data_ptr(), T, ids.data_ptr(), w.data_ptr(), k, ctypes.byref(pool), None,
                                  None, y.data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 3, moe.status_str(rc)
    torch.cuda.synchronize()
    assert bool(torch.isnan(y).all())
