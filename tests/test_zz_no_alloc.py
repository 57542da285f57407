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
    L = moe.lib()
    pool = moe._Pool(moe.Q4_K, 4096, 4096, 256, 1 << 20)
    # T=16, k=32, I=4096: the h scratch alone is 8 MiB > 2 MiB
    rc = L.moe_expert_ffn_noalloc(1 << 20, 16, 1 << 20, 1 << 20, 32, ctypes.byref(pool), None, 1 << 20,
                                  ctypes.c_void_p(0))
    assert rc == 3, moe.status_str(rc)
