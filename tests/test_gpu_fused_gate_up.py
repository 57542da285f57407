"""A pool built from fused gate_up matrices (one [2I][H] matrix per expert,
gate rows first, packed as one) gives y within the stated tolerance of the
CPU oracle (which reads the separate gate and up blocks), and the same y, bit
for bit, as the pool built from separate gate and up matrices, on both layer
paths."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_y_close

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("quantized_routed_expert_router_gb300")
from quantized_routed_expert_router_gb300.device_layer import DeviceLayer  # noqa: E402


@pytest.mark.parametrize("name", ["a3b", "oss20b"])
def test_fused_gate_up_pool_matches_separate_matrices(name):
    base = synth.CONFIGS[name]
    cfg = (synth.shrink(base, H=512, I=256, E=4, k=2, shared_I=0) if name == "a3b"
           else synth.shrink(base, H=320, I=288, E=4, k=2))
    L = synth.make_layer(cfg, 0, T=2)
    ref = oracle.layer_forward(L)
    dl = DeviceLayer(L, "cuda")
    dl.forward()
    torch.cuda.synchronize()
    y_ref = dl.y.clone()
    sd = dl.sizes[2]
    entries = []
    for e in range(cfg.E):
        blocks = torch.from_numpy(np.ascontiguousarray(np.concatenate([L.gate[e], L.up[e]], axis=0))).cuda()
        gu = moe.pack(blocks, cfg.qtype, 2 * cfg.I, cfg.H)
        en = dict(gate_up=gu, down=dl.down[e * sd:(e + 1) * sd])
        if dl.bg is not None:
            en.update(b_gate=dl.bg[e], b_up=dl.bu[e], b_down=dl.bd[e])
        entries.append(en)
    pool = moe.ExpertPool(cfg.qtype, cfg.H, cfg.I, entries)
    y3 = torch.empty_like(dl.y)
    dl.ffn(pool=pool, y=y3)
    y1 = torch.empty_like(dl.y)
    dl.forward_fused(pool=pool, y=y1, outputs=False)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(dl.ws_ffn) == 0 and moe.moe_read_device_status(dl.ws_layer) == 0
    assert np.array_equal(dl.ids.cpu().numpy(), ref["ids"])
    assert_y_close(y3.cpu().numpy(), ref["y"], f"{name} fused gate_up, three calls")
    assert_y_close(y1.cpu().numpy(), ref["y"], f"{name} fused gate_up, one launch")
    assert torch.equal(y3, y_ref)
    assert torch.equal(y1, y_ref)
