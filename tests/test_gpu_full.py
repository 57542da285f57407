"""Full-size layers of every synthetic workload (the shapes the benchmark and
the stacks use), fused path and three-call path, against the CPU oracle:
ids and logits bit for bit, y within the stated tolerance."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_y_close

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("quantized_routed_expert_router_gb300")
from quantized_routed_expert_router_gb300.device_layer import DeviceLayer  # noqa: E402

CASES = [("tiny", 1), ("a3b", 1), ("oss20b", 1), ("oss20b", 4), ("wide", 1), ("a22b", 1), ("a22b", 4),
         ("a22b", 16), ("a3b/q6_K", 1), ("a3b/q6_K", 4), ("wide/q3_K", 1), ("wide/q3_K", 4), ("a3b/q3_K", 16),
         ("a3b/gated", 1), ("a3b/gated", 16)]

# the two further routed-expert formats on full-size shapes: the 35B-A3B-style
# layer with Q6_K routed and shared experts, and the wide layer with Q3_K
# routed experts (Q8_0 shared expert and router as in that workload)
VARIANTS = {"a3b/q6_K": ("a3b", dict(qtype=synth.Q6_K, shared_qtype=synth.Q6_K)),
            "wide/q3_K": ("wide", dict(qtype=synth.Q3_K)),
            "a3b/q3_K": ("a3b", dict(qtype=synth.Q3_K, shared_qtype=synth.Q8_0)),
            # the 35B-A3B-style layer with a sigmoid gate on its shared expert
            "a3b/gated": ("a3b", dict(shared_gate=True))}


def config(name):
    if name in VARIANTS:
        base, kw = VARIANTS[name]
        return synth.shrink(synth.CONFIGS[base], **kw)
    return synth.CONFIGS[name]


@pytest.mark.parametrize("name,T", CASES, ids=[f"{n}-T{t}" for n, t in CASES])
def test_full_size_layer(name, T):
    cfg = config(name)
    L = synth.make_layer(cfg, 3, T=T)
    ref = oracle.layer_forward(L)
    dl = DeviceLayer(L, "cuda")
    del L.gate, L.up, L.down
    dl.forward_fused(flags=moe.LAYER_OVERLAP_PREVIOUS)
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(dl.ws_layer) == 0
    assert np.array_equal(dl.ids.cpu().numpy(), ref["ids"])
    assert np.array_equal(dl.logits.cpu().numpy(), ref["logits"])
    yf = dl.y.cpu().numpy().copy()
    assert_y_close(yf, ref["y"], f"{name} fused")
    dl.forward()
    torch.cuda.synchronize()
    assert np.array_equal(dl.ids.cpu().numpy(), ref["ids"])
    assert_y_close(dl.y.cpu().numpy(), ref["y"], f"{name} three calls")
