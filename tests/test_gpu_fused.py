"""moe_layer_forward (one launch per layer) against the CPU oracle and against
the three-call path (quantise, route, expert FFN) through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_y_close, unpack_q8_records

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("quantized_routed_expert_router_gb300")
from quantized_routed_expert_router_gb300.device_layer import DeviceLayer  # noqa: E402

SMALL = {
    "tiny q8_0": (synth.shrink(synth.CONFIGS["tiny"], E=6), 3),
    "a3b q4_K + shared": (synth.shrink(synth.CONFIGS["a3b"], H=1024, I=512, E=16, k=4, shared_I=256), 3),
    "oss20b mxfp4 + biases, ragged records": (synth.shrink(synth.CONFIGS["oss20b"], H=2880, I=320, E=6, k=3), 4),
    "wide q2_K + q8_0 shared, q8_0 router": (synth.shrink(synth.CONFIGS["wide"], H=1536, I=512, E=12, k=4,
                                                          shared_I=512), 2),
    "a22b q4_K T=16 zipf": (synth.shrink(synth.CONFIGS["a22b"], H=1024, I=768, E=24, k=4), 16),
    "a22b q4_K T=1": (synth.shrink(synth.CONFIGS["a22b"], H=1024, I=768, E=24, k=4), 1),
    # 1024 experts: the expert table stays in global memory and the top-k
    # holds 32 keys per lane; k = 32 is the largest selection
    "E1024 k32 T=1": (synth.shrink(synth.CONFIGS["a3b"], H=512, I=256, E=1024, k=32, shared_I=256), 1),
    "E1024 k32 T=3": (synth.shrink(synth.CONFIGS["a3b"], H=512, I=256, E=1024, k=32, shared_I=256), 3),
    "q6_K + q6_K shared T=1": (synth.shrink(synth.CONFIGS["a3b"], H=1024, I=512, E=16, k=4, shared_I=256,
                                            qtype=synth.Q6_K, shared_qtype=synth.Q6_K), 1),
    "q6_K + q8_0 shared T=3": (synth.shrink(synth.CONFIGS["a3b"], H=1024, I=512, E=16, k=4, shared_I=256,
                                            qtype=synth.Q6_K, shared_qtype=synth.Q8_0), 3),
    "q3_K + q8_0 shared, q8_0 router T=1": (synth.shrink(synth.CONFIGS["wide"], H=1536, I=512, E=12, k=4,
                                                         shared_I=512, qtype=synth.Q3_K), 1),
    "q3_K T=4": (synth.shrink(synth.CONFIGS["a22b"], H=1024, I=768, E=24, k=4, qtype=synth.Q3_K), 4),
    # the shared expert scaled per token by sigma(gate . x)
    "q4_K + gated shared T=1": (synth.shrink(synth.CONFIGS["a3b"], H=1024, I=512, E=16, k=4, shared_I=256,
                                             shared_gate=True), 1),
    "q4_K + gated shared T=3": (synth.shrink(synth.CONFIGS["a3b"], H=1024, I=512, E=16, k=4, shared_I=256,
                                             shared_gate=True), 3),
    "q2_K + gated q8_0 shared, q8_0 router T=2": (synth.shrink(synth.CONFIGS["wide"], H=1536, I=512, E=12, k=4,
                                                               shared_I=512, shared_gate=True), 2),
}


def np_(t):
    return t.detach().cpu().numpy()


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("flags", [0, 1])
def test_fused_layer_parity(name, flags):
    cfg, T = SMALL[name]
    L = synth.make_layer(cfg, 0, T=T, zipf=(T == 16))
    ref = oracle.layer_forward(L)
    dl = DeviceLayer(L, "cuda")
    dl.forward()                                   # three-call path
    torch.cuda.synchronize()
    y3 = np_(dl.y).copy()
    for rep in range(3):                           # the epoch advances between calls
        dl.y.fill_(float("nan"))
        dl.ids.fill_(-1)
        dl.forward_fused(flags=flags)
        torch.cuda.synchronize()
        assert moe.moe_read_device_status(dl.ws_layer) == 0
        assert np.array_equal(np_(dl.ids), ref["ids"])
        assert np.array_equal(np_(dl.logits), ref["logits"])
        assert np.allclose(np_(dl.w), ref["w"], rtol=1e-6, atol=1e-7)
        for g, w in zip(unpack_q8_records(np_(dl.xq), T, cfg.H), ref["xq"]):
            assert np.array_equal(g, w)
        assert_y_close(np_(dl.y), ref["y"], name)
        if T > 1:   # same arithmetic and summation order as the three calls
            assert np.array_equal(np_(dl.y), y3), rep
        else:       # one token: a unit's gate/up records are dealt over 16 warps
            assert_y_close(np_(dl.y), y3.astype(np.float64), name)   # (8 in the three calls)


def test_fused_ownership_partition():
    cfg = synth.shrink(synth.CONFIGS["wide"], H=1024, I=512, E=16, k=4, shared_I=256)
    L = synth.make_layer(cfg, 0, T=3)
    ref = oracle.layer_forward(L)
    dl = DeviceLayer(L, "cuda")
    own = np.arange(cfg.E) % 3 == 0
    ys = []
    for mask, sh in ((own, True), (~own, False)):
        y = torch.empty_like(dl.y)
        dl.forward_fused(pool=dl.make_pool(mask), shared=dl.shared if sh else None, y=y)
        torch.cuda.synchronize()
        ys.append(np_(y).astype(np.float64))
        assert_y_close(ys[-1], oracle.expert_ffn(L, ref["xq"], ref["ids"], ref["w"], owned=mask, shared=sh)["y"],
                       "partial")
    assert_y_close(ys[0] + ys[1], ref["y"], "sum of partials")
    # nothing owned and no shared expert: y = 0
    y = torch.full_like(dl.y, 7.0)
    dl.forward_fused(pool=dl.make_pool(np.zeros(cfg.E, bool)), shared=None, y=y)
    torch.cuda.synchronize()
    assert not np_(y).any()


def test_fused_back_to_back_layers_with_overlap():
    """a stack of distinct layers launched back to back with the overlap flag"""
    cfg = synth.shrink(synth.CONFIGS["a3b"], H=1024, I=512, E=32, k=4, shared_I=256)
    layers = [synth.make_layer(cfg, l, T=1) for l in range(6)]
    dls = [DeviceLayer(L, "cuda") for L in layers]
    for _ in range(2):
        for dl in dls:
            dl.forward_fused(flags=moe.LAYER_OVERLAP_PREVIOUS, outputs=False)
        torch.cuda.synchronize()
        for L, dl in zip(layers, dls):
            assert moe.moe_read_device_status(dl.ws_layer) == 0
            assert_y_close(np_(dl.y), oracle.layer_forward(L)["y"], f"layer {L.layer}")


def test_fused_stack_replayed_from_a_cuda_graph():
    """The benchmark's launch configuration: a stack of distinct layers captured
    once in a CUDA graph with the overlap flag, replayed many times.  Every
    replay must give the oracle's y (the per-launch epoch advances on the
    device, so stale words of an earlier replay are never taken), and y must
    be written afresh by each replay."""
    cfg = synth.shrink(synth.CONFIGS["a3b"], H=1024, I=512, E=32, k=4, shared_I=256)
    layers = [synth.make_layer(cfg, l, T=1) for l in range(5)]
    refs = [oracle.layer_forward(L)["y"] for L in layers]
    dls = [DeviceLayer(L, "cuda") for L in layers]
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for dl in dls:   # one eager pass first (kernel attributes are set on first use)
            dl.forward_fused(flags=moe.LAYER_OVERLAP_PREVIOUS, outputs=False)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for dl in dls:
            dl.forward_fused(flags=moe.LAYER_OVERLAP_PREVIOUS, outputs=False)
    for rep in range(4):
        for dl in dls:
            dl.y.fill_(float("nan"))
        torch.cuda.synchronize()
        for _ in range(rep + 1):
            g.replay()
        torch.cuda.synchronize()
        for L, dl, ref in zip(layers, dls, refs):
            assert moe.moe_read_device_status(dl.ws_layer) == 0
            assert_y_close(np_(dl.y), ref, f"replay {rep}, layer {L.layer}")


@pytest.mark.parametrize("T", [1, 3])
@pytest.mark.parametrize("E,k", [(64, 6), (256, 8), (64, 2)])
def test_fused_topk_ties_take_the_lowest_index(T, E, k):
    """Router rows repeated in groups of 8 give exactly equal logits: the
    one-launch selection must keep the k largest with the lower expert index
    first on ties, as the oracle does."""
    cfg = synth.shrink(synth.CONFIGS["a3b"], H=512, I=256, E=E, k=k, shared_I=0)
    L = synth.make_layer(cfg, 0, T=T)
    base = synth.normal(6, 1, 0.02, E // 8, cfg.H)
    L.router = np.ascontiguousarray(np.repeat(base, 8, axis=0))
    ref = oracle.layer_forward(L)
    assert len(np.unique(ref["logits"][0])) < E          # ties are present
    dl = DeviceLayer(L, "cuda")
    dl.forward_fused()
    torch.cuda.synchronize()
    assert moe.moe_read_device_status(dl.ws_layer) == 0
    assert np.array_equal(np_(dl.logits), ref["logits"])
    assert np.array_equal(np_(dl.ids), ref["ids"])
    assert_y_close(np_(dl.y), ref["y"], f"ties E{E} k{k} T{T}")
