"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Integer and index results are compared bit for bit (q8 codes and scales,
router logits and ids, per-sub-block int32 dots); fp32 outputs are compared
with the stated tolerance max|err| <= 1e-3 * max|y_ref| + 1e-5, routing
weights to 1e-6 relative (fp32 exp against the oracle's fp64).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from helpers import assert_y_close, pack_q8_records, unpack_q8_records

pytestmark = pytest.mark.gpu

moe = pytest.importorskip("quantized_routed_expert_router_gb300")
from quantized_routed_expert_router_gb300.device_layer import DeviceLayer  # noqa: E402

DEV = "cuda"


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(DEV)


# ------------------------------------------------------------- quantiser

@pytest.mark.parametrize("n", [256, 512, 2048, 2880, 7168, 96])
@pytest.mark.parametrize("T", [1, 3, 16])
def test_quantize_bit_exact(n, T):
    x = synth.normal(11, n * 131 + T, 1.0, T, n)
    x[0, : min(n, 64)] = 0.0                     # all-zero block(s)
    x[-1, n // 2] = 40.0                          # one spike
    x[T // 2] *= 1e-4                             # tiny scale
    xq = moe.quantize(to_dev(x))
    torch.cuda.synchronize()
    got = unpack_q8_records(xq.cpu().numpy(), T, n)
    want = oracle.quantize(x)
    for g, w, name in zip(got, want, ("d", "q", "bsum")):
        assert np.array_equal(g, w), name


# ----------------------------------------------------------- integer dots

@pytest.mark.parametrize("qt,cols", [(synth.Q4_K, 2048), (synth.Q2_K, 1024), (synth.Q8_0, 512),
                                     (synth.MXFP4, 2880), (synth.MXFP4, 256), (synth.Q6_K, 2048),
                                     (synth.Q3_K, 1536), (synth.Q6_K, 256), (synth.Q3_K, 7168)])
def test_row_dots_bit_exact(qt, cols):
    rows = 64
    W = synth.matrix(qt, 3, 900 + qt, 0.02, rows, cols)
    x = synth.normal(3, 901 + qt, 1.0, 1, cols)
    d, q, bs = oracle.quantize(x)
    rec = to_dev(pack_q8_records(d, q, bs))
    packed = moe.pack(to_dev(W), qt, rows, cols)
    nsub = {synth.Q4_K: 8, synth.Q2_K: 16, synth.Q8_0: 1, synth.MXFP4: 1, synth.Q6_K: 16, synth.Q3_K: 16}[qt]
    qk = {synth.Q4_K: 256, synth.Q2_K: 256, synth.Q8_0: 32, synth.MXFP4: 32, synth.Q6_K: 256, synth.Q3_K: 256}[qt]
    n_out = cols // qk * nsub
    for row in (0, 1, 31, 32, 45, 63):
        out = torch.full((n_out + 8,), -7, dtype=torch.int32, device=DEV)
        moe.moe_debug_row_dots(packed, qt, rows, cols, row, rec, out)
        torch.cuda.synchronize()
        want = oracle.row_isums(qt, W[row], cols, q[0])
        assert np.array_equal(out[:n_out].cpu().numpy(), want), row


def test_down_dots_bit_exact_on_oracle_hq():
    """the down projection's int dots, fed the oracle's own requantised h"""
    cfg = synth.shrink(synth.CONFIGS["a3b"], H=512, I=512, E=4, k=2, shared_I=0)
    L = synth.make_layer(cfg, 0, T=1)
    res = oracle.layer_forward(L, want_h=True)
    e = int(res["ids"][0, 0])
    rec = to_dev(pack_q8_records(res["hd"][0, 0][None], res["hq"][0, 0][None], res["hbs"][0, 0][None]))
    packed = moe.pack(to_dev(L.down[e]), cfg.qtype, cfg.H, cfg.I)
    out = torch.empty(cfg.I // 256 * 8, dtype=torch.int32, device=DEV)
    for row in (0, 7, 100, 511):
        moe.moe_debug_row_dots(packed, cfg.qtype, cfg.H, cfg.I, row, rec, out)
        torch.cuda.synchronize()
        assert np.array_equal(out.cpu().numpy(), oracle.row_isums(cfg.qtype, L.down[e][row], cfg.I,
                                                                   res["hq"][0, 0]))


# ------------------------------------------------------------------ router

ROUTERS = [
    ("f32 E16 H512 k2", dict(H=512, E=16, k=2, rq=synth.F32, gating="softmax")),
    ("f32 E256 H2048 k8", dict(H=2048, E=256, k=8, rq=synth.F32, gating="softmax")),
    ("f32 E32 H2880 k4", dict(H=2880, E=32, k=4, rq=synth.F32, gating="softmax")),
    ("q8_0 E256 H7168 k8 sigmoid", dict(H=7168, E=256, k=8, rq=synth.Q8_0, gating="sigmoid")),
    ("f32 E128 H4096 k8", dict(H=4096, E=128, k=8, rq=synth.F32, gating="softmax")),
    ("f32 E100 H1024 k5 ragged", dict(H=1024, E=100, k=5, rq=synth.F32, gating="softmax")),
    ("f32 E1024 H256 k32", dict(H=256, E=1024, k=32, rq=synth.F32, gating="sigmoid")),
]


@pytest.mark.parametrize("name,p", ROUTERS, ids=[r[0] for r in ROUTERS])
@pytest.mark.parametrize("T", [1, 4, 16])
@pytest.mark.parametrize("bias", [False, True])
@pytest.mark.parametrize("renorm", [True, False])
def test_route_bit_exact_ids(name, p, T, bias, renorm):
    H, E, k, rq = p["H"], p["E"], p["k"], p["rq"]
    W = synth.matrix(rq, 5, 77 + H + E, 0.02, E, H)
    x = synth.normal(5, 78 + H, 1.0, T, H)
    b = synth.normal(5, 79, 1.0, 1, E)[0] if bias else None
    gating = oracle.SIGMOID if p["gating"] == "sigmoid" else oracle.SOFTMAX
    xq_o = oracle.quantize(x) if rq == synth.Q8_0 else None
    logits = oracle.router_logits(W, x, rq, b, xq=xq_o)
    ids, w = oracle.topk(logits, k, gating, renorm)
    xd = to_dev(x)
    xq = moe.quantize(xd)
    g_ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    g_w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    g_l = torch.empty((T, E), dtype=torch.float32, device=DEV)
    ws = torch.zeros(moe.moe_route_workspace_bytes(T, E, H), dtype=torch.uint8, device=DEV)
    for _ in range(2):   # the second call checks the ticket was rearmed
        moe.moe_route(xd, xq, to_dev(W), rq, E, None if b is None else to_dev(b), k, gating, renorm,
                      g_ids, g_w, g_l, ws)
        torch.cuda.synchronize()
        assert np.array_equal(g_l.cpu().numpy(), logits)
        assert np.array_equal(g_ids.cpu().numpy(), ids)
        gw = g_w.cpu().numpy().astype(np.float64)
        assert np.allclose(gw, w, rtol=1e-6, atol=1e-7)
    if renorm:
        assert np.allclose(gw.sum(1), 1.0, atol=1e-6)


def test_route_tie_break_lowest_index():
    """rows of identical weights give exactly equal logits: ids must be the lowest indices"""
    H, E, k, T = 512, 64, 6, 3
    base = synth.normal(6, 1, 0.02, 8, H)
    W = np.repeat(base, E // 8, axis=0)             # experts 0..7 equal, 8..15 equal, ...
    x = synth.normal(6, 2, 1.0, T, H)
    logits = oracle.router_logits(W, x)
    ids, _ = oracle.topk(logits, k)
    g_ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    g_w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    ws = torch.zeros(moe.moe_route_workspace_bytes(T, E, H), dtype=torch.uint8, device=DEV)
    xd = to_dev(x)
    moe.moe_route(xd, None, to_dev(W), synth.F32, E, None, k, oracle.SOFTMAX, True, g_ids, g_w, None, ws)
    torch.cuda.synchronize()
    assert np.array_equal(g_ids.cpu().numpy(), ids)
    assert np.array_equal(np.argsort(-logits, 1, kind="stable")[:, :k], ids)


# --------------------------------------------------------------------- FFN

SMALL = {
    "tiny q8_0 (several tiles)": (synth.shrink(synth.CONFIGS["tiny"], E=6), 3),
    "a3b q4_K + shared": (synth.shrink(synth.CONFIGS["a3b"], H=1024, I=512, E=16, k=4, shared_I=256), 3),
    "oss20b mxfp4 + biases, ragged records": (synth.shrink(synth.CONFIGS["oss20b"], H=2880, I=320, E=6, k=3), 4),
    "wide q2_K + q8_0 shared, q8_0 router": (synth.shrink(synth.CONFIGS["wide"], H=1536, I=512, E=12, k=4,
                                                          shared_I=512), 2),
    "a22b q4_K T=16 zipf": (synth.shrink(synth.CONFIGS["a22b"], H=1024, I=768, E=24, k=4), 16),
}


def gpu_layer(L, **kw):
    dl = DeviceLayer(L, DEV, **kw)
    dl.forward()
    torch.cuda.synchronize()
    return dl


@pytest.mark.parametrize("name", list(SMALL))
def test_layer_parity(name):
    cfg, T = SMALL[name]
    L = synth.make_layer(cfg, 0, T=T, zipf=(T == 16))
    ref = oracle.layer_forward(L)
    dl = gpu_layer(L)
    assert np.array_equal(dl.ids.cpu().numpy(), ref["ids"])
    assert np.array_equal(dl.logits.cpu().numpy(), ref["logits"])
    assert np.allclose(dl.w.cpu().numpy(), ref["w"], rtol=1e-6, atol=1e-7)
    got = unpack_q8_records(dl.xq.cpu().numpy(), T, cfg.H)
    for g, w in zip(got, ref["xq"]):
        assert np.array_equal(g, w)
    assert_y_close(dl.y.cpu().numpy(), ref["y"], name)
    assert moe.moe_read_device_status(dl.ws_ffn) == 0


@pytest.mark.parametrize("name", list(SMALL))
def test_ffn_on_oracle_routing(name):
    """the expert FFN alone, fed the oracle's xq, ids and weights"""
    cfg, T = SMALL[name]
    L = synth.make_layer(cfg, 1, T=T)
    ref = oracle.layer_forward(L)
    dl = DeviceLayer(L, DEV)
    dl.xq.copy_(to_dev(pack_q8_records(*ref["xq"])))
    ids = to_dev(ref["ids"].astype(np.int32))
    w = to_dev(ref["w"].astype(np.float32))
    dl.ffn(ids=ids, w=w)
    torch.cuda.synchronize()
    y_ref = oracle.expert_ffn(L, ref["xq"], ref["ids"], ref["w"].astype(np.float32).astype(np.float64))["y"]
    assert_y_close(dl.y.cpu().numpy(), y_ref, name)


def test_batch_invariance_and_determinism():
    cfg = synth.shrink(synth.CONFIGS["a22b"], H=1024, I=512, E=32, k=4)
    L16 = synth.make_layer(cfg, 2, T=16, zipf=True)
    dl16 = gpu_layer(L16)
    y16 = dl16.y.cpu().numpy().copy()
    dl16.forward()
    torch.cuda.synchronize()
    assert np.array_equal(dl16.y.cpu().numpy(), y16)          # run to run
    for t in (0, 5, 15):
        L1 = synth.make_layer(cfg, 2, T=16, zipf=True)
        L1.x = L16.x[t:t + 1].copy()
        dl1 = gpu_layer(L1)
        assert np.array_equal(dl1.ids.cpu().numpy()[0], dl16.ids.cpu().numpy()[t])
        assert np.array_equal(dl1.y.cpu().numpy()[0], y16[t])  # bit-identical across batch sizes


def test_ownership_partition_and_null_slots():
    cfg = synth.shrink(synth.CONFIGS["wide"], H=1024, I=512, E=16, k=4, shared_I=256)
    L = synth.make_layer(cfg, 0, T=3)
    ref = oracle.layer_forward(L)
    dl = gpu_layer(L)
    own = np.arange(cfg.E) % 2 == 0
    ys = []
    for mask, sh in ((own, True), (~own, False)):
        pool = dl.make_pool(mask)
        y = torch.empty_like(dl.y)
        dl.ffn(pool=pool, shared=dl.shared if sh else None, y=y)
        torch.cuda.synchronize()
        ys.append(y.cpu().numpy().astype(np.float64))
        ref_part = oracle.expert_ffn(L, ref["xq"], ref["ids"], ref["w"], owned=mask, shared=sh)["y"]
        assert_y_close(ys[-1], ref_part, "partial")
    assert_y_close(ys[0] + ys[1], ref["y"], "sum of partials")


def test_bad_ids_are_flagged_and_skipped():
    cfg = synth.shrink(synth.CONFIGS["tiny"], E=8, k=3)
    L = synth.make_layer(cfg, 0, T=2)
    ref = oracle.layer_forward(L)
    dl = DeviceLayer(L, DEV)
    dl.quantize()
    ids = np.array([[1, 99, 4], [2, 2, -1]], np.int32)
    w = np.array([[0.5, 0.25, 0.25], [0.6, 0.3, 0.1]], np.float32)
    dl.ffn(ids=to_dev(ids), w=to_dev(w))
    flags = moe.moe_read_device_status(dl.ws_ffn, clear=True)
    assert flags == (moe.DEV_BAD_ID | moe.DEV_DUP_ID)
    assert moe.moe_read_device_status(dl.ws_ffn) == 0
    keep_ids = np.array([[1, 4], [2, 0]], np.int32)
    keep_w = np.array([[0.5, 0.25], [0.6, 0.0]])
    y_ref = oracle.expert_ffn(L, ref["xq"], keep_ids, keep_w)["y"]
    assert_y_close(dl.y.cpu().numpy(), y_ref, "skipped slots")


def test_zero_tokens_and_errors():
    cfg = synth.shrink(synth.CONFIGS["tiny"], E=4)
    L = synth.make_layer(cfg, 0, T=1)
    dl = DeviceLayer(L, DEV)
    dl.ffn(T=0)   # no-op
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_expert_ffn(dl.xq, 1, dl.ids, dl.w, dl.k, dl.pool, None, dl.y, dl.ws_ffn[:64])
    assert ei.value.status == 3
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_expert_ffn(dl.xq, 17, dl.ids, dl.w, dl.k, dl.pool, None, dl.y, dl.ws_ffn)
    assert ei.value.status == 1


@pytest.mark.parametrize("T", [1, 5, 16])
@pytest.mark.parametrize("H", [512, 2880, 7168])
def test_route_shared_gate_weight(T, H):
    """moe_route's per-token shared-expert weight sigma(w . x): the fp32 logit
    in the router's fixed order (bit-exact with the oracle's one-row router)
    through fp32 exp, against the oracle's fp64 sigmoid of the same logit."""
    E, k = 16, 2
    W = synth.normal(7, H, 0.02, E, H)
    g = synth.normal(7, H + 1, 0.02, 1, H)[0]
    x = synth.normal(7, H + 2, 1.0, T, H)
    _, want = oracle.shared_gate(g, x)
    ids = torch.empty((T, k), dtype=torch.int32, device=DEV)
    w = torch.empty((T, k), dtype=torch.float32, device=DEV)
    sc = torch.full((T,), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.zeros(moe.moe_route_workspace_bytes(T, E, H), dtype=torch.uint8, device=DEV)
    moe.moe_route(to_dev(x), None, to_dev(W), synth.F32, E, None, k, oracle.SOFTMAX, True, ids, w, None, ws,
                  shared_gate=to_dev(g), shared_scale=sc)
    torch.cuda.synchronize()
    assert np.allclose(sc.cpu().numpy(), want, rtol=1e-6, atol=0)


def test_sum_partials_adds_in_rank_order():
    """moe_sum_partials: y = ((p0 + p1) + p2) + ..., bit for bit the rank-order
    fp32 sum, for an odd length of float4 groups and one rank."""
    for R, n in ((3, 4 * 1001), (1, 64), (8, 4096 * 4)):
        parts = synth.normal(5, R * 7 + n, 1.0, R, n)
        want = parts[0].copy()
        for r in range(1, R):
            want = (want + parts[r]).astype(np.float32)
        y = torch.full((n,), float("nan"), device=DEV)
        moe.moe_sum_partials(to_dev(parts), y)
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy(), want)
