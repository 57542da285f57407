"""Pins for the CPU oracle against the block definitions, closed forms,
invariants and fp64 brute force (no GPU).

Every check here is chosen so that a plausible slip in the oracle (a dropped
term, a wrong nibble or sub-block index, a transposed operand, a wrong scale
bias, truncation instead of rounding) fails at least one of them.
"""
import json
import os
import struct

import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle
import synth
from oracle import brute

GOLD = os.path.join(os.path.dirname(__file__), "golden", "blocks.json")


# ------------------------------------------------------------- helpers

def f16_bytes(v):
    return np.array([v], np.float16).view(np.uint8).tolist()


def pack_q4k(d, dmin, sc, m, q):
    s = [0] * 12
    for j in range(4):
        s[j] = sc[j] & 63
        s[j + 4] = m[j] & 63
    for j in range(4, 8):
        s[j + 4] = (sc[j] & 15) | ((m[j] & 15) << 4)
        s[j - 4] |= (sc[j] >> 4) << 6
        s[j] |= (m[j] >> 4) << 6
    qs = [0] * 128
    for g in range(4):
        for l in range(32):
            qs[32 * g + l] = q[64 * g + l] | (q[64 * g + 32 + l] << 4)
    return np.array(f16_bytes(d) + f16_bytes(dmin) + s + qs, np.uint8)


def pack_q2k(d, dmin, sc, m, q):
    s = [(sc[j] & 15) | ((m[j] & 15) << 4) for j in range(16)]
    qs = [0] * 64
    for n in range(2):
        for sh in range(4):
            for l in range(32):
                qs[32 * n + l] |= q[128 * n + 32 * sh + l] << (2 * sh)
    return np.array(s + qs + f16_bytes(d) + f16_bytes(dmin), np.uint8)


def pack_q8_0(d, q):
    return np.array(f16_bytes(d) + [int(v) & 255 for v in q], np.uint8)


def pack_mxfp4(e, codes):
    return np.array([e] + [codes[j] | (codes[j + 16] << 4) for j in range(16)], np.uint8)


def pack_q6k(d, sc, c):
    """c: stored 6-bit codes (value c - 32) in element order; sc: 16 int8 scales."""
    ql, qh = [0] * 128, [0] * 64
    for i, v in enumerate(c):
        half, quarter, lane = divmod(i, 128)[0], (i % 128) // 32, i % 32
        byte = 64 * half + 32 * (quarter % 2) + lane
        ql[byte] |= (v & 15) << (4 * (quarter // 2))
        qh[32 * half + lane] |= (v >> 4) << (2 * quarter)
    return np.array(ql + qh + [v & 255 for v in sc] + f16_bytes(d), np.uint8)


def pack_q3k(d, s6, q):
    """q: signed 3-bit codes in [-4, 3] in element order; s6: 16 stored 6-bit scales."""
    hm, qs, sc = [0] * 32, [0] * 64, [0] * 12
    for i, v in enumerate(q):
        half, quarter, lane = i // 128, (i % 128) // 32, i % 32
        qs[32 * half + lane] |= ((v + 4) % 4) << (2 * quarter)
        if v >= 0:
            hm[lane] |= 1 << (4 * half + quarter)
    for j, v in enumerate(s6):
        sc[j % 8] |= (v & 15) << (4 * (j // 8))
        sc[8 + j % 4] |= (v >> 4) << (2 * (j // 4))
    return np.array(hm + qs + sc + f16_bytes(d), np.uint8)


E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def golden_cases():
    with open(GOLD) as f:
        return json.load(f)["cases"]


def build_golden(case):
    qt = case["qtype"]
    if qt == "q4_K":
        q = [i % 16 for i in range(256)]
        blk = pack_q4k(case["d"], case["dmin"], case["sc"], case["m"], q)
        vals = [case["d"] * case["sc"][i // 32] * q[i] - case["dmin"] * case["m"][i // 32] for i in range(256)]
        xq = np.ones(256, np.int8)
        return oracle.Q4_K, blk, 256, vals, xq
    if qt == "q2_K":
        q = [i % 4 for i in range(256)]
        blk = pack_q2k(case["d"], case["dmin"], case["sc"], case["m"], q)
        vals = [case["d"] * case["sc"][i // 16] * q[i] - case["dmin"] * case["m"][i // 16] for i in range(256)]
        return oracle.Q2_K, blk, 256, vals, np.full(256, 2, np.int8)
    if qt == "q8_0":
        q = [i - 16 for i in range(32)]
        blk = pack_q8_0(case["d"], q)
        return oracle.Q8_0, blk, 32, [case["d"] * v for v in q], np.full(32, 3, np.int8)
    if qt == "mxfp4":
        codes = [i % 16 for i in range(32)]
        blk = pack_mxfp4(case["e"], codes)
        scale = 2.0 ** (case["e"] - 127)
        vals = [scale * (-E2M1[c & 7] if c & 8 else E2M1[c & 7]) for c in codes]
        return oracle.MXFP4, blk, 32, vals, np.arange(1, 33).astype(np.int8)
    if qt == "q6_K":
        c = [i // 4 for i in range(256)]
        blk = pack_q6k(case["d"], case["sc"], c)
        vals = [case["d"] * case["sc"][i // 16] * (c[i] - 32) for i in range(256)]
        return oracle.Q6_K, blk, 256, vals, np.ones(256, np.int8)
    if qt == "q3_K":
        q = [(7 * i + i // 128) % 8 - 4 for i in range(256)]
        blk = pack_q3k(case["d"], case["s6"], q)
        vals = [case["d"] * (case["s6"][i // 16] - 32) * q[i] for i in range(256)]
        return oracle.Q3_K, blk, 256, vals, np.ones(256, np.int8)
    raise ValueError(qt)


# ------------------------------------------------------------- formats

def test_f16_decode_every_code():
    codes = np.arange(65536, dtype=np.uint16)
    ref = codes.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16(int(c)) for c in codes], np.float32)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.all(np.isnan(got[np.isnan(ref)]))


@pytest.mark.parametrize("case", golden_cases(), ids=lambda c: c["name"])
def test_golden_blocks(case):
    qt, blk, n, vals, xq = build_golden(case)
    assert np.array_equal(oracle.dequant_row(qt, blk, n), np.array(vals))
    assert np.array_equal(brute.dequant(qt, blk[None], n)[0], np.array(vals))
    assert oracle.row_isums(qt, blk, n, xq).tolist() == case["isums"]
    B = case["x_block"]
    xd = np.full(n // B if n >= B else 1, case["x_d"], np.float32)
    bsum = xq.astype(np.int64).reshape(-1, 16).sum(1).astype(np.int16)
    assert oracle.row_dot(qt, blk, n, xd, xq, bsum, B) == case["dot"]


def test_closed_form_zero_codes_give_minus_dmin_m():
    sc = [5, 9, 63, 0, 17, 40, 1, 33]
    m = [63, 0, 7, 21, 50, 13, 62, 4]
    blk = pack_q4k(0.125, 0.0625, sc, m, [0] * 256)
    got = oracle.dequant_row(oracle.Q4_K, blk, 256)
    assert np.array_equal(got, np.repeat([-0.0625 * v for v in m], 32))
    sc2, m2 = list(range(16)), [(3 * j) % 16 for j in range(16)]
    blk2 = pack_q2k(0.5, 0.25, sc2, m2, [0] * 256)
    got2 = oracle.dequant_row(oracle.Q2_K, blk2, 256)
    assert np.array_equal(got2, np.repeat([-0.25 * v for v in m2], 16))
    # Q8_0 and MXFP4: d*0 = 0 exactly
    assert np.array_equal(oracle.dequant_row(oracle.Q8_0, pack_q8_0(0.75, [0] * 32), 32), np.zeros(32))
    assert np.array_equal(oracle.dequant_row(oracle.MXFP4, pack_mxfp4(140, [0] * 32), 32), np.zeros(32))


@pytest.mark.parametrize("pos", [0, 31, 32, 100, 255])
def test_closed_form_single_code(pos):
    sc = [3, 7, 11, 13, 19, 23, 29, 31]
    q = [0] * 256
    q[pos] = 9
    blk = pack_q4k(0.25, 0.0, sc, [0] * 8, q)
    got = oracle.dequant_row(oracle.Q4_K, blk, 256)
    want = np.zeros(256)
    want[pos] = 0.25 * sc[pos // 32] * 9
    assert np.array_equal(got, want)
    q2 = [0] * 256
    q2[pos] = 3
    sc2 = [j % 15 + 1 for j in range(16)]
    blk2 = pack_q2k(0.5, 0.0, sc2, [0] * 16, q2)
    want2 = np.zeros(256)
    want2[pos] = 0.5 * sc2[pos // 16] * 3
    assert np.array_equal(oracle.dequant_row(oracle.Q2_K, blk2, 256), want2)


# every (half, quarter, lane-group) field of the 256-element K-quant layouts
POSITIONS = [0, 15, 16, 31, 32, 47, 63, 64, 95, 96, 127, 128, 159, 160, 191, 200, 224, 255]


@pytest.mark.parametrize("pos", POSITIONS)
def test_closed_form_single_code_q6k_q3k(pos):
    """one non-zero code among zero values lands on exactly its element"""
    sc = [(-1) ** j * (j + 2) for j in range(16)]
    c = [32] * 256                      # stored 32 is the value 0
    c[pos] = 5                          # value -27
    want = np.zeros(256)
    want[pos] = 0.5 * sc[pos // 16] * (5 - 32)
    assert np.array_equal(oracle.dequant_row(oracle.Q6_K, pack_q6k(0.5, sc, c), 256), want)
    c[pos] = 63                         # value 31: both high bits set
    want[pos] = 0.5 * sc[pos // 16] * 31
    assert np.array_equal(oracle.dequant_row(oracle.Q6_K, pack_q6k(0.5, sc, c), 256), want)
    s6 = [(5 * j + 1) % 64 for j in range(16)]
    for v in (-4, -1, 1, 3):
        q = [0] * 256
        q[pos] = v
        want = np.zeros(256)
        want[pos] = 0.25 * (s6[pos // 16] - 32) * v
        assert np.array_equal(oracle.dequant_row(oracle.Q3_K, pack_q3k(0.25, s6, q), 256), want)


def test_q6k_q3k_extreme_codes_and_scales():
    """int8 scale -128 and 127, 6-bit scale 0 (= -32) and 63 (= 31), codes at both ends"""
    sc = [-128, 127] * 8
    c = [0 if (i // 16) % 2 == 0 else 63 for i in range(256)]
    got = oracle.dequant_row(oracle.Q6_K, pack_q6k(0.125, sc, c), 256)
    want = np.where((np.arange(256) // 16) % 2 == 0, 0.125 * -128 * -32, 0.125 * 127 * 31)
    assert np.array_equal(got, want)
    s6 = [0, 63] * 8
    q = [-4 if (i // 16) % 2 == 0 else 3 for i in range(256)]
    got = oracle.dequant_row(oracle.Q3_K, pack_q3k(2.0, s6, q), 256)
    want = np.where((np.arange(256) // 16) % 2 == 0, 2.0 * -32 * -4, 2.0 * 31 * 3)
    assert np.array_equal(got, want)


def test_q6k_q3k_zero_scale_or_code_give_zero():
    rng = np.random.default_rng(11)
    c = rng.integers(0, 64, 256).tolist()
    assert not oracle.dequant_row(oracle.Q6_K, pack_q6k(0.5, [0] * 16, c), 256).any()
    q = rng.integers(-4, 4, 256).tolist()
    assert not oracle.dequant_row(oracle.Q3_K, pack_q3k(0.5, [32] * 16, q), 256).any()
    assert not oracle.dequant_row(oracle.Q3_K, pack_q3k(0.5, list(range(16)), [0] * 256), 256).any()


def test_mxfp4_lattice_table():
    for e in (120, 127, 131):
        blk = pack_mxfp4(e, [c % 16 for c in range(32)])
        got = oracle.dequant_row(oracle.MXFP4, blk, 32)
        want = [2.0 ** (e - 127) * (-E2M1[c & 7] if c & 8 else E2M1[c & 7]) for c in [i % 16 for i in range(32)]]
        assert np.array_equal(got, np.array(want))


@pytest.mark.parametrize("qt,rms_bound", [(synth.Q8_0, 0.01), (synth.Q4_K, 0.12), (synth.Q2_K, 0.45),
                                          (synth.MXFP4, 0.2), (synth.Q6_K, 0.03), (synth.Q3_K, 0.25)])
def test_encoder_roundtrip(qt, rms_bound):
    """generator encoder -> oracle decoder reproduces the fp32 weights to quantisation noise"""
    w = synth.normal(7, 123, 0.02, 64, 512)
    blocks = synth.encode(qt, w)
    deq = np.stack([oracle.dequant_row(qt, blocks[r], 512) for r in range(64)])
    assert np.array_equal(deq, brute.dequant(qt, blocks, 512))
    rel = np.sqrt(np.mean((deq - w) ** 2)) / np.sqrt(np.mean(w.astype(np.float64) ** 2))
    assert rel < rms_bound, rel
    # elementwise bound: no element further than one (sub-)block step from its source
    if qt == synth.Q8_0:
        d = np.abs(w).reshape(64, -1, 32).max(-1, keepdims=True) / 127
        assert np.all(np.abs(deq - w).reshape(64, -1, 32) <= 0.5 * d * 1.01 + 1e-12)
    if qt in (synth.Q6_K, synth.Q3_K):
        # the largest |w| of each 16-sub-block comes back within a bounded number
        # of steps (step = amax/31 for Q6_K, amax/4 for Q3_K): half a step of
        # rounding plus the rounding of the sub-block scale; a 3-bit code tops
        # out at +3, so a positive Q3_K maximum can lose one whole step more
        top, steps = (31, 0.75) if qt == synth.Q6_K else (4, 1.5)
        amax = np.abs(w.astype(np.float64)).reshape(64, -1, 16).max(-1)
        dmax = np.abs(deq).reshape(64, -1, 16).max(-1)
        assert np.all(np.abs(dmax - amax) <= steps * amax / top + 1e-12)


# -------------------------------------------------------------- int dots

@pytest.mark.parametrize("qt", [synth.Q8_0, synth.Q4_K, synth.Q2_K, synth.MXFP4, synth.Q6_K, synth.Q3_K])
def test_row_isums_equal_integer_dot_of_codes(qt):
    """random code bytes with unit scales: values are the integer codes themselves"""
    rng = np.random.default_rng(3)
    n = 512
    if qt == synth.Q4_K:
        blocks = [pack_q4k(1.0, 0.0, [1] * 8, [0] * 8, rng.integers(0, 16, 256).tolist()) for _ in range(2)]
        sub = 32
    elif qt == synth.Q2_K:
        blocks = [pack_q2k(1.0, 0.0, [1] * 16, [0] * 16, rng.integers(0, 4, 256).tolist()) for _ in range(2)]
        sub = 16
    elif qt == synth.Q6_K:
        blocks = [pack_q6k(1.0, [1] * 16, rng.integers(0, 64, 256).tolist()) for _ in range(2)]
        sub = 16
    elif qt == synth.Q3_K:
        blocks = [pack_q3k(1.0, [33] * 16, rng.integers(-4, 4, 256).tolist()) for _ in range(2)]
        sub = 16
    elif qt == synth.Q8_0:
        blocks = [pack_q8_0(1.0, rng.integers(-128, 128, 32).tolist()) for _ in range(16)]
        sub = 32
    else:
        blocks = [pack_mxfp4(128, rng.integers(0, 16, 32).tolist()) for _ in range(16)]
        sub = 32
    row = np.concatenate(blocks)
    codes = brute.dequant(qt, row[None], n)[0]
    if qt == synth.MXFP4:
        codes = codes * 1.0  # e=128 -> value 2*E2M1 = the integer lattice
    xq = rng.integers(-127, 128, n).astype(np.int8)
    want = (codes * xq).reshape(-1, sub).sum(1).astype(np.int64)
    got = oracle.row_isums(qt, row, n, xq)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("qt", [synth.Q8_0, synth.Q4_K, synth.Q2_K, synth.MXFP4, synth.Q6_K, synth.Q3_K])
@pytest.mark.parametrize("B", [256, 32])
def test_row_dot_matches_fp64_dequant_matmul(qt, B):
    if qt in (synth.Q4_K, synth.Q2_K, synth.Q6_K, synth.Q3_K) and B == 32:
        pytest.skip("K-quants are paired with 256-blocks of activations")
    H = 1024
    W = synth.matrix(qt, 1, 77, 0.02, 8, H)
    x = synth.normal(1, 78, 1.0, 1, H)
    xd, xq, xbs = oracle.quantize(x, B)
    xv = brute.act_values(xd, xq)[0]
    dense = brute.dequant(qt, W, H)
    for r in range(8):
        got = oracle.row_dot(qt, W[r], H, xd[0], xq[0], xbs[0], B)
        want = float(dense[r] @ xv)
        scale = float(np.abs(dense[r]) @ np.abs(xv))
        assert abs(got - want) <= 1e-13 * scale, (r, got, want)


# -------------------------------------------------------------- quantiser

@pytest.mark.parametrize("B", [256, 32])
@pytest.mark.parametrize("sigma", [1.0, 1e-3, 3e4])
def test_quantize_invariants(B, sigma):
    x = synth.normal(5, 9, sigma, 4, 2048)
    d, q, bs = oracle.quantize(x, B)
    qb = q.reshape(4, -1, B).astype(np.int64)
    assert np.all(np.abs(qb) <= 127)
    assert np.all(np.abs(qb).max(-1) == 127)
    amax = np.abs(x).reshape(4, -1, B).max(-1)
    assert np.array_equal(d, (amax / np.float32(127)).astype(np.float32))
    err = np.abs(x.reshape(4, -1, B).astype(np.float64) - d[..., None].astype(np.float64) * qb)
    assert np.all(err <= 0.5 * d[..., None] * (1 + 1e-5))
    assert np.array_equal(bs.astype(np.int64), q.astype(np.int64).reshape(4, -1, 16).sum(-1))
    d2, q2, _ = oracle.quantize(-x, B)
    assert np.array_equal(d2, d) and np.array_equal(q2, -q)


def test_quantize_special_cases():
    x = np.zeros((1, 512), np.float32)
    x[0, 300] = -2.5
    d, q, bs = oracle.quantize(x, 256)
    assert d[0, 0] == 0 and not q[0, :256].any()
    assert q[0, 300] == -127 and np.count_nonzero(q[0]) == 1
    assert d[0, 1] == np.float32(2.5) / np.float32(127)
    # ties go to the even code: amax = 127 makes the scale exactly 1
    y = np.zeros((1, 256), np.float32)
    y[0, :6] = [127.0, 2.5, 3.5, -2.5, 0.5, -1.5]
    _, qy, _ = oracle.quantize(y, 256)
    assert qy[0, :6].tolist() == [127, 2, 4, -2, 0, -2]


# ------------------------------------------------------------------ router

@pytest.mark.parametrize("H", [512, 2048, 2880, 4096, 7168])
def test_router_canonical_order_exact_on_integers(H):
    """integer-valued inputs: every fp32 step is exact, so the canonical sum
    must equal the exact integer dot - any dropped or doubled element fails"""
    rng = np.random.default_rng(H)
    W = rng.integers(-8, 9, (5, H)).astype(np.float32)
    x = rng.integers(-8, 9, (3, H)).astype(np.float32)
    got = oracle.router_logits(W, x)
    want = (x.astype(np.int64) @ W.T.astype(np.int64)).astype(np.float32)
    assert np.array_equal(got, want)
    bias = rng.integers(-4, 5, 5).astype(np.float32)
    assert np.array_equal(oracle.router_logits(W, x, bias=bias), want + bias)


@pytest.mark.parametrize("H", [512, 2880, 4096])
def test_router_fp32_within_rounding_of_fp64(H):
    W = synth.normal(2, 5, 0.02, 64, H)
    x = synth.normal(2, 6, 1.0, 2, H)
    got = oracle.router_logits(W, x).astype(np.float64)
    want = oracle.router_logits_f64(W, x)
    bound = (H + 40) * 2.0 ** -24 * (np.abs(x.astype(np.float64)) @ np.abs(W.T.astype(np.float64)))
    assert np.all(np.abs(got - want) <= bound)


def test_router_q8_0_exact_and_close():
    H = 7168
    rng = np.random.default_rng(11)
    # unit scales, small codes: exact integer arithmetic end to end
    rows = []
    for _ in range(3):
        rows.append(np.concatenate([pack_q8_0(1.0, rng.integers(-5, 6, 32).tolist()) for _ in range(H // 32)]))
    W = np.stack(rows)
    xq = rng.integers(-5, 6, (2, H)).astype(np.int8)
    xd = np.ones((2, H // 256), np.float32)
    got = oracle.router_logits(W, np.zeros((2, H), np.float32), oracle.Q8_0, xq=(xd, xq, None))
    codes = brute.dequant(oracle.Q8_0, W, H)
    assert np.array_equal(got, (xq.astype(np.float64) @ codes.T).astype(np.float32))
    # realistic scales: within fp32 rounding of the fp64 dequantised dot
    Wr = synth.matrix(synth.Q8_0, 3, 9, 0.02, 16, H)
    x = synth.normal(3, 10, 1.0, 2, H)
    xqr = oracle.quantize(x)
    got = oracle.router_logits(Wr, x, oracle.Q8_0, xq=xqr).astype(np.float64)
    dense = brute.dequant(oracle.Q8_0, Wr, H)
    xv = brute.act_values(xqr[0], xqr[1])
    want = xv @ dense.T
    assert np.all(np.abs(got - want) <= 1e-5 * (np.abs(xv) @ np.abs(dense.T)))


def test_topk_matches_stable_sort_with_ties():
    rng = np.random.default_rng(4)
    logits = rng.integers(-3, 4, (50, 32)).astype(np.float32)    # many exact ties
    ids, _ = oracle.topk(logits, 6)
    want = np.argsort(-logits, axis=1, kind="stable")[:, :6]
    assert np.array_equal(ids, want)


def test_topk_weights():
    logits = synth.normal(9, 1, 1.5, 20, 64)
    ids, w = oracle.topk(logits, 64, oracle.SOFTMAX, renorm=False)
    full = softmax(logits.astype(np.float64), axis=1)
    assert np.allclose(w, np.take_along_axis(full, ids, 1), rtol=1e-13, atol=0)
    ids, w = oracle.topk(logits, 8, oracle.SOFTMAX, renorm=True)
    assert np.allclose(w.sum(1), 1.0, atol=1e-14)
    sel = np.take_along_axis(logits.astype(np.float64), ids, 1)
    assert np.allclose(w, softmax(sel, axis=1), rtol=1e-13)
    assert np.all(np.diff(w, axis=1) <= 0)
    ids, w = oracle.topk(logits, 8, oracle.SIGMOID, renorm=True)
    s = expit(np.take_along_axis(logits.astype(np.float64), ids, 1))
    assert np.allclose(w, s / s.sum(1, keepdims=True), rtol=1e-13)
    ids, w = oracle.topk(logits, 8, oracle.SIGMOID, renorm=False)
    assert np.allclose(w, expit(np.take_along_axis(logits.astype(np.float64), ids, 1)), rtol=1e-13)


def test_topk_permutation():
    logits = synth.normal(9, 2, 1.0, 10, 128)
    perm = np.random.default_rng(1).permutation(128)
    ids, w = oracle.topk(logits, 8)
    ids_p, w_p = oracle.topk(logits[:, perm], 8)
    assert np.array_equal(perm[ids_p], ids)
    assert np.array_equal(w_p, w)


# --------------------------------------------------------------------- FFN

SMALL = {
    "q8_0": synth.shrink(synth.CONFIGS["tiny"], E=6, k=2),
    "q4_K+shared": synth.shrink(synth.CONFIGS["a3b"], H=512, I=256, E=8, k=3, shared_I=256),
    "mxfp4+bias": synth.shrink(synth.CONFIGS["oss20b"], H=320, I=288, E=5, k=2),
    "q2_K+q8_0shared": synth.shrink(synth.CONFIGS["wide"], H=512, I=256, E=8, k=3, shared_I=256),
    "q6_K+shared": synth.shrink(synth.CONFIGS["a3b"], H=512, I=256, E=8, k=3, shared_I=256,
                                qtype=synth.Q6_K, shared_qtype=synth.Q6_K),
    "q3_K+q8_0shared": synth.shrink(synth.CONFIGS["wide"], H=512, I=256, E=8, k=3, shared_I=256,
                                    qtype=synth.Q3_K),
    # x in 256-blocks, h in 32-blocks: a slip that used H's block for h fails here
    "q8_0 H512/I288": synth.shrink(synth.CONFIGS["tiny"], H=512, I=288, E=6, k=2),
}


def np_quantize(x):
    """The activation rule restated in numpy fp32 (IEEE division, round half
    to even): per block of B (256, else 32), d = amax/127 and
    q = rint(x * (127/amax)); zero blocks give d = 0, q = 0."""
    x = np.asarray(x, np.float32)
    n = x.shape[-1]
    B = 256 if n % 256 == 0 else 32
    xb = x.reshape(-1, n // B, B)
    amax = np.abs(xb).max(axis=-1)
    with np.errstate(divide="ignore", invalid="ignore"):
        d = np.where(amax > 0, amax / np.float32(127), np.float32(0)).astype(np.float32)
        isc = np.where(amax > 0, np.float32(127) / amax, np.float32(0)).astype(np.float32)
    q = np.clip(np.rint((xb * isc[..., None]).astype(np.float32)), -127, 127).astype(np.int8)
    return d.reshape(x.shape[:-1] + (n // B,)), q.reshape(x.shape)


@pytest.mark.parametrize("name", list(SMALL))
def test_ffn_matches_fp64_brute_force(name):
    cfg = SMALL[name]
    L = synth.make_layer(cfg, 0, T=3)
    res = oracle.layer_forward(L, want_h=True)
    xq = res["xq"]
    xv = brute.act_values(xq[0], xq[1])
    T, k = res["ids"].shape
    # g, u and h against dense fp64 products; h is stored in fp32
    for t in range(T):
        for s in range(k):
            g, u = brute.expert_gu(L, int(res["ids"][t, s]), xv[t:t + 1])
            h64 = (brute.silu(g) * u)[0]
            h32 = res["h"][t, s].astype(np.float64)
            assert np.all(np.abs(h32 - h64) <= 2.0 ** -23 * np.abs(h64) + 1e-30)
            # the routed h goes into the down projection requantised with the
            # activation rule at I's own block size
            d_np, q_np = np_quantize(res["h"][t, s])
            assert np.array_equal(np.asarray(res["hd"][t, s], np.float32).reshape(-1), d_np.reshape(-1))
            assert np.array_equal(np.asarray(res["hq"][t, s]).reshape(-1), q_np.reshape(-1))
    hq_sh = None
    if cfg.has_shared:
        g, u = brute.expert_gu(L, 0, xv, shared=True)
        hs = (brute.silu(g) * u).astype(np.float32)
        hq_sh = oracle.quantize(hs)[:2]
    want = brute.ffn_given_hq(L, xq, res["ids"], res["w"], (res["hd"], res["hq"]), hq_sh)
    scale = np.abs(want).max()
    assert np.max(np.abs(res["y"] - want)) <= 1e-12 * scale


def test_ffn_k1_is_a_single_dense_quantised_ffn():
    cfg = synth.shrink(synth.CONFIGS["tiny"], E=4, k=1)
    L = synth.make_layer(cfg, 0, T=2)
    xq = oracle.quantize(L.x)
    ids = np.array([[2], [2]], np.int32)
    res = oracle.expert_ffn(L, xq, ids, np.ones((2, 1)), want_h=True)
    xv = brute.act_values(xq[0], xq[1])
    g, u = brute.expert_gu(L, 2, xv)
    hq = oracle.quantize((brute.silu(g) * u).astype(np.float32))
    o = brute.expert_o(L, 2, brute.act_values(hq[0], hq[1]))
    assert np.allclose(res["y"], o, rtol=0, atol=1e-12 * np.abs(o).max())


def test_ffn_expert_permutation_leaves_y_unchanged():
    cfg = SMALL["q4_K+shared"]
    L = synth.make_layer(cfg, 0, T=2)
    base = oracle.layer_forward(L)
    perm = np.random.default_rng(8).permutation(cfg.E)
    Lp = synth.make_layer(cfg, 0, T=2)
    Lp.router, Lp.gate, Lp.up, Lp.down = L.router[perm], L.gate[perm], L.up[perm], L.down[perm]
    res = oracle.layer_forward(Lp)
    inv = np.argsort(perm)
    assert np.array_equal(perm[res["ids"]], base["ids"])
    assert np.array_equal(res["y"], base["y"])
    assert np.array_equal(inv[base["ids"]], res["ids"])


def test_ffn_ownership_partition_sums_to_full():
    cfg = SMALL["q2_K+q8_0shared"]
    L = synth.make_layer(cfg, 0, T=3)
    full = oracle.layer_forward(L)
    own0 = np.arange(cfg.E) % 2 == 0
    y0 = oracle.expert_ffn(L, full["xq"], full["ids"], full["w"], owned=own0, shared=True)["y"]
    y1 = oracle.expert_ffn(L, full["xq"], full["ids"], full["w"], owned=~own0, shared=False)["y"]
    assert np.allclose(y0 + y1, full["y"], rtol=0, atol=1e-12 * np.abs(full["y"]).max())


def test_ffn_skips_out_of_range_ids():
    cfg = SMALL["q8_0"]
    L = synth.make_layer(cfg, 0, T=1)
    xq = oracle.quantize(L.x)
    ok = oracle.expert_ffn(L, xq, np.array([[1, 3]], np.int32), np.array([[0.25, 0.75]]))
    bad = oracle.expert_ffn(L, xq, np.array([[1, 99]], np.int32), np.array([[0.25, 0.75]]))
    only1 = oracle.expert_ffn(L, xq, np.array([[1]], np.int32), np.array([[0.25]]))
    assert bad["bad_ids"] == 1 and ok["bad_ids"] == 0
    assert np.array_equal(bad["y"], only1["y"])


def test_synth_is_deterministic():
    a = synth.matrix(synth.Q4_K, 0, 42, 0.02, 33, 512)
    b = synth.matrix(synth.Q4_K, 0, 42, 0.02, 33, 512)
    c = synth.matrix(synth.Q4_K, 1, 42, 0.02, 33, 512)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    x = synth.normal(0, 1, 1.0, 1, 100000)
    assert abs(x.mean()) < 0.02 and abs(x.std() - 1) < 0.02


def test_zipf_router_bias_skews_selection():
    """The 16-token batch of the 235B-A22B-style stack adds b_e = -1.1 ln(rank_e)
    to the logits, ranks a seeded permutation of 1..E per layer: tokens then
    share experts far more often than with the plain router."""
    cfg = synth.CONFIGS["a22b"]
    b0, b0_again, b1 = synth.zipf_bias(cfg, 0), synth.zipf_bias(cfg, 0), synth.zipf_bias(cfg, 1)
    expect = np.sort((-1.1 * np.log(np.arange(1, cfg.E + 1, dtype=np.float64))).astype(np.float32))
    assert np.array_equal(np.sort(b0), expect)
    assert np.array_equal(b0, b0_again) and not np.array_equal(b0, b1)
    small = synth.shrink(cfg, H=512)
    L = synth.make_layer(small, 0, T=16, zipf=False, with_experts=False)
    W = np.asarray(L.router, np.float32).reshape(small.E, small.H)
    plain = oracle.router_logits(W, L.x)
    skewed = oracle.router_logits(W, L.x, bias=synth.zipf_bias(small, 0))
    u_plain = len(np.unique(oracle.topk(plain, small.k)[0]))
    u_skewed = len(np.unique(oracle.topk(skewed, small.k)[0]))
    assert u_skewed < u_plain, (u_skewed, u_plain)


# ------------------------------------------------------- shared-expert gate
# READING (oracle.c, oracle_expert_ffn): the shared expert's output is scaled
# per token by sigma(w . x), w the f32 gate vector; without it the weight is 1.

GATED = synth.shrink(synth.CONFIGS["a3b"], H=512, I=256, E=8, k=3, shared_I=256, shared_gate=True)


def _parts(L):
    """y with the shared expert left out, and with it at weight 1"""
    xq = oracle.quantize(L.x)
    logits = oracle.router_logits(L.router, L.x)
    ids, w = oracle.topk(logits, L.cfg.k)
    routed = oracle.expert_ffn(L, xq, ids, w, shared=False)["y"]
    full = oracle.expert_ffn(L, xq, ids, w, shared=True)["y"]
    return routed, full


def test_shared_gate_zero_vector_halves_the_shared_expert():
    L = synth.make_layer(GATED, 0, T=3)
    L.shexp_gate = np.zeros(GATED.H, np.float32)           # sigma(0) = 1/2 exactly
    routed, full = _parts(L)
    res = oracle.layer_forward(L)
    assert np.all(res["shared_scale"] == 0.5)
    want = routed + 0.5 * (full - routed)
    assert np.max(np.abs(res["y"] - want)) <= 1e-12 * np.abs(want).max()


def test_shared_gate_saturates_to_one_and_zero():
    L = synth.make_layer(GATED, 0, T=2)
    routed, full = _parts(L)
    # a gate along token 0's own hidden state, scaled up: logit +huge for it
    L.shexp_gate = (1e4 * L.x[0]).astype(np.float32)
    res = oracle.layer_forward(L)
    assert res["shared_logit"][0] > 1e3 and res["shared_scale"][0] == 1.0
    assert np.array_equal(res["y"][0], full[0])
    L.shexp_gate = (-1e4 * L.x[0]).astype(np.float32)
    res = oracle.layer_forward(L)
    assert res["shared_scale"][0] < 1e-300
    assert np.max(np.abs(res["y"][0] - routed[0])) <= 1e-12 * np.abs(routed[0]).max()


def test_shared_gate_logit_against_fp64_dot_and_per_token_scale():
    L = synth.make_layer(GATED, 1, T=4)
    assert L.shexp_gate is not None and L.shexp_gate.shape == (GATED.H,)
    res = oracle.layer_forward(L)
    w64 = L.shexp_gate.astype(np.float64)
    for t in range(4):
        exact = float(np.dot(w64, L.x[t].astype(np.float64)))
        bound = GATED.H * 2.0 ** -24 * float(np.dot(np.abs(w64), np.abs(L.x[t].astype(np.float64)))) * 2
        assert abs(float(res["shared_logit"][t]) - exact) <= bound
        assert res["shared_scale"][t] == 1.0 / (1.0 + np.exp(-float(res["shared_logit"][t])))
    # y = routed + s_t * (full - routed) token by token
    routed, full = _parts(L)
    want = routed + res["shared_scale"][:, None] * (full - routed)
    assert np.max(np.abs(res["y"] - want)) <= 1e-12 * np.abs(want).max()
