"""CPU oracle for the quantized routed-expert MoE FFN.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs are the only callers.
The product path (the CUDA library and its binding) never imports this
package, and this package never imports the product.

``oracle.c`` holds the integer-dot oracle (plain scalar C, fp64 scale
combines, fp32 wherever a float decides an integer).  ``brute.py`` holds an
independent fp64 dequantise-then-matmul used to pin it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_oracle.so")
_lock = threading.Lock()
_h = None

F32, Q8_0, Q4_K, Q2_K, MXFP4, Q6_K, Q3_K = 0, 1, 2, 3, 4, 5, 6
SOFTMAX, SIGMOID = 0, 1
_P = ctypes.c_void_p


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "oracle.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                           "-o", tmp, src, "-lm"])
    os.replace(tmp, _SO)
    return _SO


class _Pool(ctypes.Structure):
    _fields_ = [("qtype", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int), ("E", ctypes.c_int),
                ("gate", _P), ("up", _P), ("down", _P), ("bg", _P), ("bu", _P), ("bd", _P),
                ("owned", _P)]


def _lib():
    global _h
    with _lock:
        if _h is None:
            build()
            L = ctypes.CDLL(_SO)
            i, f, d = ctypes.c_int, ctypes.c_float, ctypes.c_double
            L.oracle_f16.restype = f
            L.oracle_f16.argtypes = [ctypes.c_uint16]
            L.oracle_quantize.restype = i
            L.oracle_quantize.argtypes = [_P, i, i, _P, _P, _P]
            L.oracle_router_f32.restype = i
            L.oracle_router_f32.argtypes = [_P, i, i, _P, i, _P, _P]
            L.oracle_router_q8_0.restype = i
            L.oracle_router_q8_0.argtypes = [_P, i, i, _P, _P, i, i, _P, _P]
            L.oracle_router_f64.restype = i
            L.oracle_router_f64.argtypes = [_P, i, i, _P, i, _P, _P]
            L.oracle_topk.restype = i
            L.oracle_topk.argtypes = [_P, i, i, i, i, i, _P, _P]
            L.oracle_row_isums.restype = i
            L.oracle_row_isums.argtypes = [i, _P, i, _P, _P]
            L.oracle_row_dot.restype = d
            L.oracle_row_dot.argtypes = [i, _P, i, _P, _P, _P, i]
            L.oracle_dequant_row.restype = i
            L.oracle_dequant_row.argtypes = [i, _P, i, _P]
            L.oracle_expert_ffn.restype = i
            L.oracle_expert_ffn.argtypes = [ctypes.POINTER(_Pool), ctypes.POINTER(_Pool), i, i,
                                            _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]
            _h = L
        return _h


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a):
    return None if a is None else a.ctypes.data


def f16(h: int) -> float:
    return _lib().oracle_f16(h)


def act_block(n: int) -> int:
    return 256 if n % 256 == 0 else 32


def quantize(x: np.ndarray, B: int | None = None):
    """q8 activations of x [T, n]: (d [T, n/B] f32, q [T, n] i8, bsum [T, n/16] i16)."""
    x = _c(np.atleast_2d(x), np.float32)
    T, n = x.shape
    B = B or act_block(n)
    d = np.zeros((T, n // B), np.float32)
    q = np.zeros((T, n), np.int8)
    bs = np.zeros((T, n // 16), np.int16)
    for t in range(T):
        rc = _lib().oracle_quantize(x[t].ctypes.data, n, B, d[t].ctypes.data, q[t].ctypes.data,
                                    bs[t].ctypes.data)
        if rc:
            raise ValueError("oracle_quantize: bad block size")
    return d, q, bs


def router_logits(W, x, qtype=F32, bias=None, xq=None):
    """fp32 router logits [T, E] in the canonical order (Q8_0: needs xq=(d, q, bsum))."""
    x = _c(np.atleast_2d(x), np.float32)
    T, H = x.shape
    E = W.shape[0]
    out = np.zeros((T, E), np.float32)
    b = None if bias is None else _c(bias, np.float32)
    if qtype == F32:
        W = _c(W, np.float32)
        rc = _lib().oracle_router_f32(W.ctypes.data, E, H, x.ctypes.data, T, _ptr(b), out.ctypes.data)
    else:
        if xq is None:
            xq = quantize(x)
        xd, xqq = _c(xq[0], np.float32), _c(xq[1], np.int8)
        W = _c(W, np.uint8)
        B = H // xd.shape[1]
        rc = _lib().oracle_router_q8_0(W.ctypes.data, E, H, xd.ctypes.data, xqq.ctypes.data, B, T,
                                       _ptr(b), out.ctypes.data)
    if rc:
        raise ValueError("router: unsupported shape")
    return out


def router_logits_f64(W, x, bias=None):
    x = _c(np.atleast_2d(x), np.float32)
    W = _c(W, np.float32)
    T, H = x.shape
    E = W.shape[0]
    out = np.zeros((T, E), np.float64)
    b = None if bias is None else _c(bias, np.float32)
    _lib().oracle_router_f64(W.ctypes.data, E, H, x.ctypes.data, T, _ptr(b), out.ctypes.data)
    return out


def topk(logits, k, gating=SOFTMAX, renorm=True):
    logits = _c(np.atleast_2d(logits), np.float32)
    T, E = logits.shape
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    if _lib().oracle_topk(logits.ctypes.data, T, E, k, gating, int(bool(renorm)), ids.ctypes.data,
                          w.ctypes.data):
        raise ValueError("topk: bad k/E")
    return ids, w


def row_isums(qtype, row, cols, xq_row):
    qk = {Q4_K: 256, Q2_K: 256, Q6_K: 256, Q3_K: 256, Q8_0: 32, MXFP4: 32}[qtype]
    nsub = {Q4_K: 8, Q2_K: 16, Q6_K: 16, Q3_K: 16, Q8_0: 1, MXFP4: 1}[qtype]
    out = np.zeros(cols // qk * nsub, np.int32)
    row, xq_row = _c(row, np.uint8), _c(xq_row, np.int8)
    if _lib().oracle_row_isums(qtype, row.ctypes.data, cols, xq_row.ctypes.data, out.ctypes.data):
        raise ValueError("row_isums: bad shape")
    return out


def row_dot(qtype, row, cols, xd, xq, xbs, B):
    row, xd, xq, xbs = _c(row, np.uint8), _c(xd, np.float32), _c(xq, np.int8), _c(xbs, np.int16)
    return _lib().oracle_row_dot(qtype, row.ctypes.data, cols, xd.ctypes.data, xq.ctypes.data,
                                 xbs.ctypes.data, B)


def dequant_row(qtype, row, cols):
    out = np.zeros(cols, np.float64)
    row = _c(row, np.uint8)
    if _lib().oracle_dequant_row(qtype, row.ctypes.data, cols, out.ctypes.data):
        raise ValueError("dequant_row: bad shape")
    return out


def _pool(qtype, H, I, E, gate, up, down, bg=None, bu=None, bd=None, owned=None, keep=None):
    arrs = [_c(gate, np.uint8), _c(up, np.uint8), _c(down, np.uint8),
            None if bg is None else _c(bg, np.float32), None if bu is None else _c(bu, np.float32),
            None if bd is None else _c(bd, np.float32),
            None if owned is None else _c(owned, np.uint8)]
    keep.extend(a for a in arrs if a is not None)
    return _Pool(qtype, H, I, E, *[_ptr(a) for a in arrs])


def expert_ffn(layer, xq, ids, w, owned=None, shared=True, want_h=False, shared_scale=None):
    """y [T, H] (fp64) for q8 activations xq=(d, q, bsum), ids [T, k], w [T, k].

    layer: a ``synth.Layer``.  owned: optional bool[E] ("not mine" slots are
    skipped).  shared: include the shared expert, added last with weight
    shared_scale[t] (fp64 [T]; 1 when None)."""
    cfg = layer.cfg
    T, k = ids.shape
    keep = []
    pool = _pool(cfg.qtype, cfg.H, cfg.I, cfg.E, layer.gate, layer.up, layer.down,
                 layer.bg, layer.bu, layer.bd, owned, keep)
    sp = None
    if shared and cfg.has_shared:
        sp = _pool(cfg.shared_qtype, cfg.H, cfg.shared_I, 1, layer.sgate, layer.sup, layer.sdown,
                   keep=keep)
    xd, xqq, xbs = (_c(a, t) for a, t in zip(xq, (np.float32, np.int8, np.int16)))
    ids = _c(ids, np.int32)
    w = _c(w, np.float64)
    ss = None if shared_scale is None else _c(shared_scale, np.float64)
    y = np.zeros((T, cfg.H), np.float64)
    I = cfg.I
    BI = act_block(I)
    h = np.zeros((T, k, I), np.float32) if want_h else None
    hd = np.zeros((T, k, I // BI), np.float32) if want_h else None
    hq = np.zeros((T, k, I), np.int8) if want_h else None
    hbs = np.zeros((T, k, I // 16), np.int16) if want_h else None
    bad = _lib().oracle_expert_ffn(ctypes.byref(pool), ctypes.byref(sp) if sp is not None else None,
                                   T, k, xd.ctypes.data, xqq.ctypes.data, xbs.ctypes.data,
                                   ids.ctypes.data, w.ctypes.data, _ptr(ss), y.ctypes.data,
                                   _ptr(h), _ptr(hd), _ptr(hq), _ptr(hbs))
    if bad < 0:
        raise ValueError("expert_ffn: unsupported shape")
    out = {"y": y, "bad_ids": bad}
    if want_h:
        out.update(h=h, hd=hd, hq=hq, hbs=hbs)
    return out


def shared_gate(w_gate, x):
    """Per-token shared-expert weight sigma(w . x) for the f32 gate vector
    w_gate [H] (READING in oracle.c: the shared-expert gate tensor of the
    pulsar README's qwen35moe notes).  The logit is a one-row router GEMV in
    the router's fixed summation order (fp32, ``router_logits``); the sigmoid
    is taken in fp64.  Returns (logit fp32 [T], weight fp64 [T])."""
    l = router_logits(np.asarray(w_gate, np.float32).reshape(1, -1), x)[:, 0]
    with np.errstate(over="ignore"):   # exp(-l) = inf for a very negative logit: weight 0
        return l, 1.0 / (1.0 + np.exp(-l.astype(np.float64)))


def layer_forward(layer, owned=None, shared=True, want_h=False):
    """The whole hot path for one synth.Layer: quantise, route, top-k, expert FFN."""
    cfg = layer.cfg
    xq = quantize(layer.x)
    logits = router_logits(layer.router, layer.x, cfg.router_qtype, layer.router_bias, xq=xq)
    ids, w = topk(logits, cfg.k, SIGMOID if cfg.gating == "sigmoid" else SOFTMAX, cfg.renorm)
    sg = getattr(layer, "shexp_gate", None)
    sg_l, sg_w = shared_gate(sg, layer.x) if (sg is not None and shared and cfg.has_shared) else (None, None)
    res = expert_ffn(layer, xq, ids, w, owned=owned, shared=shared, want_h=want_h, shared_scale=sg_w)
    res.update(xq=xq, logits=logits, ids=ids, w=w, shared_logit=sg_l, shared_scale=sg_w)
    return res
