"""Seeded synthetic inputs for the quantized routed-expert MoE FFN.

Input generation only: normal draws from counter-keyed splitmix64 streams and
the GGUF-style weight block encoders live in ``synth.c``.  Nothing here computes
any step of the MoE path; the CUDA library and the CPU oracle both consume
what this module produces, and neither is imported here.

Shapes, value distributions and routing structure follow the five synthetic
workloads of the MoE-layer decode study (pulsar README, model table and
"MoE resolve" passage): weights ~N(0, 0.02^2), expert biases ~N(0, 0.01^2),
hidden states ~N(0, 1), router ~N(0, 0.02^2), and for the 16-token batch of the
235B-A22B-style stack a Zipf(1.1) prior over experts added as a router bias
b_e = -1.1 ln(rank_e) with a seeded random rank permutation per layer.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SO = os.path.join(_HERE, "_synth.so")
_lock = threading.Lock()
_lib_handle = None

# qtype codes: the library's public enum (moe_qtype)
F32, Q8_0, Q4_K, Q2_K, MXFP4, Q6_K, Q3_K = 0, 1, 2, 3, 4, 5, 6
QTYPE_NAMES = {F32: "f32", Q8_0: "q8_0", Q4_K: "q4_K", Q2_K: "q2_K", MXFP4: "mxfp4", Q6_K: "q6_K",
               Q3_K: "q3_K"}
# (elements per block, bytes per block)
BLOCK = {F32: (1, 4), Q8_0: (32, 34), Q4_K: (256, 144), Q2_K: (256, 84), MXFP4: (32, 17),
         Q6_K: (256, 210), Q3_K: (256, 110)}


def build(force: bool = False) -> str:
    """Compile synth.c into _synth.so with gcc (deterministic fp: no contraction)."""
    src = os.path.join(_HERE, "synth.c")
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(src):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                           "-shared", "-pthread", "-o", tmp, src, "-lm"])
    os.replace(tmp, _SO)
    return _SO


def _lib():
    global _lib_handle
    with _lock:
        if _lib_handle is None:
            build()
            lib = ctypes.CDLL(_SO)
            lib.synth_matrix.restype = ctypes.c_int
            lib.synth_matrix.argtypes = [ctypes.c_int, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_float,
                                         ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int,
                                         ctypes.c_int64]
            lib.synth_encode.restype = ctypes.c_int
            lib.synth_encode.argtypes = [ctypes.c_int, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_void_p]
            lib.synth_row_bytes.restype = ctypes.c_int64
            lib.synth_row_bytes.argtypes = [ctypes.c_int, ctypes.c_int64]
            _lib_handle = lib
        return _lib_handle


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def row_bytes(qtype: int, cols: int) -> int:
    rb = _lib().synth_row_bytes(qtype, cols)
    if rb < 0:
        raise ValueError(f"{QTYPE_NAMES.get(qtype, qtype)} cannot hold rows of {cols} elements")
    return int(rb)


def matrix(qtype: int, seed: int, stream: int, sigma: float, rows: int, cols: int, row0: int = 0) -> np.ndarray:
    """rows x cols draws of N(0, sigma^2), encoded as qtype blocks: uint8 [rows, row_bytes]
    (F32: float32 [rows, cols]).  Output row r is row row0 + r of the stream."""
    rb = row_bytes(qtype, cols)
    out = np.empty((rows, rb), dtype=np.uint8)
    rc = _lib().synth_matrix(qtype, seed, stream, sigma, rows, cols, out.ctypes.data, _threads(), row0)
    if rc != 0:
        raise RuntimeError(f"synth_matrix failed ({rc})")
    return out.view(np.float32) if qtype == F32 else out


def encode(qtype: int, w: np.ndarray) -> np.ndarray:
    """Encode an fp32 matrix [rows, cols] into qtype blocks (uint8 [rows, row_bytes])."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    rows, cols = w.shape
    out = np.empty((rows, row_bytes(qtype, cols)), dtype=np.uint8)
    if _lib().synth_encode(qtype, w.ctypes.data, rows, cols, out.ctypes.data) != 0:
        raise ValueError("encode failed")
    return out


def normal(seed: int, stream: int, sigma: float, rows: int, cols: int) -> np.ndarray:
    return matrix(F32, seed, stream, sigma, rows, cols)


# ------------------------------------------------------------------ configs

@dataclass(frozen=True)
class MoEConfig:
    name: str
    cid: int
    H: int
    E: int
    I: int
    k: int
    qtype: int                 # routed expert weights
    gating: str = "softmax"    # "softmax" | "sigmoid"
    renorm: bool = True
    router_qtype: int = F32
    shared_I: int = 0          # 0: no shared expert
    shared_qtype: int = -1
    shared_gate: bool = False  # a sigmoid gate vector on the shared expert (f32 [H])
    biases: bool = False
    layers: int = 1
    tokens: tuple = (1,)
    zipf_tokens: tuple = ()
    note: str = ""

    @property
    def has_shared(self) -> bool:
        return self.shared_I > 0


CONFIGS = {
    "tiny": MoEConfig("tiny", 1, H=512, E=16, I=256, k=2, qtype=Q8_0,
                      note="tiny single MoE layer: H512 E16 I256 top-2 softmax, Q8_0 experts"),
    "a3b": MoEConfig("a3b", 2, H=2048, E=256, I=512, k=8, qtype=Q4_K,
                     shared_I=512, shared_qtype=Q4_K,
                     note="35B-A3B-style layer: H2048 E256 I512 top-8 softmax + shared, Q4_K"),
    "oss20b": MoEConfig("oss20b", 3, H=2880, E=32, I=2880, k=4, qtype=MXFP4, biases=True,
                        layers=24, tokens=(1, 4),
                        note="gpt-oss-20B-style layer: H2880 E32 I2880 top-4 softmax, MXFP4 + biases"),
    "wide": MoEConfig("wide", 4, H=7168, E=256, I=2048, k=8, qtype=Q2_K, gating="sigmoid",
                      router_qtype=Q8_0, shared_I=2048, shared_qtype=Q8_0, layers=8,
                      note="DeepSeek/Kimi-style wide layer: H7168 E256 I2048 top-8 sigmoid + shared, "
                           "Q2_K routed, Q8_0 shared and router"),
    "a22b": MoEConfig("a22b", 5, H=4096, E=128, I=1536, k=8, qtype=Q4_K, layers=48,
                      tokens=(1, 4, 16), zipf_tokens=(16,),
                      note="235B-A22B-style stack: H4096 E128 I1536 top-8 softmax, Q4_K"),
}

# tensor codes inside a stream id
_T_X, _T_ROUTER, _T_GATE, _T_UP, _T_DOWN, _T_BG, _T_BU, _T_BD = 1, 2, 3, 4, 5, 6, 7, 8
_T_SGATE, _T_SUP, _T_SDOWN, _T_SHGATE = 9, 10, 11, 12
SIG_W, SIG_B, SIG_X, SIG_R = 0.02, 0.01, 1.0, 0.02


def stream_id(cid: int, tensor: int, layer: int, expert: int = 0) -> int:
    return (cid << 56) | (tensor << 48) | (layer << 32) | expert


def act_block(n: int) -> int:
    """Activation quantisation block: 256 where n is a multiple of 256, else 32."""
    if n % 256 == 0:
        return 256
    if n % 32 == 0:
        return 32
    raise ValueError(f"width {n} is not a multiple of 32")


@dataclass
class Layer:
    cfg: MoEConfig
    layer: int
    T: int
    x: np.ndarray                      # float32 [T, H]
    router: np.ndarray                 # float32 [E, H] or uint8 [E, row_bytes]
    router_bias: np.ndarray | None     # float32 [E]
    gate: np.ndarray                   # uint8 [E, I, row_bytes(H)]
    up: np.ndarray
    down: np.ndarray                   # uint8 [E, H, row_bytes(I)]
    bg: np.ndarray | None = None       # float32 [E, I]
    bu: np.ndarray | None = None
    bd: np.ndarray | None = None       # float32 [E, H]
    sgate: np.ndarray | None = None    # uint8 [1, Is, row_bytes(H)]
    sup: np.ndarray | None = None
    sdown: np.ndarray | None = None
    shexp_gate: np.ndarray | None = None   # float32 [H]: the shared expert's gate vector
    extra: dict = field(default_factory=dict)


def zipf_bias(cfg: MoEConfig, layer: int, seed: int = 0, s: float = 1.1) -> np.ndarray:
    rng = np.random.default_rng([seed, cfg.cid, layer, 0x21F])
    rank = rng.permutation(cfg.E) + 1
    return (-s * np.log(rank.astype(np.float64))).astype(np.float32)


def make_x(cfg: MoEConfig, layer: int, T: int, seed: int = 0) -> np.ndarray:
    return normal(seed, stream_id(cfg.cid, _T_X, layer), SIG_X, T, cfg.H)


def make_layer(cfg: MoEConfig, layer: int = 0, T: int = 1, seed: int = 0,
               zipf: bool | None = None, with_experts: bool = True) -> Layer:
    """One MoE layer of cfg with its T-token input, all drawn from seeded streams.

    Token t's hidden state does not depend on T, and every tensor of layer l is
    drawn from its own stream, so layers are independent (router logits drawn
    independently per layer)."""
    c, H, I, E = cfg.cid, cfg.H, cfg.I, cfg.E
    if zipf is None:
        zipf = T in cfg.zipf_tokens
    x = make_x(cfg, layer, T, seed)
    router = matrix(cfg.router_qtype, seed, stream_id(c, _T_ROUTER, layer), SIG_R, E, H)
    rbias = zipf_bias(cfg, layer, seed) if zipf else None
    L = Layer(cfg, layer, T, x, router, rbias, None, None, None)
    if not with_experts:
        return L
    # expert e's matrix is rows [e*rows, (e+1)*rows) of its tensor's stream
    L.gate = matrix(cfg.qtype, seed, stream_id(c, _T_GATE, layer), SIG_W, E * I, H).reshape(E, I, -1)
    L.up = matrix(cfg.qtype, seed, stream_id(c, _T_UP, layer), SIG_W, E * I, H).reshape(E, I, -1)
    L.down = matrix(cfg.qtype, seed, stream_id(c, _T_DOWN, layer), SIG_W, E * H, I).reshape(E, H, -1)
    if cfg.biases:
        L.bg = normal(seed, stream_id(c, _T_BG, layer), SIG_B, E, I)
        L.bu = normal(seed, stream_id(c, _T_BU, layer), SIG_B, E, I)
        L.bd = normal(seed, stream_id(c, _T_BD, layer), SIG_B, E, H)
    if cfg.has_shared:
        Is, qs = cfg.shared_I, cfg.shared_qtype
        L.sgate = matrix(qs, seed, stream_id(c, _T_SGATE, layer), SIG_W, Is, H)[None]
        L.sup = matrix(qs, seed, stream_id(c, _T_SUP, layer), SIG_W, Is, H)[None]
        L.sdown = matrix(qs, seed, stream_id(c, _T_SDOWN, layer), SIG_W, H, Is)[None]
        if cfg.shared_gate:
            L.shexp_gate = normal(seed, stream_id(c, _T_SHGATE, layer), SIG_R, 1, H)[0]
    return L


def shrink(cfg: MoEConfig, **kw) -> MoEConfig:
    """A smaller variant of cfg (same formats, routing and structure)."""
    d = {f: getattr(cfg, f) for f in cfg.__dataclass_fields__}
    d.update(kw)
    return MoEConfig(**d)
