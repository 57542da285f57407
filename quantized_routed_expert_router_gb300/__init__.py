"""Python binding of the GB300 quantized routed-expert MoE FFN library.

Argument marshalling only: every step of the path runs in the CUDA library
``_moe.so`` (C ABI, ``include/moe.h``); this module passes tensor addresses,
sizes and the current CUDA stream through ctypes.  PyTorch supplies device
memory and streams.  Importing works without a GPU; the library must have
been built (``_build.build()``) - there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

F32, Q8_0, Q4_K, Q2_K, MXFP4, Q6_K, Q3_K = 0, 1, 2, 3, 4, 5, 6
SOFTMAX, SIGMOID = 0, 1
DEV_BAD_ID, DEV_DUP_ID = 0x1, 0x2
MAX_TOKENS, MAX_K, MAX_EXPERTS = 16, 32, 1024

EXPORTS = ["moe_act_block", "moe_q8_row_bytes", "moe_packed_bytes", "moe_pack_weights", "moe_quantize_q8K",
           "moe_route", "moe_route_workspace_bytes", "moe_expert_ffn", "moe_ffn_workspace_bytes",
           "moe_read_device_status", "moe_debug_row_dots", "moe_status_str", "moe_expert_ffn_noalloc",
           "moe_layer_forward", "moe_layer_workspace_bytes", "moe_sum_partials", "moe_debug_set_exchange_wait"]
LAYER_OVERLAP_PREVIOUS = 0x1
DEV_TIMEOUT = 0x4

_P = ctypes.c_void_p
_lib_handle = None


class MoeError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        super().__init__(f"{call}: {status_str(status)} (status {status})")


class _Expert(ctypes.Structure):
    _fields_ = [("gate", _P), ("up", _P), ("down", _P), ("b_gate", _P), ("b_up", _P), ("b_down", _P)]


class _Pool(ctypes.Structure):
    _fields_ = [("qtype", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int), ("E", ctypes.c_int),
                ("experts", _P)]


def library_path() -> str:
    return _build.SO


def lib():
    """The loaded C library.  Raises if it has not been built."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(_build.SO):
            raise RuntimeError(f"CUDA library not built: {_build.SO} is missing (run __graft_entry__.build())")
        L = ctypes.CDLL(_build.SO)
        i, sz = ctypes.c_int, ctypes.c_size_t
        L.moe_act_block.restype = i
        L.moe_act_block.argtypes = [i]
        L.moe_q8_row_bytes.restype = sz
        L.moe_q8_row_bytes.argtypes = [i]
        L.moe_packed_bytes.restype = sz
        L.moe_packed_bytes.argtypes = [i, i, i]
        L.moe_pack_weights.restype = i
        L.moe_pack_weights.argtypes = [_P, i, i, i, _P, _P]
        L.moe_quantize_q8K.restype = i
        L.moe_quantize_q8K.argtypes = [_P, i, i, _P, _P]
        L.moe_route.restype = i
        L.moe_route.argtypes = [_P, _P, i, i, _P, i, i, _P, i, i, i, _P, _P, _P, _P, _P, _P, sz, _P]
        L.moe_route_workspace_bytes.restype = sz
        L.moe_route_workspace_bytes.argtypes = [i, i, i]
        L.moe_expert_ffn.restype = i
        L.moe_expert_ffn.argtypes = [_P, i, _P, _P, i, ctypes.POINTER(_Pool), ctypes.POINTER(_Pool), _P, _P, _P, sz,
                                     _P]
        L.moe_expert_ffn_noalloc.restype = i
        L.moe_expert_ffn_noalloc.argtypes = [_P, i, _P, _P, i, ctypes.POINTER(_Pool), ctypes.POINTER(_Pool), _P, _P,
                                             _P]
        L.moe_layer_forward.restype = i
        L.moe_layer_forward.argtypes = [_P, i, _P, i, _P, i, i, i, ctypes.POINTER(_Pool), ctypes.POINTER(_Pool),
                                        _P, _P, _P, _P, _P, _P, _P, sz, ctypes.c_uint, _P]
        L.moe_layer_workspace_bytes.restype = sz
        L.moe_layer_workspace_bytes.argtypes = [i, i, ctypes.POINTER(_Pool), ctypes.POINTER(_Pool)]
        L.moe_ffn_workspace_bytes.restype = sz
        L.moe_ffn_workspace_bytes.argtypes = [i, i, ctypes.POINTER(_Pool), ctypes.POINTER(_Pool)]
        L.moe_read_device_status.restype = i
        L.moe_read_device_status.argtypes = [_P, i, ctypes.POINTER(ctypes.c_uint32), _P]
        L.moe_debug_row_dots.restype = i
        L.moe_debug_row_dots.argtypes = [_P, i, i, i, i, _P, _P, _P]
        L.moe_sum_partials.restype = i
        L.moe_sum_partials.argtypes = [_P, i, sz, _P, _P]
        L.moe_debug_set_exchange_wait.restype = i
        L.moe_debug_set_exchange_wait.argtypes = [ctypes.c_longlong]
        L.moe_status_str.restype = ctypes.c_char_p
        L.moe_status_str.argtypes = [i]
        _lib_handle = L
    return _lib_handle


def status_str(s: int) -> str:
    return lib().moe_status_str(s).decode()


def _check(s: int, call: str):
    if s != 0:
        raise MoeError(s, call)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


# ------------------------------------------------------------------ sizes

def moe_act_block(n: int) -> int:
    return lib().moe_act_block(n)


def moe_q8_row_bytes(n: int) -> int:
    return lib().moe_q8_row_bytes(n)


def moe_packed_bytes(qtype: int, rows: int, cols: int) -> int:
    return lib().moe_packed_bytes(qtype, rows, cols)


# ------------------------------------------------------------------ calls

def moe_pack_weights(blocks: torch.Tensor, qtype: int, rows: int, cols: int, packed: torch.Tensor, stream=None):
    _check(lib().moe_pack_weights(_ptr(blocks), qtype, rows, cols, _ptr(packed), _stream(stream)),
           "moe_pack_weights")


def moe_quantize_q8K(x: torch.Tensor, xq: torch.Tensor, stream=None):
    T, n = x.shape
    _check(lib().moe_quantize_q8K(_ptr(x), T, n, _ptr(xq), _stream(stream)), "moe_quantize_q8K")


def moe_route_workspace_bytes(T: int, E: int, H: int) -> int:
    return lib().moe_route_workspace_bytes(T, E, H)


def moe_route(hidden, xq, w_router, rtype: int, E: int, router_bias, k: int, gating: int, renormalize: bool,
              ids, weights, logits_out, ws, T: int | None = None, H: int | None = None, stream=None,
              shared_gate=None, shared_scale=None):
    if T is None or H is None:
        T, H = hidden.shape
    _check(lib().moe_route(_ptr(hidden), _ptr(xq), T, H, _ptr(w_router), rtype, E, _ptr(router_bias), k, gating,
                           int(bool(renormalize)), _ptr(ids), _ptr(weights), _ptr(logits_out), _ptr(shared_gate),
                           _ptr(shared_scale), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_route")


class ExpertPool:
    """A moe_pool: packed expert matrices plus the device pointer table.

    entries: list of dicts with packed 'gate', 'up', 'down' tensors (or None
    for "not mine") and optional 'b_gate', 'b_up', 'b_down' fp32 tensors.
    A fused gate_up tensor (GGUF files may store gate and up as one [2I][H]
    matrix, gate rows first) packed as one matrix is given as 'gate_up': its
    first moe_packed_bytes(qtype, I, H) bytes are the gate, the rest the up
    projection (packed tiles of 32 rows are contiguous)."""

    def __init__(self, qtype: int, H: int, I: int, entries: list, device=None):
        self.qtype, self.H, self.I, self.E = qtype, H, I, len(entries)
        self._keep = []
        rows = []
        for en in entries:
            if en is not None and en.get("gate_up") is not None:
                if en.get("gate") is not None or en.get("up") is not None:
                    raise ValueError("give either 'gate_up' or 'gate' and 'up'")
                half = moe_packed_bytes(qtype, I, H)
                gu = en["gate_up"]
                if half == 0 or gu.numel() * gu.element_size() != 2 * half:
                    raise ValueError(f"'gate_up' must hold 2 x {half} packed bytes")
                flat = gu.reshape(-1).view(torch.uint8)
                en = dict(en, gate=flat[:half], up=flat[half:])
                del en["gate_up"]
            if en is None or en.get("gate") is None:
                rows.append([0] * 6)
                continue
            vals = [en.get(n) for n in ("gate", "up", "down", "b_gate", "b_up", "b_down")]
            self._keep.extend(v for v in vals if v is not None)
            rows.append([0 if v is None else v.data_ptr() for v in vals])
        device = device or (self._keep[0].device if self._keep else torch.device("cuda"))
        self.table = torch.tensor(rows, dtype=torch.int64).reshape(-1, 6).to(device)
        self.c = _Pool(qtype, H, I, self.E, self.table.data_ptr())


def moe_ffn_workspace_bytes(T: int, k: int, pool: ExpertPool, shared: ExpertPool | None) -> int:
    return lib().moe_ffn_workspace_bytes(T, k, ctypes.byref(pool.c),
                                         ctypes.byref(shared.c) if shared is not None else None)


def moe_expert_ffn(xq, T: int, ids, weights, k: int, pool: ExpertPool, shared: ExpertPool | None, y, ws,
                   stream=None, shared_scale=None):
    _check(lib().moe_expert_ffn(_ptr(xq), T, _ptr(ids), _ptr(weights), k, ctypes.byref(pool.c),
                                ctypes.byref(shared.c) if shared is not None else None, _ptr(shared_scale), _ptr(y),
                                _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)), "moe_expert_ffn")


def moe_expert_ffn_noalloc(xq, T: int, ids, weights, k: int, pool: ExpertPool, shared: ExpertPool | None, y,
                           stream=None, shared_scale=None):
    """moe_expert_ffn with the library's fixed device scratch (no workspace, no allocation)."""
    _check(lib().moe_expert_ffn_noalloc(_ptr(xq), T, _ptr(ids), _ptr(weights), k, ctypes.byref(pool.c),
                                        ctypes.byref(shared.c) if shared is not None else None,
                                        _ptr(shared_scale), _ptr(y), _stream(stream)), "moe_expert_ffn_noalloc")


def moe_layer_workspace_bytes(T: int, k: int, pool: ExpertPool, shared: ExpertPool | None) -> int:
    return lib().moe_layer_workspace_bytes(T, k, ctypes.byref(pool.c),
                                           ctypes.byref(shared.c) if shared is not None else None)


def moe_layer_forward(hidden, w_router, rtype: int, router_bias, k: int, gating: int, renormalize: bool,
                      pool: ExpertPool, shared: ExpertPool | None, y, ws, ids_out=None, weights_out=None,
                      logits_out=None, xq_out=None, flags: int = 0, T: int | None = None, stream=None,
                      shared_gate=None):
    T = hidden.shape[0] if T is None else T
    _check(lib().moe_layer_forward(_ptr(hidden), T, _ptr(w_router), rtype, _ptr(router_bias), k, gating,
                                   int(bool(renormalize)), ctypes.byref(pool.c),
                                   ctypes.byref(shared.c) if shared is not None else None, _ptr(shared_gate),
                                   _ptr(y),
                                   _ptr(ids_out), _ptr(weights_out), _ptr(logits_out), _ptr(xq_out), _ptr(ws),
                                   ws.numel() * ws.element_size(), flags, _stream(stream)), "moe_layer_forward")


def moe_sum_partials(parts, y, stream=None):
    """y = the partial outputs parts [R, ...] summed in rank order (expert parallelism)."""
    R = parts.shape[0]
    n = y.numel()
    if parts.numel() != R * n:
        raise ValueError("parts must hold R partials of y's size")
    _check(lib().moe_sum_partials(_ptr(parts), R, n, _ptr(y), _stream(stream)), "moe_sum_partials")


def moe_debug_set_exchange_wait(cycles: int):
    """Test hook: bound on a layer launch's waits for other blocks' words (0: default)."""
    _check(lib().moe_debug_set_exchange_wait(int(cycles)), "moe_debug_set_exchange_wait")


def moe_read_device_status(ws, clear: bool = True, stream=None) -> int:
    flags = ctypes.c_uint32(0)
    s = lib().moe_read_device_status(_ptr(ws), int(clear), ctypes.byref(flags), _stream(stream))
    if s not in (0, 5):
        raise MoeError(s, "moe_read_device_status")
    return flags.value


def moe_debug_row_dots(packed, qtype: int, rows: int, cols: int, row: int, xq, isums, stream=None):
    _check(lib().moe_debug_row_dots(_ptr(packed), qtype, rows, cols, row, _ptr(xq), _ptr(isums),
                                    _stream(stream)), "moe_debug_row_dots")


# ----------------------------------------------------------- conveniences

def device_bytes(n: int, device="cuda") -> torch.Tensor:
    """A 256-byte aligned uint8 device buffer (torch's allocator aligns to 512)."""
    return torch.empty(max(int(n), 16), dtype=torch.uint8, device=device)


def pack(blocks: torch.Tensor, qtype: int, rows: int, cols: int, stream=None) -> torch.Tensor:
    """Pack one GGUF-style block matrix (device uint8) into a new device buffer."""
    out = device_bytes(moe_packed_bytes(qtype, rows, cols), blocks.device)
    moe_pack_weights(blocks, qtype, rows, cols, out, stream)
    return out


def quantize(x: torch.Tensor, stream=None) -> torch.Tensor:
    T, n = x.shape
    xq = device_bytes(T * moe_q8_row_bytes(n), x.device)
    moe_quantize_q8K(x, xq, stream)
    return xq


def unpack_q8(xq: torch.Tensor, T: int, n: int):
    """Split q8 records (host or device uint8) into (d [T, n/B], q [T, n], bsum [T, n/16]) tensors."""
    B = moe_act_block(n)
    rb = moe_q8_row_bytes(n)
    a = ((4 * (n // B)) + 15) & ~15
    r = xq[: T * rb].reshape(T, rb)
    d = r[:, : 4 * (n // B)].contiguous().view(torch.float32)
    q = r[:, a: a + n].contiguous().view(torch.int8)
    bs = r[:, a + n: a + n + 2 * (n // 16)].contiguous().view(torch.int16)
    return d, q, bs
