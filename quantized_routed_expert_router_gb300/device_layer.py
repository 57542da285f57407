"""Device-resident MoE layer: uploads one layer's tensors, packs the expert
matrices once, builds the expert pointer tables and runs the hot path
(quantise -> route -> expert FFN) through the C ABI.

Marshalling only.  The layer object is duck-typed (the fields of a decode
layer: x, router, router_bias, gate/up/down blocks, biases, shared expert)."""
from __future__ import annotations

import numpy as np
import torch

from . import (ExpertPool, F32, SIGMOID, SOFTMAX, device_bytes, moe_expert_ffn, moe_ffn_workspace_bytes,
               moe_layer_forward, moe_layer_workspace_bytes, moe_pack_weights, moe_packed_bytes,
               moe_q8_row_bytes, moe_quantize_q8K, moe_route, moe_route_workspace_bytes)


def _dev(a, device, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(device, non_blocking=False)


def pack_stack(blocks: np.ndarray, qtype: int, rows_per: int, cols: int, device) -> tuple[torch.Tensor, int]:
    """Pack [E, rows_per, row_bytes] blocks as one matrix; returns (buffer, bytes per expert)."""
    E = blocks.shape[0]
    src = _dev(blocks.reshape(E * rows_per, -1), device)
    out = device_bytes(moe_packed_bytes(qtype, E * rows_per, cols), device)
    moe_pack_weights(src, qtype, E * rows_per, cols, out)
    del src
    return out, moe_packed_bytes(qtype, rows_per, cols)


class DeviceLayer:
    def __init__(self, L, device="cuda", owned=None, with_shared=True, T: int | None = None):
        cfg = L.cfg
        self.cfg = cfg
        self.device = torch.device(device)
        self.T = L.x.shape[0] if T is None else T
        self.H, self.I, self.E, self.k = cfg.H, cfg.I, cfg.E, cfg.k
        self.x = _dev(L.x, device)
        self.router_qtype = cfg.router_qtype
        self.router = _dev(L.router, device)
        self.router_bias = None if L.router_bias is None else _dev(L.router_bias, device)
        self.gating = SIGMOID if cfg.gating == "sigmoid" else SOFTMAX
        self.renorm = cfg.renorm
        q, H, I, E = cfg.qtype, cfg.H, cfg.I, cfg.E
        self.gate, sg = pack_stack(L.gate, q, I, H, device)
        self.up, su = pack_stack(L.up, q, I, H, device)
        self.down, sd = pack_stack(L.down, q, H, I, device)
        self.bg = None if L.bg is None else _dev(L.bg, device)
        self.bu = None if L.bu is None else _dev(L.bu, device)
        self.bd = None if L.bd is None else _dev(L.bd, device)
        self.sizes = (sg, su, sd)
        self.pool = self.make_pool(owned)
        self.shared = None
        if with_shared and cfg.has_shared:
            Is, qs = cfg.shared_I, cfg.shared_qtype
            self.sgate, _ = pack_stack(L.sgate, qs, Is, H, device)
            self.sup, _ = pack_stack(L.sup, qs, Is, H, device)
            self.sdown, _ = pack_stack(L.sdown, qs, H, Is, device)
            self.shared = ExpertPool(qs, H, Is, [dict(gate=self.sgate, up=self.sup, down=self.sdown)], self.device)
        shg = getattr(L, "shexp_gate", None)   # the shared expert's gate vector, if the layer has one
        self.shared_gate = None if (shg is None or self.shared is None) else _dev(shg, device)
        self.alloc(self.T)

    def make_pool(self, owned=None) -> ExpertPool:
        sg, su, sd = self.sizes
        entries = []
        for e in range(self.E):
            if owned is not None and not owned[e]:
                entries.append(None)
                continue
            en = dict(gate=self.gate[e * sg:(e + 1) * sg], up=self.up[e * su:(e + 1) * su],
                      down=self.down[e * sd:(e + 1) * sd])
            if self.bg is not None:
                en.update(b_gate=self.bg[e], b_up=self.bu[e], b_down=self.bd[e])
            entries.append(en)
        return ExpertPool(self.cfg.qtype, self.H, self.I, entries, self.device)

    def alloc(self, T: int):
        d = self.device
        self.xq = device_bytes(T * moe_q8_row_bytes(self.H), d)
        self.ids = torch.empty((T, self.k), dtype=torch.int32, device=d)
        self.w = torch.empty((T, self.k), dtype=torch.float32, device=d)
        self.logits = torch.empty((T, self.E), dtype=torch.float32, device=d)
        self.y = torch.empty((T, self.H), dtype=torch.float32, device=d)
        self.shared_scale = torch.empty(T, dtype=torch.float32, device=d) if self.shared_gate is not None else None
        self.ws_route = torch.zeros(moe_route_workspace_bytes(T, self.E, self.H), dtype=torch.uint8, device=d)
        self.ws_ffn = torch.zeros(moe_ffn_workspace_bytes(T, self.k, self.pool, self.shared), dtype=torch.uint8,
                                  device=d)
        self.ws_layer = torch.zeros(moe_layer_workspace_bytes(T, self.k, self.pool, self.shared),
                                    dtype=torch.uint8, device=d)

    def quantize(self, x=None, stream=None):
        moe_quantize_q8K(self.x if x is None else x, self.xq, stream)

    def route(self, x=None, stream=None, logits=True):
        x = self.x if x is None else x
        moe_route(x, self.xq, self.router, self.router_qtype, self.E, self.router_bias, self.k, self.gating,
                  self.renorm, self.ids, self.w, self.logits if logits else None, self.ws_route, stream=stream,
                  shared_gate=self.shared_gate, shared_scale=self.shared_scale)

    def ffn(self, ids=None, w=None, pool=None, shared="default", y=None, stream=None, T=None):
        T = self.T if T is None else T
        sh = self.shared if shared == "default" else shared
        moe_expert_ffn(self.xq, T, self.ids if ids is None else ids, self.w if w is None else w, self.k,
                       self.pool if pool is None else pool, sh, self.y if y is None else y, self.ws_ffn, stream,
                       shared_scale=self.shared_scale if sh is not None else None)

    def forward(self, x=None, stream=None, logits=True):
        """three calls: moe_quantize_q8K, moe_route, moe_expert_ffn"""
        self.quantize(x, stream)
        self.route(x, stream, logits)
        self.ffn(stream=stream)
        return self.y

    def forward_fused(self, x=None, stream=None, outputs=True, flags=0, pool=None, shared="default", y=None):
        """one call: moe_layer_forward"""
        x = self.x if x is None else x
        sh = self.shared if shared == "default" else shared
        moe_layer_forward(x, self.router, self.router_qtype, self.router_bias, self.k, self.gating, self.renorm,
                          self.pool if pool is None else pool, sh,
                          self.y if y is None else y, self.ws_layer,
                          ids_out=self.ids if outputs else None, weights_out=self.w if outputs else None,
                          logits_out=self.logits if outputs else None, xq_out=self.xq if outputs else None,
                          flags=flags, stream=stream, shared_gate=self.shared_gate if sh is not None else None)
        return self.y
