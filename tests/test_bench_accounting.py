"""The benchmark's roofline numerator: algorithmic bytes of one layer step.

Counted as the unique chosen experts' packed gate/up/down bytes (+ their
biases), the shared expert, the router and the activations.  The figures are
the block sizes of the formats multiplied out by hand: Q4_K is 144 bytes per
256 weights, so a 512 x 2048 matrix is 512 * 8 * 144 = 589,824 bytes.
"""
import importlib.util
import os
import types

import numpy as np
import torch

import quantized_routed_expert_router_gb300 as moe
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)


def fake_layer(cfg, ids, router_bytes_per_elem=4):
    """the attributes layer_bytes reads, without a device"""
    sizes = (moe.moe_packed_bytes(cfg.qtype, cfg.I, cfg.H), moe.moe_packed_bytes(cfg.qtype, cfg.I, cfg.H),
             moe.moe_packed_bytes(cfg.qtype, cfg.H, cfg.I))
    router = torch.zeros(cfg.E * cfg.H * 4 // router_bytes_per_elem,
                         dtype=torch.float32 if router_bytes_per_elem == 4 else torch.uint8)
    return types.SimpleNamespace(ids=torch.tensor(ids, dtype=torch.int32), sizes=sizes, router=router,
                                 shared=object() if cfg.shared_I else None)


def test_35b_a3b_style_layer_bytes_at_one_token():
    cfg = synth.CONFIGS["a3b"]
    b = bench.layer_bytes(cfg, fake_layer(cfg, [[3, 9, 17, 40, 77, 120, 200, 255]]), moe)
    per_expert = 3 * 512 * 8 * 144                       # gate, up: 512 x 2048; down: 2048 x 512
    assert per_expert == 1_769_472
    assert b["unique"] == 8
    assert b["experts"] == 8 * per_expert
    assert b["shared"] == per_expert                     # shared expert: same shape and format
    assert b["router"] == 256 * 2048 * 4
    assert b["act"] == 2048 * 4 * 2 + 8 * 8
    assert b["total"] == 18_038_848


def test_repeated_experts_are_counted_once():
    cfg = synth.CONFIGS["a3b"]
    ids = [[1, 2, 3, 4, 5, 6, 7, 8], [1, 2, 3, 4, 9, 10, 11, 12]]   # two tokens, 12 unique experts
    b = bench.layer_bytes(cfg, fake_layer(cfg, ids), moe)
    assert b["unique"] == 12
    assert b["experts"] == 12 * 1_769_472
    assert b["act"] == 2 * 2048 * 4 * 2 + 2 * 8 * 8


def test_biases_count_for_gpt_oss_style_experts():
    cfg = synth.CONFIGS["oss20b"]
    b = bench.layer_bytes(cfg, fake_layer(cfg, [[0, 5, 9, 31]]), moe)
    per_expert = 2 * moe.moe_packed_bytes(synth.MXFP4, 2880, 2880) + moe.moe_packed_bytes(synth.MXFP4, 2880, 2880)
    assert b["experts"] == 4 * per_expert + 4 * (2 * 2880 + 2880) * 4
    assert b["shared"] == 0
