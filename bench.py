#!/usr/bin/env python
"""MoE-layer decode throughput of the GB300 quantized routed-expert FFN.

One step = one batch of T tokens through an L-layer stack of distinct MoE
layers (each layer: quantise -> route -> routed + shared expert FFN), replayed
from a CUDA graph.  Layers are timed as decode: each layer's kernels start
after the previous layer's finish (stream order).  Every layer has its own
seeded weights and hidden states, so a step touches L x (per-layer bytes) of
HBM - far more than the 129 MB L2 - and no L2 flush is needed.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "MoE-layer decode tokens/s and achieved HBM GB/s vs ~8 TB/s peak (1xGB300)"
UNIT = "layer-tok/s"
DEFAULT_LAYERS = {"tiny": 64, "a3b": 40, "oss20b": 24, "wide": 8, "a22b": 48}
FALLBACK_HBM_GBS = 6800.0


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default="a22b")
    p.add_argument("--also", default="a3b",
                   help="comma list of further workloads timed after the main one and reported under "
                        "config.also (T=1, default stack depth); 'none' to skip")
    p.add_argument("--layers", type=int, default=0)
    p.add_argument("--tokens", type=int, default=1)
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--no-overlap", action="store_true", help="launch layers without the overlap flag")
    p.add_argument("--split", choices=["tokens", "experts"], default="tokens",
                   help="tokens: every rank decodes its own tokens (replicas); experts: every rank holds the "
                        "experts e with e %% world == rank (rank 0 also the shared expert) of the same layers, "
                        "and each layer's partial outputs are gathered and summed in rank order")
    return p.parse_args()


def rank_env():
    """(rank, world size, local rank) from the torchrun environment; (0, 1, 0) alone."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(seed: int, rank: int) -> int:
    """Seed of a rank's tokens: every rank decodes its own tokens (data parallel)."""
    return seed + 7919 * rank


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest value over all ranks (the slowest rank sets the job's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def expert_owner_mask(E: int, rank: int, world: int) -> np.ndarray:
    """Experts rank `rank` holds under the expert-parallel split: e % world == rank."""
    return np.arange(E) % world == rank


def rank_order_sum(parts):
    """Host-side statement of the reduction moe_sum_partials performs on the
    device: the partials added in rank order."""
    y = np.array(parts[0], copy=True)
    for p in parts[1:]:
        y = y + p
    return y


def job_throughput(world: int, steps: int, layers: int, tokens: int, seconds: float) -> float:
    """Layer-tokens per second of the whole job: every rank processed steps x layers x tokens."""
    return world * steps * layers * tokens / seconds


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def csrc_hash():
    h = hashlib.sha256()
    d = os.path.join(ROOT, "quantized_routed_expert_router_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def traffic_record(kernel_key: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel sources are unchanged."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        rec = d.get(kernel_key)
        if rec and rec.get("csrc_hash") == csrc_hash():
            return float(rec["bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.p is not None:
            time.sleep(0.2)
            self.p.terminate()
            try:
                self.out, _ = self.p.communicate(timeout=5)
            except Exception:
                self.p.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), active=f[4], hw=f[5], hwt=f[6], swt=f[7],
                                 pcap=f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        smax = max(r["smax"] for r in rows)
        load = [r for r in rows if r["sm"] >= 0.5 * smax] or rows
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                              ("pcap", "sw_power_cap")):
                if r[key].lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in load), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(rows)}


def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def time_oracle(layers, threads, steps=None, seconds=None):
    """The CPU oracle's layer forward on `threads` host threads at once.

    Thread i runs oracle.layer_forward over the seeded layers in turn, starting
    at layer i, for `steps` layer-steps or until `seconds` have passed.  The
    oracle's work runs in C behind ctypes, which releases the GIL, so the
    threads run in parallel; the oracle keeps no global state.  Returns
    (layer-steps done by all threads, wall seconds)."""
    import threading

    import oracle
    done, errors = [0] * threads, []
    t0 = time.perf_counter()

    def work(i):
        n = 0
        try:
            while (steps is None or n < steps) and (seconds is None or time.perf_counter() - t0 < seconds):
                oracle.layer_forward(layers[(i + n) % len(layers)])
                n += 1
        except Exception as e:  # surfaced after the join
            errors.append(e)
        done[i] = n

    pool = [threading.Thread(target=work, args=(i,)) for i in range(threads)]
    for t in pool:
        t.start()
    for t in pool:
        t.join()
    dt = time.perf_counter() - t0
    if errors:
        raise errors[0]
    return sum(done), dt


def layer_bytes(cfg, dl, moe):
    """Algorithmic HBM bytes of one layer-step: unique chosen experts + shared + router + activations."""
    ids = dl.ids.cpu().numpy()
    unique = len(np.unique(ids))
    T = ids.shape[0]
    per_expert = sum(dl.sizes)
    shared = 0
    if dl.shared is not None:
        shared = (2 * moe.moe_packed_bytes(cfg.shared_qtype, cfg.shared_I, cfg.H)
                  + moe.moe_packed_bytes(cfg.shared_qtype, cfg.H, cfg.shared_I))
    bias = (2 * cfg.I + cfg.H) * 4 * unique if cfg.biases else 0
    router = dl.router.numel() * dl.router.element_size()
    act = T * cfg.H * 4 * 2 + T * cfg.k * 8
    return dict(experts=unique * per_expert + bias, shared=shared, router=router, act=act, unique=unique,
                total=unique * per_expert + bias + shared + router + act)


def run_reference(args, cfg, L, rank, world):
    import synth
    if rank != 0:
        return
    nsample = 2
    layers = [synth.make_layer(cfg, l, T=args.tokens, seed=args.seed) for l in range(nsample)]
    C = host_threads()
    time_oracle(layers, C, steps=args.warmup)
    n, dt = time_oracle(layers, C, steps=args.steps)
    v = n * args.tokens / dt
    sample = (f"one {cfg.name} layer x {args.tokens} token(s) per host thread per step ({C} threads at once), "
              f"cycling over {nsample} seeded layers; scalar C oracle")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",   # exact int32 dots, fp64 scale combine
            "data": "synthetic",
            "config": {"workload": workload_name(cfg, L, args.tokens), "tokens": args.tokens, "layers": L},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": C, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_name(cfg, L, T):
    return f"{cfg.name}: {cfg.note}; {L}-layer stack of distinct layers, {T} token(s) per step (decode)"


class Stack:
    """L distinct seeded layers of one workload on the device, captured as
    CUDA graphs: one fused launch per layer ("step"), the three calls per
    layer ("three") and the FFN call alone ("ffn")."""

    def __init__(self, cfg, L, T, seed, dev, stream, overlap, keep_host=0, owned=None, with_shared=True):
        import torch
        import synth
        import quantized_routed_expert_router_gb300 as moe
        from quantized_routed_expert_router_gb300.device_layer import DeviceLayer
        self.cfg, self.L, self.T = cfg, L, T
        t_gen = time.perf_counter()
        self.layers, self.host_sample = [], []
        for l in range(L):
            Lh = synth.make_layer(cfg, l, T=T, seed=seed)
            self.layers.append(DeviceLayer(Lh, dev, owned=owned, with_shared=with_shared))
            if l < keep_host:
                self.host_sample.append(Lh)
            del Lh
        # one contiguous input and output buffer for the whole stack, so the
        # end-to-end leg moves each step's inputs and results in one copy each
        self.X = torch.empty((L, T, cfg.H), dtype=torch.float32, device=dev)
        self.Y = torch.empty((L, T, cfg.H), dtype=torch.float32, device=dev)
        for l, dl in enumerate(self.layers):
            self.X[l].copy_(dl.x)
            dl.x, dl.y = self.X[l], self.Y[l]
        torch.cuda.synchronize()
        self.gen_s = time.perf_counter() - t_gen
        flags = moe.LAYER_OVERLAP_PREVIOUS if overlap else 0

        def step_fused():
            for dl in self.layers:
                dl.forward_fused(flags=flags, outputs=False)

        def step_three(ffn_only=False):
            for dl in self.layers:
                if not ffn_only:
                    dl.quantize()
                    dl.route(logits=False)
                dl.ffn()

        with torch.cuda.stream(stream):
            step_three()                  # eager once: kernel attributes, ids for the byte count
            step_fused()
        torch.cuda.synchronize()
        bad = [moe.moe_read_device_status(dl.ws_layer) for dl in self.layers]
        if any(bad):
            raise RuntimeError(f"device status after the first fused step: {bad}")
        self.bytes_l = [layer_bytes(cfg, dl, moe) for dl in self.layers]
        self.step_bytes = sum(b["total"] for b in self.bytes_l)
        self.graphs = {}
        for name, fn in (("step", step_fused), ("three", step_three), ("ffn", lambda: step_three(ffn_only=True))):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                fn()
            self.graphs[name] = g
        torch.cuda.synchronize()

    def status(self):
        import quantized_routed_expert_router_gb300 as moe
        return [moe.moe_read_device_status(dl.ws_layer) for dl in self.layers]


def timed(g, K, W, stream, world, dev):
    """Device milliseconds of K graph replays after W untimed ones, max over ranks."""
    import torch
    import torch.distributed as dist
    for _ in range(W):
        g.replay()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(K):
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    return max_over_ranks(e0.elapsed_time(e1), world, dev)


def side_figures(S, K, W, stream, world, dev, peak):
    """A further workload's fused-stack figures (reported beside the main line)."""
    ms = timed(S.graphs["step"], K, W, stream, world, dev)
    st = S.status()
    if any(st):
        raise RuntimeError(f"device status after the timed region ({S.cfg.name}): {st}")
    us = 1e3 * ms / (K * S.L)
    gbs = (S.step_bytes / S.L) / (us / 1e6) / 1e9
    return {"workload": workload_name(S.cfg, S.L, S.T), "steps": K, "layer_tok_s": job_throughput(
        world, K, S.L, S.T, ms / 1e3), "us_per_layer": us, "bytes_per_layer": S.step_bytes / S.L,
        "hbm_gbs": gbs, "hbm_frac_of_measured": gbs / peak, "setup_s": S.gen_s}


def run_expert_parallel(args, cfg, L, T, rank, world, local, dev, stream, peak, peak_src):
    """Expert parallelism over the ranks: the same L layers and tokens on every
    rank; rank r holds the experts with e % world == r (rank 0 also the shared
    expert), runs the layer call on that pool (NULL entries: "not mine") and
    gets a partial y; the partials of each layer are gathered and summed in
    rank order (moe_sum_partials) before the next layer, as decode needs.
    Eager launches (the gather is a collective between them)."""
    import torch
    import torch.distributed as dist
    import quantized_routed_expert_router_gb300 as moe
    owned = expert_owner_mask(cfg.E, rank, world)
    S = Stack(cfg, L, T, args.seed, dev, stream, not args.no_overlap, owned=owned, with_shared=(rank == 0))
    gathered = torch.empty((world, T, cfg.H), dtype=torch.float32, device=dev)
    Yfull = torch.empty((L, T, cfg.H), dtype=torch.float32, device=dev)
    flags = 0 if args.no_overlap else moe.LAYER_OVERLAP_PREVIOUS

    def step():
        for l, dl in enumerate(S.layers):
            dl.forward_fused(flags=flags, outputs=False)
            if world > 1:
                dist.all_gather_into_tensor(gathered, dl.y)
                moe.moe_sum_partials(gathered, Yfull[l])
            else:
                Yfull[l].copy_(dl.y)

    K, W = args.steps, max(3, args.warmup)
    with torch.cuda.stream(stream):
        for _ in range(W):
            step()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as cs:
            e0.record(stream)
            for _ in range(K):
                step()
            e1.record(stream)
            torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    status = S.status()
    if any(status):
        raise RuntimeError(f"device status after the timed region: {status}")
    if rank == 0:
        value = K * L * T / (ms / 1e3)   # every rank served the same tokens
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
                "ms_per_step": ms / K, "higher_is_better": True, "scaling": "strong", "vs_baseline": None,
                "dtype": "int8", "data": "synthetic",
                "config": {"workload": workload_name(cfg, L, T), "tokens": T, "layers": L,
                           "parallelism": f"ep{world}: expert e on rank e % {world}, shared expert on rank 0, "
                                          "partial y gathered and summed in rank order per layer",
                           "us_per_layer": 1e3 * ms / (K * L), "setup_s": S.gen_s},
                "cpu_baseline": None, "e2e": None, "gpu_launches": K * L * (2 if world > 1 else 1),
                "clocks": cs.summary()}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    args = parse()
    import synth
    cfg = synth.CONFIGS[args.config]
    L = args.layers or DEFAULT_LAYERS.get(args.config, cfg.layers)
    rank, world, local = rank_env()
    if args.impl == "reference":
        return run_reference(args, cfg, L, rank, world)

    import torch
    import torch.distributed as dist
    from quantized_routed_expert_router_gb300 import _build
    _build.build()

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    T = args.tokens
    stream = torch.cuda.Stream(device=dev)
    peak, peak_src = peaks()

    if args.split == "experts":
        return run_expert_parallel(args, cfg, L, T, rank, world, local, dev, stream, peak, peak_src)

    # ---- workload: L distinct layers, each rank its own tokens (seed offset)
    keep = 2 if (world == 1 and not args.no_cpu) else 0
    S = Stack(cfg, L, T, rank_seed(args.seed, rank), dev, stream, not args.no_overlap, keep_host=keep)
    layers, X, Y = S.layers, S.X, S.Y
    bytes_l, step_bytes = S.bytes_l, S.step_bytes
    graphs = S.graphs

    K, W = args.steps, max(3, args.warmup)
    with ClockSampler(local) as cs:
        ms = timed(graphs["step"], K, W, stream, world, dev)
    clocks = cs.summary()
    status = S.status()
    if any(status):
        raise RuntimeError(f"device status after the timed region: {status}")
    K3 = max(3, K // 4)
    ms_three = timed(graphs["three"], K3, W, stream, world, dev)
    ms_ffn = timed(graphs["ffn"], K3, W, stream, world, dev)

    # ---- end to end through the public API: pinned H2D of every layer's input,
    # the captured public-API calls, D2H of every layer's y, per step
    e2e = None
    if not args.no_e2e:
        xs = torch.empty((L, T, cfg.H), dtype=torch.float32).pin_memory()
        ys = torch.empty((L, T, cfg.H), dtype=torch.float32).pin_memory()
        xs.copy_(X.cpu())
        ke = max(1, min(K, 500))
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            for _ in range(ke):
                X.copy_(xs, non_blocking=True)
                graphs["step"].replay()
                ys.copy_(Y, non_blocking=True)
                stream.synchronize()
        dt = max_over_ranks(time.perf_counter() - t0, world, dev)
        e2e = {"value": job_throughput(world, ke, L, T, dt), "unit": UNIT, "h2d_bytes_per_step": L * T * cfg.H * 4,
               "d2h_bytes_per_step": L * T * cfg.H * 4, "steps": ke,
               "mode": "pinned H2D + graph replay of the public C-ABI calls + D2H + stream sync, wall clock"}

    # ---- further workloads, reported beside the main line (not the headline)
    also = {}
    for name in [a for a in args.also.split(",") if a and a != "none" and a != args.config]:
        c2 = synth.CONFIGS[name]
        S2 = Stack(c2, DEFAULT_LAYERS.get(name, c2.layers), 1, rank_seed(args.seed, rank), dev, stream,
                   not args.no_overlap)
        also[name] = side_figures(S2, K, W, stream, world, dev, peak)
        del S2
        torch.cuda.empty_cache()

    value = job_throughput(world, K, L, T, ms / 1e3)
    launch_ms = ms / (K * L)
    achieved = (step_bytes / L) / (launch_ms / 1e3) / 1e9
    traffic = traffic_record(f"layer_kernel:{cfg.name}:T{T}")
    cpu = None
    if world == 1 and not args.no_cpu and S.host_sample:
        # after every GPU leg, so the host threads disturb no GPU timing
        n1, dt1 = time_oracle(S.host_sample, 1, steps=100000, seconds=4.0)
        C = host_threads()
        n, dt = time_oracle(S.host_sample, C, steps=100000, seconds=6.0)
        cpu = {"value": n * T / dt, "unit": UNIT, "cores": C, "kind": "oracle",
               "sample": f"{n} layer-steps of {cfg.name} (T={T}) on {C} host threads at once over "
                         f"{len(S.host_sample)} seeded layers, scalar C oracle, {dt:.1f} s",
               "single_thread": {"value": n1 * T / dt1, "cores": 1,
                                 "sample": f"{n1} layer-steps on one thread, {dt1:.1f} s"}}
    if rank == 0:
        uniq = [b["unique"] for b in bytes_l]
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int8",   # int8 x int8 -> int32 sub-block dots; fp32 scale combine
            "data": "synthetic",
            "config": {"workload": workload_name(cfg, L, T), "tokens": T, "layers": L,
                       "l2": f"inputs larger than L2: {step_bytes / 1e6:.0f} MB of distinct weights touched "
                             f"per step (L2 129 MB)",
                       "stack_tok_s": world * K * T / (ms / 1e3),
                       "hbm_gbs": step_bytes * K / (ms / 1e3) / 1e9,
                       "hbm_frac_of_measured": step_bytes * K / (ms / 1e3) / 1e9 / peak,
                       "us_per_layer": 1e3 * ms / (K * L),
                       "bytes_per_layer": step_bytes / L, "unique_experts_per_layer": float(np.mean(uniq)),
                       "path": "moe_layer_forward (one launch per layer)"
                               + ("" if args.no_overlap else ", overlap flag (programmatic dependent launch)"),
                       "three_call_us_per_layer": 1e3 * ms_three / (K3 * L),
                       "three_call_ffn_us_per_layer": 1e3 * ms_ffn / (K3 * L),
                       "setup_s": S.gen_s,
                       "also": also},
            "roofline": {"bound": "hbm", "kernel": "layer_kernel (moe_layer_forward)",
                         "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "peak_source": peak_src, "traffic": traffic,
                         "algorithmic_bytes_per_launch": step_bytes / L,
                         "launch_us": 1e3 * launch_ms},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": K * L,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
