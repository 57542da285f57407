"""World-size-2 runs of the multi-rank host logic on CPU ranks (gloo).

Two things are covered:

- the benchmark's data-parallel rank logic: the rank environment, distinct
  token seeds per rank, max-over-ranks timing and the job-wide throughput;
- the expert-ownership split of one layer, through the benchmark's
  expert-parallel host logic (``bench.expert_owner_mask``,
  ``bench.rank_order_sum``): rank r owns the experts with e % 2 == r and
  rank 0 owns the shared expert; the partial y's are gathered and summed in
  rank order, and the sum must equal the unsplit layer - also with a gated
  shared expert, whose weight applies on rank 0 only.

The split follows the pulsar README's "MoE resolve" passage: a NULL expert
pointer means "not mine", and the per-card partial results are summed. Here
the oracle stands in for each rank's expert FFN; the GPU side of the same
split is covered by the ownership tests of the CUDA path.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        import synth

        r, w, local = bench.rank_env()
        slowest = bench.max_over_ranks(1.5 + rank, w)
        rate = bench.job_throughput(w, steps=10, layers=4, tokens=2, seconds=0.5)

        cfg = synth.shrink(synth.CONFIGS["a3b"], H=512, I=256, E=8, k=3, shared_I=256)
        mine = synth.make_layer(cfg, 0, T=2, seed=bench.rank_seed(0, rank), with_experts=False)
        xs = [torch.zeros(mine.x.shape, dtype=torch.float32) for _ in range(w)]
        dist.all_gather(xs, torch.from_numpy(np.ascontiguousarray(mine.x, dtype=np.float32)))

        errs = []
        owned = bench.expert_owner_mask(cfg.E, rank, w)
        for gated in (False, True):
            c = synth.shrink(cfg, shared_gate=gated)
            layer = synth.make_layer(c, 0, T=2, seed=0)   # the same layer on every rank
            full = oracle.layer_forward(layer)
            part = oracle.expert_ffn(layer, full["xq"], full["ids"], full["w"], owned=owned, shared=(rank == 0),
                                     shared_scale=full["shared_scale"])["y"]
            parts = [torch.zeros(part.shape, dtype=torch.float64) for _ in range(w)]
            dist.all_gather(parts, torch.from_numpy(np.ascontiguousarray(part, dtype=np.float64)))
            y = bench.rank_order_sum([p.numpy() for p in parts])
            errs.append(float(np.max(np.abs(y - full["y"]))) / float(np.max(np.abs(full["y"]))))
        masks = [torch.zeros(cfg.E, dtype=torch.uint8) for _ in range(w)]
        dist.all_gather(masks, torch.from_numpy(owned.astype(np.uint8)))
        cover = sum(m.numpy().astype(int) for m in masks)   # every expert on exactly one rank
        out.put((rank, r, w, local, slowest, rate,
                 bool(np.array_equal(xs[0].numpy(), xs[1].numpy())), max(errs), bool(np.all(cover == 1))))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_rank_logic_and_expert_split():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        res = sorted(out.get(timeout=240) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    for rank, (r, r_env, w, local, slowest, rate, same_x, rel_err, cover) in enumerate(res):
        assert (r, r_env, w, local) == (rank, rank, 2, rank)
        assert slowest == 2.5                         # the slower rank's time on both ranks
        assert rate == 2 * 10 * 4 * 2 / 0.5           # every rank's layer-tokens count
        assert not same_x                             # each rank decodes its own tokens
        assert rel_err <= 1e-12                       # the split sums to the unsplit layer
        assert cover                                  # the ownership masks partition the experts
