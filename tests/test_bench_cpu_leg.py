"""The benchmark's CPU legs time the oracle on several host threads at once:
the step count is exact and concurrent calls give the serial results bit for
bit (the oracle keeps no global state)."""
import threading

import numpy as np

import bench
import oracle
import synth


def _layers():
    cfg = synth.shrink(synth.CONFIGS["a3b"], H=512, I=256, E=8, k=3, shared_I=256)
    return [synth.make_layer(cfg, l, T=2) for l in range(2)]


def test_time_oracle_counts_every_thread_step():
    layers = _layers()
    n, dt = bench.time_oracle(layers, 3, steps=4)
    assert n == 12 and dt > 0
    n, dt = bench.time_oracle(layers, 2, seconds=0.2)
    assert n >= 2 and dt >= 0.2
    assert bench.host_threads() >= 1


def test_concurrent_oracle_calls_match_serial():
    layers = _layers()
    serial = [oracle.layer_forward(L) for L in layers]
    got = [None] * 8

    def run(i):
        got[i] = oracle.layer_forward(layers[i % 2])

    pool = [threading.Thread(target=run, args=(i,)) for i in range(8)]
    for t in pool:
        t.start()
    for t in pool:
        t.join()
    for i, r in enumerate(got):
        want = serial[i % 2]
        assert np.array_equal(r["ids"], want["ids"])
        assert np.array_equal(r["w"], want["w"])
        assert np.array_equal(r["y"], want["y"])


def test_time_oracle_surfaces_errors():
    cfg = synth.shrink(synth.CONFIGS["tiny"], E=4, k=2)
    bad = synth.make_layer(cfg, 0, T=1)
    bad.x = bad.x[:, :100]        # a width the quantiser refuses
    try:
        bench.time_oracle([bad], 2, steps=1)
    except ValueError:
        return
    raise AssertionError("an error inside a timing thread was swallowed")
