"""Host checks of the seeded input recipes shared by the tests and the benchmark."""
import numpy as np

import workloads as wl


def test_batches_are_deterministic_and_seeded():
    a = wl.make_batch(256, (64, 32), 3, "q4", seed=5)
    b = wl.make_batch(256, (64, 32), 3, "q4", seed=5)
    c = wl.make_batch(256, (64, 32), 3, "q4", seed=6)
    assert np.array_equal(a.x, b.x) and all(np.array_equal(p[1], q[1]) for p, q in zip(a.jobs, b.jobs))
    assert not np.array_equal(a.x, c.x)
    assert a.x.shape == (3, 256) and a.x.dtype == np.float32
    assert [n for _, _, n in a.jobs] == [64, 32]
    assert a.weight_bytes == sum(wl.weight_bytes("q4", n, 256) for n in (64, 32))
    assert a.flops == 2 * 3 * 256 * 96


def test_workload_table():
    names = [w.name for w in wl.WORKLOADS]
    assert len(set(names)) == len(names)
    for w in wl.WORKLOADS:
        assert w.fmts and w.ts and w.batches
        for bt in w.batches:
            for fmt in w.fmts:
                assert bt.n_in % (8 if fmt == "bf16" else 32) == 0
    fused = wl.GATE_UP_FUSED
    assert fused.fused and all(len(bt.n_outs) == 2 and bt.n_outs[0] == bt.n_outs[1] for bt in fused.batches)
    b = wl.make_workload_batch(fused, fused.batches[0], 1, "q8")
    assert b.fused
    assert not wl.make_workload_batch(wl.TINY, wl.TINY.batches[0], 1, "bf16").fused


def test_head_inputs():
    c = wl.HeadConfig("small", 64, 96, 12, 5)
    a = wl.make_head_inputs(c.h, c.vocab, c.n_cent, seed=1)
    b = wl.make_head_inputs(c.h, c.vocab, c.n_cent, seed=1)
    assert np.array_equal(a.ordering, b.ordering) and np.array_equal(a.embed, b.embed)
    assert sorted(a.ordering.tolist()) == list(range(c.vocab))          # a permutation
    assert a.ordering.dtype == np.uint32 and a.x.shape == (c.h,)
    assert a.centroids.size == 2 * c.n_cent * c.h and a.embed.size == 2 * c.vocab * c.h
    full = wl.CENTROID_HEAD
    assert full.vocab % full.n_cent == 0 and full.top_k <= full.n_cent
