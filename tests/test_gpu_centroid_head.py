"""GPU parity of the centroid-masked LM head (oxinfer 0.0.1, src/drafter.rs, end of
`Drafter::step`): centroid logits, top-k centroids in rank order, the exact logits
of their clusters' tokens, and the first maximum.

Where floating point decides an index (the selection, the winner), exact inputs
(small integers, every sum exact in fp32 and f64) must give exactly the oracle's
decision, ties included; random inputs must give a valid decision: every choice
within the logit bar of the oracle's.
"""
import numpy as np
import pytest

import oracle
import workloads as wl
from gpu_util import lib

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sil():
    import torch
    torch.cuda.set_device(0)
    return lib()


def _run(sil, inp: wl.HeadInputs, top_k, x=None, ordering=None):
    import torch
    k = min(top_k, inp.n_cent)
    per = inp.vocab // inp.n_cent
    cw = sil.upload_weight("bf16", inp.centroids, inp.n_cent, inp.h)
    ew = sil.upload_weight("bf16", inp.embed, inp.vocab, inp.h)
    xd = torch.from_numpy(inp.x if x is None else x).cuda()
    od = torch.from_numpy((inp.ordering if ordering is None else ordering).view(np.int32)).cuda()
    tok = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    score = torch.full((1,), float("nan"), device="cuda")
    sel = torch.full((k,), -1, dtype=torch.int32, device="cuda")
    scores = torch.full((k * per,), float("nan"), device="cuda")
    sil.centroid_head(xd, cw, ew, od, top_k, tok, score, sel, scores)
    torch.cuda.synchronize()
    cw.free()
    ew.free()
    return {"token": int(tok.cpu().view(torch.int32)[0]) & 0xFFFFFFFF, "score": float(score.cpu()[0]),
            "sel": sel.cpu().numpy().astype(np.int64), "scores": scores.cpu().numpy(), "per": per}


def _inputs(h, vocab, n_cent, x, cw, ew, order):
    import torch
    enc = lambda a: wl.encode_bf16(wl.bf16_bits(torch.from_numpy(np.asarray(a, dtype=np.float32))))
    return wl.HeadInputs(h, vocab, n_cent, np.asarray(x, dtype=np.float32), enc(cw), enc(ew),
                         np.asarray(order, dtype=np.uint32))


def _check_valid(inp, top_k, got):
    """Random inputs: the GPU's selection, logits and winner are valid under the bar."""
    k = min(top_k, inp.n_cent)
    per = got["per"]
    cl, sel_ref = oracle.default().centroid_select(inp.centroids, inp.n_cent, inp.h, inp.x, k)
    _, mag_c = oracle.linear("bf16", inp.centroids, inp.n_cent, inp.h, inp.x.reshape(1, -1))
    tol_c = oracle.tolerance(mag_c[0])
    sel = got["sel"]
    assert len(set(sel.tolist())) == k and sel.min() >= 0 and sel.max() < inp.n_cent
    kth = cl[sel_ref[-1]]
    # every chosen centroid is within the bar of the k-th best, and rank order holds within it
    assert np.all(cl[sel] >= kth - tol_c[sel] - tol_c[sel_ref[-1]])
    assert np.all(cl[sel[:-1]] >= cl[sel[1:]] - tol_c[sel[:-1]] - tol_c[sel[1:]])
    # the logits of the chosen clusters, element by element
    sc_ref, mag = oracle.default().cluster_scores(inp.embed, inp.vocab, inp.h, inp.ordering, per, sel, inp.x)
    ok, worst, idx = oracle.check(got["scores"], sc_ref, mag)
    assert ok, (worst, idx)
    # the winner: a first maximum of the GPU's own logits, and a maximum of the oracle's within the bar
    pos = int(np.argmax(got["scores"]))
    assert got["token"] == int(inp.ordering[sel[pos // per] * per + pos % per])
    assert got["score"] == got["scores"][pos]
    tol = oracle.tolerance(mag)
    best = int(np.argmax(sc_ref))
    assert sc_ref[pos] >= sc_ref[best] - tol[pos] - tol[best]


def test_worked_example(sil):
    # the oracle's hand-built example: logits 1, 2, 3, 1 (tie c0 / c3), tied token scores
    x = np.zeros(8, np.float32)
    x[:2] = (1, 2)
    cw = np.zeros((4, 8), np.float32)
    cw[:, :2] = [(1, 0), (0, 1), (3, 0), (1, 0)]
    ew = np.zeros((8, 8), np.float32)
    ew[:, :2] = [(0, 0), (-1, 0), (10, 0), (1, 1), (10, 0), (4, 0), (2, 0.5), (0, 1.5)]
    inp = _inputs(8, 8, 4, x, cw, ew, [5, 1, 7, 0, 3, 6, 2, 4])
    for k, sel, tok, score in ((3, [2, 1, 0], 5, 4.0), (2, [2, 1], 3, 3.0), (4, [2, 1, 0, 3], 2, 10.0),
                               (9, [2, 1, 0, 3], 2, 10.0)):
        got = _run(sil, inp, k)
        assert list(got["sel"]) == sel and got["token"] == tok and got["score"] == score, (k, got)
    got = _run(sil, inp, 3)
    assert list(got["scores"]) == [3.0, 3.0, 3.0, 0.0, 4.0, -1.0]


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("top_k", [1, 5, 40])
def test_integer_exact_ties(sil, seed, top_k):
    # small integers: every logit is exact on both sides, so the GPU must take exactly
    # the oracle's decisions, including its tie rules (lower centroid index, first maximum)
    rng = np.random.default_rng(seed)
    h, n_cent, per = 64, 48, 8
    vocab = n_cent * per
    x = rng.integers(-1, 3, size=h)
    cw = rng.integers(-1, 2, size=(n_cent, h))
    ew = rng.integers(-1, 2, size=(vocab, h))
    inp = _inputs(h, vocab, n_cent, x, cw, ew, rng.permutation(vocab))
    ref = oracle.centroid_head(inp.centroids, n_cent, inp.embed, vocab, h, inp.ordering, inp.x, top_k)
    got = _run(sil, inp, top_k)
    assert list(got["sel"]) == list(ref["sel"])
    assert np.array_equal(got["scores"].astype(np.float64), ref["scores"])
    assert got["token"] == ref["token"] and got["score"] == ref["score"]


@pytest.mark.parametrize("n_cent,top_k", [(4096, 32), (16384, 32), (700, 31), (33, 32), (4096, 33)])
def test_equal_logits_take_the_lowest_indices(sil, n_cent, top_k):
    # every centroid logit equal: the k lowest indices win, in order.  For k <= 32 this is
    # the in-kernel selection's worst case (hundreds of keys pass its first threshold);
    # k = 33 takes the separate selection kernel
    rng = np.random.default_rng(n_cent + top_k)
    h, per = 16, 2
    vocab = n_cent * per
    x = rng.integers(-1, 3, size=h)
    cw = np.ones((n_cent, h))
    ew = rng.integers(-2, 3, size=(vocab, h))
    inp = _inputs(h, vocab, n_cent, x, cw, ew, rng.permutation(vocab))
    ref = oracle.centroid_head(inp.centroids, n_cent, inp.embed, vocab, h, inp.ordering, inp.x, top_k)
    got = _run(sil, inp, top_k)
    assert list(got["sel"]) == list(range(min(top_k, n_cent))) == list(ref["sel"])
    assert np.array_equal(got["scores"].astype(np.float64), ref["scores"])
    assert got["token"] == ref["token"] and got["score"] == ref["score"]


@pytest.mark.parametrize("h,top_k", [(104, 8), (40, 40), (8, 3), (2568, 32), (4104, 5)])
def test_ragged_head_widths(sil, h, top_k):
    # widths that are a multiple of 8 (bf16 weights need it) but of no larger power of
    # two: a row ends mid-way through a lane's 16-byte vectors; integer data keeps every
    # decision exact (4104 > 4096 takes the row loop that does not hold a row in registers)
    rng = np.random.default_rng(h)
    n_cent, per = 48, 4
    vocab = n_cent * per
    x = rng.integers(-1, 3, size=h)
    cw = rng.integers(-1, 2, size=(n_cent, h))
    ew = rng.integers(-1, 2, size=(vocab, h))
    inp = _inputs(h, vocab, n_cent, x, cw, ew, rng.permutation(vocab))
    ref = oracle.centroid_head(inp.centroids, n_cent, inp.embed, vocab, h, inp.ordering, inp.x, top_k)
    got = _run(sil, inp, top_k)
    assert list(got["sel"]) == list(ref["sel"])
    assert np.array_equal(got["scores"].astype(np.float64), ref["scores"])
    assert got["token"] == ref["token"] and got["score"] == ref["score"]


def test_nan_centroid_and_no_winner(sil):
    # a NaN centroid logit ranks last; when every logit is NaN the token is 0 and the score -inf
    h, n_cent, per = 16, 4, 2
    x = np.ones(h, np.float32)
    cw = np.ones((n_cent, h), np.float32)
    cw[1, 0] = np.nan
    ew = np.ones((n_cent * per, h), np.float32)
    inp = _inputs(h, n_cent * per, n_cent, x, cw, ew, np.arange(n_cent * per))
    got = _run(sil, inp, 4)
    assert list(got["sel"]) == [0, 2, 3, 1]
    ew[:] = np.nan
    inp = _inputs(h, n_cent * per, n_cent, x, cw, ew, np.arange(n_cent * per))
    got = _run(sil, inp, 2)
    assert got["token"] == 0 and got["score"] == -np.inf


@pytest.mark.parametrize("h,n_cent,per,top_k", [(512, 256, 16, 7), (1024, 100, 3, 100), (256, 1, 64, 4),
                                                (2048, 4000, 2, 33), (136, 16384, 1, 300)])
def test_random_valid(sil, h, n_cent, per, top_k):
    inp = wl.make_head_inputs(h, n_cent * per, n_cent, seed=h + n_cent)
    got = _run(sil, inp, top_k)
    _check_valid(inp, top_k, got)


def test_full_size(sil):
    c = wl.CENTROID_HEAD
    inp = wl.make_head_inputs(c.h, c.vocab, c.n_cent, seed=0)
    got = _run(sil, inp, c.top_k)
    _check_valid(inp, c.top_k, got)


def test_repeat_calls_and_state_reset(sil):
    # the per-stream best key and counter return to zero: repeated calls agree, and a
    # different x gives that x's answer
    inp = wl.make_head_inputs(512, 1024, 64, seed=9)
    a = _run(sil, inp, 8)
    b = _run(sil, inp, 8)
    assert a["token"] == b["token"] and np.array_equal(a["scores"], b["scores"])
    x2 = wl.make_x(1, 512, seed=10)[0]
    inp2 = wl.HeadInputs(inp.h, inp.vocab, inp.n_cent, x2, inp.centroids, inp.embed, inp.ordering)
    _check_valid(inp2, 8, _run(sil, inp2, 8))


def test_out_of_range_ordering_is_flagged(sil):
    # an ordering entry >= vocab is skipped (never read, never wins) and reported once
    inp = wl.make_head_inputs(64, 32, 4, seed=3)
    order = inp.ordering.copy()
    order[:8] = 1000                         # all of cluster 0
    cen = np.zeros((4, 64), np.float32)
    cen[0, :] = 1.0                          # make cluster 0 rank first
    inp = _inputs(64, 32, 4, inp.x if inp.x.sum() > 0 else -inp.x, cen, np.zeros((32, 64)), order)
    got = _run(sil, inp, 2)
    assert got["sel"][0] == 0 and np.all(np.isnan(got["scores"][:8]))
    with pytest.raises(sil.ILError) as ei:
        sil.check_device_status()
    assert ei.value.code == -1
    sil.check_device_status()                # cleared


def test_rejects(sil):
    import torch
    inp = wl.make_head_inputs(64, 64, 8, seed=1)
    cw = sil.upload_weight("bf16", inp.centroids, 8, 64)
    ew = sil.upload_weight("bf16", inp.embed, 64, 64)
    q8 = sil.upload_weight("q8", wl.make_batch(64, (64,), 1, "q8").jobs[0][1], 64, 64)
    odd = sil.upload_weight("bf16", wl.make_batch(64, (60,), 1, "bf16").jobs[0][1], 60, 64)
    x = torch.from_numpy(inp.x).cuda()
    od = torch.from_numpy(inp.ordering.view(np.int32)).cuda()
    tok = torch.zeros(1, dtype=torch.int32, device="cuda")
    before = sil.get_stats()["launches"]
    for args, code in [((x, cw, q8, od, 2, tok), -3), ((x, q8, ew, od, 2, tok), -3),
                       ((x[:32], cw, ew, od, 2, tok), -2), ((x, cw, odd, od, 2, tok), -2),
                       ((x, cw, ew, od, 0, tok), -1)]:
        with pytest.raises(sil.ILError) as ei:
            sil.centroid_head(*args)
        assert ei.value.code == code, args
    assert sil.get_stats()["launches"] == before
    for w in (cw, ew, q8, odd):
        w.free()
