"""Full-size workloads, in the launch configuration the benchmark times
(fused uly_sp_attention with the workload's head groups): the first and last
row of every Q tile of every run in every shard (one head per rank) and
random rows against the oracle, computed row by row, and the whole output
against the staged path bit for bit."""
import numpy as np
import pytest

import oracle
import synth
from tests import _helpers as H

pytestmark = pytest.mark.gpu


def _runs_of_shard(w, plan, p):
    """Output rows of shard p as the attention kernel tiles them: the
    replicated rows (prefix: first, suffix: last) and the shard's image rows,
    each a run of its own whose 128-row Q tiles start at the run's start."""
    rq = plan.shard_rows(p)
    if w.mode == "prefix":
        return [(0, w.R), (w.R, rq - w.R)]
    if w.mode == "suffix":
        img = rq - w.R
        return [(0, img), (img, w.R)]
    return [(0, rq)]


def _samples(w, plan, n_random=48, seed=0):
    """(shard, b, row, head) of the rows checked against the oracle: in every
    shard and batch, the first and the last row of every 128-row Q tile of
    every run (the replicated rows' run included, in every shard it is
    written to), hence also the first and the last row of every shard; each
    with one q head of every rank (a different local head for each rank and
    tile); plus n_random random (shard, batch, row, head)."""
    rng = np.random.default_rng(seed)
    hl = w.Hq // w.P
    out = []
    for p in range(w.P):
        for b in range(w.B):
            for start, length in _runs_of_shard(w, plan, p):
                for t0 in range(0, length, 128):
                    for row in sorted({start + t0, start + min(t0 + 128, length) - 1}):
                        for r in range(w.P):
                            out.append((p, b, row, r * hl + int(rng.integers(hl))))
    rq = plan.shard_rows_q
    for _ in range(n_random):
        out.append((int(rng.integers(w.P)), int(rng.integers(w.B)), int(rng.integers(rq)), int(rng.integers(w.Hq))))
    return out


@pytest.mark.parametrize("name", ["wan1.3b", "wan14b", "gqa", "fp8"])
def test_full_size_sampled_and_fused_equals_staged(name):
    import torch
    w = synth.WORKLOADS[name]
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    o = H.run_fused(plan, w, d, head_groups=w.head_groups, mask="ranges" if w.valid else "none")
    torch.cuda.synchronize()
    assert plan.sync_status() == 0
    H.assert_written(o)
    # sampled rows against the oracle
    s = H.oracle_shape(w)
    heads = H.oracle_heads(w, data)
    samples = _samples(w, plan)
    hl = w.Hq // w.P
    by_rank = {}
    for i, (p, b, row, h) in enumerate(samples):
        by_rank.setdefault(h // hl, []).append((i, b, oracle.out_row(s, p, row), h % hl))
    ref = np.zeros((len(samples), w.D))
    for r, items in by_rank.items():
        sel = np.array([[b, n, j] for (_, b, n, j) in items], dtype=np.int32)
        vals = H.oracle_rank_attention(w, data, heads, r, sel=sel)
        for (i, *_), v in zip(items, vals):
            ref[i] = v
    host = [x.float().cpu().numpy() for x in o]
    got = np.stack([host[p][b, row, h] for (p, b, row, h) in samples]).astype(np.float64)
    ok, err, nbad = H.within(got, ref, H.TOL[w.dtype])
    assert ok, "max err %g, %d values out of tolerance (%d rows)" % (err, nbad, len(samples))
    print("%s: %d (row, head) outputs against the oracle, max |err| %.3g" % (name, len(samples), err))
    del heads
    # the whole fused output equals the staged path's
    oh, o_staged = H.run_staged(plan, w, d, head_groups=w.head_groups, mask="ranges" if w.valid else "none")
    torch.cuda.synchronize()
    H.assert_written(oh)
    for a, b in zip(o, o_staged):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # key mask and key ranges give the same bytes
    if w.valid:
        o_mask = H.run_fused(plan, w, d, head_groups=w.head_groups, mask="mask")
        torch.cuda.synchronize()
        for a, b in zip(o, o_mask):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_full_size_head_groups_bit_identical_wan14b():
    import torch
    w = synth.WORKLOADS["wan14b"]
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    whole = H.run_fused(plan, w, d, head_groups=1, mask="ranges")
    torch.cuda.synchronize()
    H.assert_written(whole)
    for g in (2, 5):
        split = H.run_fused(plan, w, d, head_groups=g, mask="ranges")
        torch.cuda.synchronize()
        for a, b in zip(whole, split):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), g
