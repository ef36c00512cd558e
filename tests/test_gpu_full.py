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


def test_full_size_ring_one_launch_wan14b():
    """uly_ring_attention at full size (wan14b, 4 virtual ring ranks, key
    chunks of equal rows): rank 0's walk starts at key 0 and equals the
    plain call bit for bit; every rank's first and last row of every
    128-row Q tile (one local head each) against the oracle; the whole output
    within tolerance of the plain call."""
    import torch
    w = synth.WORKLOADS["wan14b"]
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    qh, kh, vh = H.empty_heads(plan, w, H.in_dtype(w))
    plan.to_heads(d["q"], d["k"], d["v"], qh, kh, vh)
    shape_o = (w.B, plan.heads_rows_q, w.Hq // w.P, w.D)
    kw = dict(key_ranges=d["key_ranges"], head_groups=w.head_groups)
    op = [torch.full(shape_o, float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(w.P)]
    plan.attention(qh, kh, vh, op, **kw)
    nk = plan.heads_rows_kv
    bounds = [int(x) for x in np.linspace(0, nk, w.P + 1)]
    orng = [torch.full(shape_o, float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(w.P)]
    plan.ring_attention(qh, kh, vh, orng, bounds, **kw)
    torch.cuda.synchronize()
    assert plan.sync_status() == 0
    H.assert_written(orng)
    assert torch.equal(orng[0].view(torch.int16), op[0].view(torch.int16))
    tol = H.TOL[w.dtype]
    for r in range(w.P):
        a, b = orng[r].double(), op[r].double()
        assert bool(((a - b).abs() <= tol * (1 + b.abs())).all()), "rank %d" % r
    heads = H.oracle_heads(w, data)
    rng = np.random.default_rng(1)
    hl = w.Hq // w.P
    nq = plan.heads_rows_q
    rows = sorted({n for t0 in range(0, nq, 128) for n in (t0, min(t0 + 128, nq) - 1)})
    checked = 0
    for r in range(w.P):
        sel = np.array([[b, n, int(rng.integers(hl))] for b in range(w.B) for n in rows], dtype=np.int32)
        ref = H.oracle_rank_attention(w, data, heads, r, sel=sel)
        host = orng[r].float().cpu().numpy()
        got = np.stack([host[b, n, j] for b, n, j in sel]).astype(np.float64)
        ok, err, nbad = H.within(got, ref, tol)
        assert ok, "rank %d: max err %g (%d)" % (r, err, nbad)
        checked += len(sel)
    print("ring one launch: %d (row, head) outputs against the oracle" % checked)
