"""Full-size workloads, in the launch configuration the benchmark times
(fused uly_sp_attention with the workload's head groups): sampled output
rows against the oracle, computed one by one, and the whole output against
the staged path bit for bit."""
import numpy as np
import pytest

import oracle
import synth
from tests import _helpers as H

pytestmark = pytest.mark.gpu


def _samples(w, plan, n_random=48, seed=0):
    """(shard, b, row, head): first/last rows of every run and random rows."""
    rng = np.random.default_rng(seed)
    rq = plan.shard_rows_q
    rows = {0, rq - 1}
    if w.mode == "prefix":
        rows |= {w.R - 1, w.R, w.R + 127, w.R + 128}
    if w.mode == "suffix":
        rows |= {w.S_l - 1, w.S_l, w.S_l + w.R - 1}
    rows |= {127, 128, 255, 256}
    out = []
    for p in sorted({0, w.P - 1}):
        for row in sorted(x for x in rows if 0 <= x < rq):
            out.append((p, int(rng.integers(w.B)), row, int(rng.integers(w.Hq))))
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
    got = np.stack([o[p][b, row, h].float().cpu().numpy() for (p, b, row, h) in samples]).astype(np.float64)
    ok, err, nbad = H.within(got, ref, H.TOL[w.dtype])
    assert ok, "max err %g, %d values out of tolerance" % (err, nbad)
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
