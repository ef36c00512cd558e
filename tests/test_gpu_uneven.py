"""Uneven shards (a different number of image rows per shard, the seq_lens
of sglang's varlen all-to-all): layout bit exact against the oracle, and
attention through the staged, fused and pipelined paths against the oracle
and bit-identical to each other, for every replicated-row mode."""
import numpy as np
import pytest

import oracle
import synth
from tests import _helpers as H

pytestmark = pytest.mark.gpu


def _w(name, mode, lens, R, Hq, Hkv, D, dtype="bf16", B=1, valid=None, seed=61):
    return synth.Workload(name, B=B, P=len(lens), S_l=0, R=R if mode != "none" else 0, mode=mode, Hq=Hq, Hkv=Hkv,
                          D=D, dtype=dtype, std_q=1.0, std_kv=1.0, seed=seed, valid=valid, lens=tuple(lens))


CASES = [
    _w("uneven-prefix", "prefix", (300, 45, 129, 200), 150, 8, 8, 128, B=2, valid=((0, 60), (150, 150 + 674))),
    _w("uneven-suffix-fp8", "suffix", (130, 257), 100, 8, 8, 128, dtype="e4m3", valid=((0, 387 + 40),)),
    _w("uneven-kvprefix-gqa", "kv_prefix", (256, 10, 300), 64, 12, 3, 128, B=2),
    _w("uneven-none-d64", "none", (1, 127, 128, 129), 0, 8, 4, 64),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_uneven_layout_bit_exact(w):
    import torch
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    for p in range(w.P):
        assert plan.shard_rows(p) == w.rows_shard(False, p)
        assert plan.shard_rows(p, True) == w.rows_shard(True, p)
    qh, kh, vh = H.empty_heads(plan, w, H.in_dtype(w))
    plan.to_heads(d["q"], d["k"], d["v"], qh, kh, vh)
    torch.cuda.synchronize()
    want = H.oracle_heads(w, data)
    for got_list, want_list in zip((qh, kh, vh), want):
        for g, wnt in zip(got_list, want_list):
            np.testing.assert_array_equal(H.bits(g).view(wnt.dtype), wnt)
    rng = np.random.default_rng(7)
    oh_np = [rng.integers(0, 1 << 16, size=(w.B, plan.heads_rows_q, w.Hq // w.P, w.D), dtype=np.uint16)
             for _ in range(w.P)]
    oh = [torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16) for a in oh_np]
    o = [torch.zeros((w.B, plan.shard_rows(p), w.Hq, w.D), dtype=torch.bfloat16, device="cuda") for p in range(w.P)]
    plan.to_seq(oh, o)
    torch.cuda.synchronize()
    for g, wnt in zip(o, oracle.to_seq(H.oracle_shape(w), oh_np)):
        np.testing.assert_array_equal(H.bits(g).view(np.uint16), wnt)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_uneven_attention_paths(w):
    import torch
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    oh, o = H.run_staged(plan, w, d)
    of = H.run_fused(plan, w, d)
    qh, kh, vh = H.empty_heads(plan, w, H.in_dtype(w))
    ohp = [torch.empty_like(x) for x in oh]
    op = [torch.full_like(x, float("nan")) for x in of]
    plan.pipelined_attention(d["q"], d["k"], d["v"], qh, kh, vh, ohp, op, key_mask=d["key_mask"],
                             q_scale=d["q_scale"], k_scale=d["k_scale"], v_scale=d["v_scale"])
    torch.cuda.synchronize()
    assert plan.sync_status() == 0
    _, want = H.oracle_path(w, data)
    for p in range(w.P):
        ok, err, nbad = H.within(H.host_f64(o[p]), want[p], H.TOL[w.dtype])
        assert ok, "shard %d: max err %g (%d)" % (p, err, nbad)
        assert torch.equal(o[p].view(torch.int16), of[p].view(torch.int16))
        assert torch.equal(o[p].view(torch.int16), op[p].view(torch.int16))
