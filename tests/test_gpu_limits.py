"""The largest rank count a plan takes (16 virtual ranks, where the segment
table, the host path's chunk list and its copy-kernel task table are full):
layout bit exact against the oracle, the fused and staged paths against the
oracle and bit-identical to each other, the pipelined and host-buffer paths
bit-identical to the fused one.  (One rank more is refused: a CPU test.)"""
import numpy as np
import pytest

import synth
from tests import _helpers as H

pytestmark = pytest.mark.gpu


def _w(name, mode, S_l, R, Hq, Hkv, D, dtype="bf16", B=1, valid=None, lens=None, seed=81):
    return synth.Workload(name, B=B, P=16, S_l=S_l, R=R if mode != "none" else 0, mode=mode, Hq=Hq, Hkv=Hkv,
                          D=D, dtype=dtype, std_q=1.0, std_kv=1.0, seed=seed, valid=valid, lens=lens)


CASES = [
    _w("p16-prefix-d64", "prefix", 40, 24, 16, 16, 64, valid=((0, 10), (24, 24 + 640))),
    _w("p16-gqa-suffix", "suffix", 33, 20, 32, 16, 128, B=2),
    _w("p16-fp8-kvprefix", "kv_prefix", 29, 48, 16, 16, 128, dtype="e4m3"),
    _w("p16-uneven", "prefix", 0, 16, 16, 16, 128, lens=tuple([1, 130] + [7 * i + 3 for i in range(14)]),
       valid=((0, 9), (16, 16 + 131 + sum(7 * i + 3 for i in range(14))))),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_sixteen_ranks_layout_and_paths(w):
    import torch
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    # layout, bit exact
    qh, kh, vh = H.empty_heads(plan, w, H.in_dtype(w))
    plan.to_heads(d["q"], d["k"], d["v"], qh, kh, vh)
    torch.cuda.synchronize()
    for got_list, want_list in zip((qh, kh, vh), H.oracle_heads(w, data)):
        for g, want in zip(got_list, want_list):
            np.testing.assert_array_equal(H.bits(g).view(want.dtype), want)
    # fused against the oracle; staged bit-identical to fused
    o = H.run_fused(plan, w, d)
    oh, o_staged = H.run_staged(plan, w, d)
    torch.cuda.synchronize()
    H.assert_written(o)
    _, want = H.oracle_path(w, data)
    for p in range(w.P):
        ok, err, nbad = H.within(H.host_f64(o[p]), want[p], H.TOL[w.dtype])
        assert ok, "shard %d: max err %g (%d)" % (p, err, nbad)
        assert torch.equal(o[p].view(torch.int16), o_staged[p].view(torch.int16))


@pytest.mark.parametrize("w", CASES[:2], ids=lambda w: w.name)
def test_sixteen_ranks_pipelined_and_host(w):
    import torch
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    want = H.run_fused(plan, w, d)
    qh, kh, vh = H.empty_heads(plan, w, H.in_dtype(w))
    oh = [torch.empty((w.B, plan.heads_rows_q, w.Hq // w.P, w.D), dtype=torch.bfloat16, device="cuda")
          for _ in range(w.P)]
    o = [torch.full_like(x, float("nan")) for x in want]
    plan.pipelined_attention(d["q"], d["k"], d["v"], qh, kh, vh, oh, o, key_mask=d["key_mask"])
    torch.cuda.synchronize()
    for a, b in zip(o, want):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    # host buffers: 16 shards x (q, k, v) fill the first chunk's task table
    pin = {n: [torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu()) for t in d[n]]
           for n in ("q", "k", "v")}
    qs = [torch.zeros_like(x) for x in d["q"]]
    ks = [torch.zeros_like(x) for x in d["k"]]
    vs = [torch.zeros_like(x) for x in d["v"]]
    o2 = [torch.full_like(x, float("nan")) for x in want]
    o_host = [torch.full(x.shape, float("nan"), dtype=x.dtype, pin_memory=True) for x in want]
    plan.sp_attention_host(pin["q"], pin["k"], pin["v"], qs, ks, vs, o2, o_host, key_mask=d["key_mask"])
    torch.cuda.current_stream().synchronize()
    assert plan.sync_status() == 0
    for p in range(w.P):
        assert torch.equal(o_host[p].view(torch.int16), want[p].cpu().view(torch.int16)), p
        assert torch.equal(qs[p].view(torch.int16), d["q"][p].view(torch.int16))
        assert torch.equal(ks[p].view(torch.int16), d["k"][p].view(torch.int16))
        assert torch.equal(vs[p].view(torch.int16), d["v"][p].view(torch.int16))

