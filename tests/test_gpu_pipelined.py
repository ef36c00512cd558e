"""Staged path with head groups pipelined over the copy engines
(uly_pipelined_attention): bit-identical to the fused path and to the
sequential staged path for every head-group count, on shapes with every
replicated-row mode."""
import pytest

import synth
from tests import _helpers as H

pytestmark = pytest.mark.gpu

CASES = [
    synth.Workload("pipe-prefix", B=2, P=4, S_l=300, R=200, mode="prefix", Hq=40, Hkv=40, D=128, dtype="bf16",
                   std_q=1.0, std_kv=1.0, seed=51, valid=((0, 77), (200, 1400))),
    synth.Workload("pipe-suffix-fp8", B=1, P=8, S_l=150, R=140, mode="suffix", Hq=40, Hkv=40, D=128, dtype="e4m3",
                   std_q=1.0, std_kv=1.0, seed=52, valid=((0, 1200 + 61),)),
    synth.Workload("pipe-kvprefix-gqa", B=2, P=4, S_l=260, R=256, mode="kv_prefix", Hq=32, Hkv=8, D=128,
                   dtype="bf16", std_q=1.0, std_kv=0.7, seed=53),
    synth.Workload("pipe-none-d64", B=1, P=2, S_l=333, R=0, mode="none", Hq=12, Hkv=6, D=64, dtype="bf16",
                   std_q=1.0, std_kv=1.0, seed=54),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_pipelined_equals_fused_and_staged(w):
    import torch
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    ref = H.run_fused(plan, w, d, head_groups=1)
    torch.cuda.synchronize()
    H.assert_written(ref)
    hq_l, hkv_l = w.Hq // w.P, w.Hkv // w.P
    for g in [x for x in range(1, 9) if hq_l % x == 0 and hkv_l % x == 0]:
        qh, kh, vh = H.empty_heads(plan, w, H.in_dtype(w))
        oh = [torch.empty((w.B, plan.heads_rows_q, hq_l, w.D), dtype=torch.bfloat16, device="cuda")
              for _ in range(w.P)]
        o = [torch.full_like(x, float("nan")) for x in ref]
        plan.pipelined_attention(d["q"], d["k"], d["v"], qh, kh, vh, oh, o, key_mask=d["key_mask"], head_groups=g,
                                 q_scale=d["q_scale"], k_scale=d["k_scale"], v_scale=d["v_scale"])
        torch.cuda.synchronize()
        assert plan.sync_status() == 0
        for a, b in zip(ref, o):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), "g=%d" % g
