"""GPU layout kernels through the C ABI against the oracle: bit exact."""
import numpy as np
import pytest

import oracle
import synth
from tests import _helpers as H

pytestmark = pytest.mark.gpu


def _w(mode, P, S_l, R, Hq, Hkv, D, dtype, B=1):
    return synth.Workload("t", B=B, P=P, S_l=S_l, R=R if mode != "none" else 0, mode=mode, Hq=Hq, Hkv=Hkv, D=D,
                          dtype=dtype, std_q=1.0, std_kv=1.0, seed=P * 100 + S_l)


CASES = [
    _w(mode, P, S_l, R, Hq, Hkv, D, dt, B)
    for mode in ("none", "prefix", "suffix", "kv_prefix")
    for (P, S_l, R, Hq, Hkv, D, dt, B) in (
        (1, 37, 5, 4, 2, 64, "bf16", 2),
        (2, 56, 16, 4, 4, 64, "bf16", 1),
        (3, 129, 130, 6, 3, 128, "bf16", 2),
        (4, 200, 17, 40, 40, 128, "bf16", 1),
        (8, 33, 9, 40, 8, 128, "e4m3", 1),
        (4, 64, 128, 8, 4, 128, "e4m3", 2),
        # runs wider than one 24 KB block buffer (P = 1, 128 heads of 256 B)
        # take the row gathers in both directions; with P = 2 the gathered
        # runs fit (16 KB) but the 32 KB output rows of to_seq do not
        (1, 70, 9, 128, 128, 128, "bf16", 1),
        (2, 90, 11, 128, 16, 128, "bf16", 2),
    )
]


def _ids(w):
    return "%s-P%d-S%d-R%d-H%d.%d-D%d-%s-B%d" % (w.mode, w.P, w.S_l, w.R, w.Hq, w.Hkv, w.D, w.dtype, w.B)


@pytest.mark.parametrize("w", CASES, ids=_ids)
def test_to_heads_bit_exact(w):
    import torch
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    qh, kh, vh = H.empty_heads(plan, w, H.in_dtype(w))
    for t in qh + kh + vh:
        t.view(torch.uint8).fill_(0xA5)
    plan.to_heads(d["q"], d["k"], d["v"], qh, kh, vh)
    torch.cuda.synchronize()
    want = H.oracle_heads(w, data)
    for got_list, want_list in zip((qh, kh, vh), want):
        for g, wnt in zip(got_list, want_list):
            np.testing.assert_array_equal(H.bits(g).view(wnt.dtype) if wnt.dtype == np.uint16 else H.bits(g), wnt)
    # k and v alone (q skipped): the same bytes
    for t in kh + vh:
        t.view(torch.uint8).fill_(0x5A)
    plan.to_heads(None, d["k"], d["v"], None, kh, vh)
    torch.cuda.synchronize()
    for got_list, want_list in zip((kh, vh), want[1:]):
        for g, wnt in zip(got_list, want_list):
            np.testing.assert_array_equal(H.bits(g).view(wnt.dtype) if wnt.dtype == np.uint16 else H.bits(g), wnt)


@pytest.mark.parametrize("w", CASES, ids=_ids)
def test_to_seq_bit_exact_and_round_trip(w):
    import torch
    plan = H.make_plan(w)
    rng = np.random.default_rng(w.seed)
    nq = plan.heads_rows_q
    oh_np = [rng.integers(0, 1 << 16, size=(w.B, nq, w.Hq // w.P, w.D), dtype=np.uint16) for _ in range(w.P)]
    oh = [torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16) for a in oh_np]
    o = [torch.zeros((w.B, plan.shard_rows_q, w.Hq, w.D), dtype=torch.bfloat16, device="cuda") for _ in range(w.P)]
    plan.to_seq(oh, o)
    torch.cuda.synchronize()
    want = oracle.to_seq(H.oracle_shape(w), oh_np)
    for g, wnt in zip(o, want):
        np.testing.assert_array_equal(H.bits(g).view(np.uint16), wnt)
    # round trip of bf16 q-shaped shards with consistent replicated rows
    if w.dtype == "bf16":
        data = synth.generate(w)
        d = H.dev_inputs(w, data)
        qh, _, _ = H.empty_heads(plan, w, torch.bfloat16)
        plan.to_heads(d["q"], None, None, qh, None, None)
        back = [torch.empty_like(x) for x in d["q"]]
        plan.to_seq(qh, back)
        torch.cuda.synchronize()
        for a, b in zip(d["q"], back):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_to_heads_full_size_wan14b():
    """Full Wan-14B-like shapes (3 x 4 x [1, 7332, 40, 128] bf16): bit exact."""
    import torch
    w = synth.WORKLOADS["wan14b"]
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    qh, kh, vh = H.empty_heads(plan, w, torch.bfloat16)
    plan.to_heads(d["q"], d["k"], d["v"], qh, kh, vh)
    torch.cuda.synchronize()
    want = H.oracle_heads(w, data)
    for got_list, want_list in zip((qh, kh, vh), want):
        for g, wnt in zip(got_list, want_list):
            assert np.array_equal(H.bits(g).view(np.uint16), wnt)
