"""uly_sp_attention_host: shards in page-locked host memory, copied in per
rank chunk, attended and copied out with the copies overlapped.  The host
output must equal uly_sp_attention's on the same inputs bit for bit, and the
device staging must hold the inputs afterwards."""
import numpy as np
import pytest

import synth
from tests import _helpers as H

pytestmark = pytest.mark.gpu


def _w(name, mode, P, S_l, R, Hq, Hkv, D, dtype="bf16", B=1, valid=None, lens=None, seed=71):
    return synth.Workload(name, B=B, P=P, S_l=S_l, R=R if mode != "none" else 0, mode=mode, Hq=Hq, Hkv=Hkv, D=D,
                          dtype=dtype, std_q=1.0, std_kv=1.0, seed=seed, valid=valid, lens=lens)


CASES = [
    synth.WORKLOADS["tiny"],
    _w("prefix-masked", "prefix", 4, 300, 200, 8, 8, 128, valid=((0, 77), (200, 1400))),
    _w("gqa-kvprefix-b2", "kv_prefix", 4, 260, 256, 16, 4, 128, B=2),
    _w("fp8-suffix", "suffix", 8, 150, 140, 16, 16, 128, dtype="e4m3", valid=((0, 1200 + 61),)),
    _w("uneven-d64", "suffix", 3, 0, 45, 6, 3, 64, lens=(100, 1, 333), valid=((0, 300), (400, 479))),
]


def _pinned(ts):
    import torch
    return [torch.empty(t.shape, dtype=t.dtype, pin_memory=True).copy_(t.cpu()) for t in ts]


def _pageable(ts):
    return [t.cpu().clone() for t in ts]


# pinned: the first chunk in and the last chunk out go through the copy
# kernel (mapped page-locked memory); pageable: every copy goes through the
# copy engine; mixed: k in pageable memory, so the first chunk falls back to
# the copy engine while the output still leaves through the kernel.
@pytest.mark.parametrize("mem", ["pinned", "pageable", "mixed"])
@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_host_path_equals_fused(w, mem):
    import torch
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    want = H.run_fused(plan, w, d)
    torch.cuda.synchronize()
    kind = {"pinned": (_pinned, _pinned, _pinned), "pageable": (_pageable, _pageable, _pageable),
            "mixed": (_pinned, _pageable, _pinned)}[mem]
    qh, kh, vh = (f(d[n]) for f, n in zip(kind, ("q", "k", "v")))
    for call in range(2):
        qs = [torch.full_like(x, 0) for x in d["q"]]
        ks = [torch.full_like(x, 0) for x in d["k"]]
        vs = [torch.full_like(x, 0) for x in d["v"]]
        o = [torch.full_like(x, float("nan")) for x in want]
        if mem == "pageable":
            o_host = [torch.full(x.shape, float("nan"), dtype=x.dtype) for x in want]
        else:
            o_host = [torch.full(x.shape, float("nan"), dtype=x.dtype, pin_memory=True) for x in want]
        plan.sp_attention_host(qh, kh, vh, qs, ks, vs, o, o_host, key_mask=d["key_mask"], q_scale=d["q_scale"],
                               k_scale=d["k_scale"], v_scale=d["v_scale"])
        torch.cuda.current_stream().synchronize()
        assert plan.sync_status() == 0
        for p in range(w.P):
            assert torch.equal(o_host[p].view(torch.int16), want[p].cpu().view(torch.int16)), (call, p)
            assert torch.equal(o[p].view(torch.int16), want[p].view(torch.int16))
            for a, b in ((qs[p], d["q"][p]), (ks[p], d["k"][p]), (vs[p], d["v"][p])):
                assert torch.equal(a.view(torch.uint8) if a.dtype == torch.uint8 else a.view(torch.int16),
                                   b.view(torch.uint8) if b.dtype == torch.uint8 else b.view(torch.int16))


def test_host_path_against_oracle():
    import torch
    w = CASES[1]
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    qh, kh, vh = (_pinned(d[n]) for n in ("q", "k", "v"))
    o = [torch.empty((w.B, plan.shard_rows(p), w.Hq, w.D), dtype=torch.bfloat16, device="cuda") for p in range(w.P)]
    o_host = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in o]
    plan.sp_attention_host(qh, kh, vh, [torch.empty_like(x) for x in d["q"]], [torch.empty_like(x) for x in d["k"]],
                           [torch.empty_like(x) for x in d["v"]], o, o_host, key_mask=d["key_mask"])
    torch.cuda.current_stream().synchronize()
    _, want = H.oracle_path(w, data)
    for p in range(w.P):
        ok, err, nbad = H.within(o_host[p].float().numpy().astype(np.float64), want[p], H.TOL[w.dtype])
        assert ok, "shard %d: max err %g (%d)" % (p, err, nbad)


def test_host_path_rejects_bad_arguments():
    import torch
    from ulysses_sequence_attention_uly_gb300 import UlyError
    w = CASES[0]
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    o = H.run_fused(plan, w, d)
    qh, kh, vh = (_pinned(d[n]) for n in ("q", "k", "v"))
    oh = _pinned(o)
    with pytest.raises(ValueError):  # a device tensor where host memory is expected
        plan.sp_attention_host(d["q"], kh, vh, d["q"], d["k"], d["v"], o, oh)
    with pytest.raises(UlyError):  # fp8 scales on a bf16 plan
        plan.sp_attention_host(qh, kh, vh, d["q"], d["k"], d["v"], o, oh, q_scale=torch.ones(4, device="cuda"),
                               k_scale=torch.ones(4, device="cuda"), v_scale=torch.ones(4, device="cuda"))
    assert plan.sync_status() == 0
