"""uly_sp_attention_noalloc through the C ABI: the allocation-free fused call
for callers whose device memory belongs to their own pool and who therefore
cannot let the library call cudaMalloc.  It runs the same kernels as the
plan-based uly_sp_attention, so its output (and its LSE output, when asked
for) must equal that call's bit for bit, on two calls in a row: the second
with other admitted keys, so that a tile table left in the shared scratch by
the first call cannot leak into it.  One case fills the scratch to its limit
of 4096 kv tiles exactly.  Collected last on purpose; it also passes alone."""
import numpy as np
import pytest

import synth
from tests import _helpers as H

pytestmark = pytest.mark.gpu

CASES = [
    (synth.WORKLOADS["tiny"], "sdpa"),
    (synth.Workload("noalloc-prefix", B=2, P=4, S_l=300, R=200, mode="prefix", Hq=8, Hkv=8, D=128, dtype="bf16",
                    std_q=1.0, std_kv=1.0, seed=21, valid=((0, 77), (200, 1400))), "sdpa"),
    (synth.Workload("noalloc-fp8", B=1, P=8, S_l=150, R=140, mode="suffix", Hq=40, Hkv=40, D=128, dtype="e4m3",
                    std_q=1.0, std_kv=1.0, seed=22, valid=((0, 1200 + 61),)), "sdpa"),
    (synth.Workload("noalloc-self", B=2, P=2, S_l=260, R=30, mode="kv_prefix", Hq=8, Hkv=2, D=64, dtype="bf16",
                    std_q=1.0, std_kv=0.7, seed=23, valid=((5, 30), (90, 400))), "self"),
    # B * kv tiles = 4 * (2 shards * 512 tiles) = 4096: the scratch's limit
    (synth.Workload("noalloc-limit", B=4, P=2, S_l=65536, R=0, mode="none", Hq=2, Hkv=2, D=64, dtype="bf16",
                    std_q=1.0, std_kv=1.0, seed=24, valid=((0, 131072 - 61),)), "sdpa"),
]


def _ranges(w, lo, hi):
    """Per-batch key ranges [B, 1, 2]: batch b admits keys [lo + b, hi - b)."""
    import torch
    r = np.array([[[lo + b, hi - b]] for b in range(w.B)], dtype=np.int32)
    return torch.from_numpy(r).cuda()


def _bits(xs):
    import torch
    return [x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32) for x in xs]


@pytest.mark.parametrize("w,rows", CASES, ids=lambda c: c.name if hasattr(c, "name") else str(c))
def test_noalloc_equals_plan_call_twice(w, rows):
    import torch
    import ulysses_sequence_attention_uly_gb300 as uly
    data = synth.generate(w)
    d = H.dev_inputs(w, data)
    plan = H.make_plan(w, masked_rows=rows)
    nk = plan.heads_rows_kv
    # first call: the workload's key mask (or its ranges), with the LSE
    # output; second call: other key ranges, O only
    calls = [dict(key_mask=d["key_mask"], key_ranges=None if d["key_mask"] is not None else d["key_ranges"],
                  lse=True),
             dict(key_mask=None, key_ranges=_ranges(w, 3, nk - 2), lse=False)]
    for call, kw in enumerate(calls):
        ref = [torch.full((w.B, plan.shard_rows_q, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
               for _ in range(w.P)]
        got = [torch.full_like(x, float("nan")) for x in ref]
        lref = lgot = None
        if kw["lse"]:
            lref = [torch.full((w.B, plan.shard_rows_q, w.Hq), float("nan"), dtype=torch.float32, device="cuda")
                    for _ in range(w.P)]
            lgot = [torch.full_like(x, float("nan")) for x in lref]
        args = dict(key_mask=kw["key_mask"], key_ranges=kw["key_ranges"], head_groups=w.head_groups,
                    q_scale=d["q_scale"], k_scale=d["k_scale"], v_scale=d["v_scale"])
        plan.sp_attention(d["q"], d["k"], d["v"], ref, lse=lref, **args)
        uly.sp_attention_noalloc(w.B, w.P, w.S_l, w.R, w.mode, w.Hq, w.Hkv, w.D, d["q"], d["k"], d["v"], got,
                                 dtype=w.dtype, masked_rows=rows, lse=lgot, **args)
        assert uly.noalloc_sync_status() == 0, "call %d: a device wait of the allocation-free call expired" % call
        assert plan.sync_status() == 0
        H.assert_written(ref)
        for a, b in zip(_bits(got), _bits(ref)):
            assert torch.equal(a, b), "call %d: output differs from uly_sp_attention" % call
        if lref is not None:
            for a, b in zip(_bits(lgot), _bits(lref)):
                assert torch.equal(a, b), "call %d: LSE differs from uly_sp_attention" % call
    plan.close()


def test_noalloc_rejects_oversized_shape():
    import torch
    import ulysses_sequence_attention_uly_gb300 as uly
    from ulysses_sequence_attention_uly_gb300 import ULY_ERR_UNSUPPORTED
    # B * ceil(keys / 128) = 2 * 2304 tiles > 4096: rejected before any launch
    # (straight through the C ABI: the binding would already refuse the small
    # stand-in tensors by their shapes; the C call rejects the shape before
    # it looks at any pointer)
    import ctypes
    B, P, S_l, Hq, D = 2, 2, 147456, 2, 128
    t = [torch.empty(16, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    desc = uly._Desc(B, P, S_l, 0, 0, Hq, Hq, D, 0, 0)
    ptrs = (ctypes.c_void_p * P)(*[x.data_ptr() for x in t])
    st = uly.lib().uly_sp_attention_noalloc(ctypes.byref(desc), ptrs, ptrs, ptrs, None, None, 0,
                                            ctypes.c_float(0.125), 0, None, None, None, ptrs, None,
                                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == ULY_ERR_UNSUPPORTED
