"""uly_sp_attention_noalloc through the C ABI: the allocation-free fused call
for callers whose device memory belongs to their own pool and who therefore
cannot let the library call cudaMalloc.  Its output must match the plan-based
uly_sp_attention's on two calls in a row (the second with a different key
mask, so a tile table left in the shared scratch by the first call cannot
leak into it).  Collected last on purpose; it also passes alone."""
import pytest

import synth
from tests import _helpers as H

pytestmark = pytest.mark.gpu

CASES = [
    synth.WORKLOADS["tiny"],
    synth.Workload("noalloc-prefix", B=2, P=4, S_l=300, R=200, mode="prefix", Hq=8, Hkv=8, D=128, dtype="bf16",
                   std_q=1.0, std_kv=1.0, seed=21, valid=((0, 77), (200, 1400))),
    synth.Workload("noalloc-fp8", B=1, P=8, S_l=150, R=140, mode="suffix", Hq=40, Hkv=40, D=128, dtype="e4m3",
                   std_q=1.0, std_kv=1.0, seed=22, valid=((0, 1200 + 61),)),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_noalloc_matches_plan_call_twice(w):
    import torch
    import ulysses_sequence_attention_uly_gb300 as uly
    data = synth.generate(w)
    d = H.dev_inputs(w, data)
    plan = H.make_plan(w)
    tol = H.TOL[w.dtype]
    masks = [d["key_mask"], None]  # second call: every key admitted
    for call, km in enumerate(masks):
        ref = [torch.full((w.B, plan.shard_rows_q, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
               for _ in range(w.P)]
        plan.sp_attention(d["q"], d["k"], d["v"], ref, key_mask=km, head_groups=w.head_groups,
                          q_scale=d["q_scale"], k_scale=d["k_scale"], v_scale=d["v_scale"])
        got = [torch.full_like(x, float("nan")) for x in ref]
        uly.sp_attention_noalloc(w.B, w.P, w.S_l, w.R, w.mode, w.Hq, w.Hkv, w.D, d["q"], d["k"], d["v"], got,
                                 dtype=w.dtype, key_mask=km, head_groups=w.head_groups,
                                 q_scale=d["q_scale"], k_scale=d["k_scale"], v_scale=d["v_scale"])
        torch.cuda.synchronize()
        H.assert_written(ref)
        for a, b in zip(got, ref):
            ok, err, nbad = H.within(H.host_f64(a), H.host_f64(b), tol)
            assert ok, "call %d: max err %g, %d out of tolerance" % (call, err, nbad)


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
