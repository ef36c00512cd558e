"""GPU attention through the C ABI against the oracle (small and ragged
shapes spanning several tiles), plus the bit-identity properties:
fused == staged, every head-group split == whole call, key_mask == ranges."""
import zlib

import numpy as np
import pytest

import synth
from tests import _helpers as H

pytestmark = pytest.mark.gpu


def _w(name, mode, P, S_l, R, Hq, Hkv, D, dtype="bf16", B=1, valid=None, std_kv=1.0, seed=None):
    return synth.Workload(name, B=B, P=P, S_l=S_l, R=R if mode != "none" else 0, mode=mode, Hq=Hq, Hkv=Hkv, D=D,
                          dtype=dtype, std_q=1.0, std_kv=std_kv, seed=seed if seed is not None else zlib.crc32(name.encode()) % 1000,
                          valid=valid)


SMALL = [
    synth.WORKLOADS["tiny"],
    # Wan-14B-like: prefix, masked text keys, tiles straddle every run end
    _w("wan14b-s", "prefix", 4, 300, 200, 8, 8, 128, valid=((0, 77), (200, 1400))),
    # Wan-1.3B-like: dense, unmasked, several tiles per run, 0.5 std
    _w("wan13b-s", "none", 4, 520, 0, 12, 12, 128),
    # GQA with a K/V-only prefix, batch 2
    _w("gqa-s", "kv_prefix", 4, 260, 256, 16, 4, 128, B=2, std_kv=0.7),
    # fp8 with a replicated suffix and masked suffix keys
    _w("fp8-s", "suffix", 8, 150, 140, 40, 40, 128, dtype="e4m3", valid=((0, 1200 + 61),)),
    # head dim 64
    _w("d64", "suffix", 2, 333, 45, 4, 2, 64, valid=((0, 300), (400, 700))),
    # ragged runs around the 128/256-row tile and unit boundaries
    _w("ragged-1", "prefix", 3, 1, 1, 6, 6, 128),
    _w("ragged-127", "prefix", 2, 127, 129, 4, 4, 128),
    _w("ragged-257", "suffix", 2, 257, 128, 4, 2, 128, B=2),
    _w("ragged-kv", "kv_prefix", 2, 255, 1, 2, 2, 64),
]


def _id(w):
    return w.name


@pytest.mark.parametrize("w", SMALL, ids=_id)
def test_staged_and_fused_match_oracle(w):
    import torch
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    oh, o = H.run_staged(plan, w, d, head_groups=1)
    of = H.run_fused(plan, w, d, head_groups=1)
    torch.cuda.synchronize()
    assert plan.sync_status() == 0
    want_oh, want_o = H.oracle_path(w, data)
    tol = H.TOL[w.dtype]
    for r in range(w.P):
        ok, err, nbad = H.within(H.host_f64(oh[r]), want_oh[r], tol)
        assert ok, "rank %d: max err %g, %d elements out of tolerance" % (r, err, nbad)
    for p in range(w.P):
        ok, err, nbad = H.within(H.host_f64(o[p]), want_o[p], tol)
        assert ok, "shard %d: max err %g, %d out of tolerance" % (p, err, nbad)
        # the fused path is the staged path, bit for bit
        assert torch.equal(o[p].view(torch.int16), of[p].view(torch.int16)), "fused != staged on shard %d" % p


@pytest.mark.parametrize("w", [x for x in SMALL if x.Hq // x.P > 1], ids=_id)
def test_head_group_splits_are_bit_identical(w):
    import torch
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    ref_f = H.run_fused(plan, w, d, head_groups=1)
    ref_oh, _ = H.run_staged(plan, w, d, head_groups=1)
    torch.cuda.synchronize()
    H.assert_written(ref_f)
    H.assert_written(ref_oh)
    hq_l, hkv_l = w.Hq // w.P, w.Hkv // w.P
    for g in range(2, hq_l + 1):
        if hq_l % g or hkv_l % g:
            continue
        f = H.run_fused(plan, w, d, head_groups=g)
        s_oh, _ = H.run_staged(plan, w, d, head_groups=g)
        torch.cuda.synchronize()
        for a, b in zip(ref_f, f):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), "fused g=%d" % g
        for a, b in zip(ref_oh, s_oh):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), "staged g=%d" % g


@pytest.mark.parametrize("w", [x for x in SMALL if x.valid is not None], ids=_id)
def test_key_mask_and_ranges_agree(w):
    import torch
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    a = H.run_fused(plan, w, d, mask="mask")
    b = H.run_fused(plan, w, d, mask="ranges")
    torch.cuda.synchronize()
    H.assert_written(a)
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_masked_keys_do_not_matter_on_gpu():
    import torch
    w = SMALL[1]
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    a = H.run_fused(plan, w, d)
    # overwrite masked text keys/values (rows 77..199 of the prefix) on every shard
    for t in d["k"] + d["v"]:
        t[:, 77:200] = 50.0
    b = H.run_fused(plan, w, d)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_fully_masked_gives_zero():
    import torch
    w = _w("allmasked", "prefix", 2, 100, 30, 4, 4, 128, B=2)
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    km = torch.ones((w.B, plan.heads_rows_kv), dtype=torch.uint8, device="cuda")
    km[1] = 0
    o = [torch.full((w.B, plan.shard_rows_q, w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
         for _ in range(w.P)]
    plan.sp_attention(d["q"], d["k"], d["v"], o, key_mask=km)
    torch.cuda.synchronize()
    data["key_mask"] = km.cpu().numpy()
    _, want = H.oracle_path(w, data)
    for p in range(w.P):
        assert torch.all(o[p][1] == 0)
        ok, err, _ = H.within(H.host_f64(o[p]), want[p], H.TOL["bf16"])
        assert ok, err


@pytest.mark.parametrize("w", [SMALL[0], SMALL[1], SMALL[3]], ids=_id)
def test_zero_masked_rows(w):
    import torch
    data = synth.generate(w)
    if data["key_mask"] is None:
        m = np.ones((w.B, w.rows_global(True)), dtype=np.uint8)
        m[:, 3:40] = 0
        data["key_mask"] = m
    plan = H.make_plan(w, masked_rows="zero")
    d = H.dev_inputs(w, data)
    oh, o = H.run_staged(plan, w, d)
    of = H.run_fused(plan, w, d)
    torch.cuda.synchronize()
    want_oh, want_o = H.oracle_path(w, data, zero_rows=True)
    for p in range(w.P):
        ok, err, _ = H.within(H.host_f64(o[p]), want_o[p], H.TOL["bf16"])
        assert ok, err
        assert np.array_equal(H.host_f64(o[p]) == 0, want_o[p] == 0)
        assert torch.equal(o[p].view(torch.int16), of[p].view(torch.int16))


def test_explicit_scale():
    import torch
    w = SMALL[2]
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    o = [torch.empty((w.B, plan.shard_rows_q, w.Hq, w.D), dtype=torch.bfloat16, device="cuda") for _ in range(w.P)]
    plan.sp_attention(d["q"], d["k"], d["v"], o, scale=0.3)
    torch.cuda.synchronize()
    data["scale"] = 0.3
    _, want = H.oracle_path(w, data)
    for p in range(w.P):
        ok, err, _ = H.within(H.host_f64(o[p]), want[p], H.TOL["bf16"])
        assert ok, err


def test_call_errors():
    import torch
    from ulysses_sequence_attention_uly_gb300 import UlyError, ULY_ERR_INVALID
    w = SMALL[0]
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    o = [torch.empty((w.B, plan.shard_rows_q, w.Hq, w.D), dtype=torch.bfloat16, device="cuda") for _ in range(w.P)]
    with pytest.raises(UlyError) as e:  # both a mask and ranges
        plan.sp_attention(d["q"], d["k"], d["v"], o, key_mask=d["key_mask"], key_ranges=d["key_ranges"])
    assert e.value.status == ULY_ERR_INVALID
    with pytest.raises(UlyError):  # 3 does not divide the 2 heads per rank
        plan.sp_attention(d["q"], d["k"], d["v"], o, head_groups=3)
    with pytest.raises(UlyError):  # bf16 with fp8 scales
        plan.sp_attention(d["q"], d["k"], d["v"], o, q_scale=torch.ones(4, device="cuda"),
                          k_scale=torch.ones(4, device="cuda"), v_scale=torch.ones(4, device="cuda"))
    with pytest.raises(UlyError):  # misaligned pointer
        raw = torch.empty(d["q"][0].numel() + 8, dtype=torch.bfloat16, device="cuda")
        bad = raw[1:1 + d["q"][0].numel()].view_as(d["q"][0])
        plan.sp_attention([bad] + d["q"][1:], d["k"], d["v"], o)
    with pytest.raises(UlyError):  # non-positive scale
        plan.sp_attention(d["q"], d["k"], d["v"], o, scale=0.0)
    assert plan.sync_status() == 0


@pytest.mark.parametrize("w", [SMALL[0], SMALL[1], SMALL[3], SMALL[4], SMALL[5]], ids=_id)
def test_masked_rows_own_segment(w):
    """ULY_ROWS_SELF: masked query rows attend only to the masked keys."""
    import torch
    data = synth.generate(w)
    if data["key_mask"] is None:
        m = np.ones((w.B, w.rows_global(True)), dtype=np.uint8)
        m[:, 3:200] = 0
        data["key_mask"] = m
    plan = H.make_plan(w, masked_rows="self")
    d = H.dev_inputs(w, data)
    oh, o = H.run_staged(plan, w, d)
    of = H.run_fused(plan, w, d)
    torch.cuda.synchronize()
    want_oh, want_o = H.oracle_path(w, data, zero_rows=2)
    for p in range(w.P):
        ok, err, nbad = H.within(H.host_f64(o[p]), want_o[p], H.TOL[w.dtype])
        assert ok, "shard %d: max err %g (%d)" % (p, err, nbad)
        assert torch.equal(o[p].view(torch.int16), of[p].view(torch.int16))


@pytest.mark.parametrize("mode", ["prefix", "suffix", "kv_prefix"])
def test_per_batch_masks_and_ranges(mode):
    """Each batch has its own valid key ranges (batch > 1 with replicated
    text rows): key_ranges and the equivalent key_mask give the same bits,
    and both match the oracle."""
    import torch
    w = _w("perbatch-" + mode, mode, 4, 150, 96, 8, 8, 128, B=3)
    data = synth.generate(w)
    nk = w.rows_global(True)
    ranges = np.array([[[0, 17], [96, 96 + 300]],
                       [[5, 90], [200, nk]],
                       [[0, nk], [nk, nk]]], dtype=np.int32)  # batch 2: all keys (and an empty range)
    if mode == "suffix":  # text rows are the last R keys
        ranges = np.array([[[0, 300], [600, 600 + 17]],
                           [[100, 650], [650, 650]],
                           [[0, nk], [nk, nk]]], dtype=np.int32)
    m = np.zeros((w.B, nk), dtype=np.uint8)
    for b in range(w.B):
        for a0, a1 in ranges[b]:
            m[b, a0:a1] = 1
    data["key_mask"], data["key_ranges"] = m, ranges
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    o_mask = H.run_fused(plan, w, d, mask="mask")
    o_rng = H.run_fused(plan, w, d, mask="ranges")
    _, o_staged = H.run_staged(plan, w, d, mask="ranges")
    torch.cuda.synchronize()
    _, want = H.oracle_path(w, data)
    for p in range(w.P):
        ok, err, nbad = H.within(H.host_f64(o_mask[p]), want[p], H.TOL["bf16"])
        assert ok, "shard %d: max err %g (%d)" % (p, err, nbad)
        assert torch.equal(o_mask[p].view(torch.int16), o_rng[p].view(torch.int16))
        assert torch.equal(o_mask[p].view(torch.int16), o_staged[p].view(torch.int16))


def test_binding_rejects_bad_tensors():
    """The binding checks shapes, element types, devices, contiguity and list
    lengths against the plan before any call reaches the C ABI."""
    import torch
    w = SMALL[1]
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    o = [torch.empty((w.B, plan.shard_rows(p), w.Hq, w.D), dtype=torch.bfloat16, device="cuda") for p in range(w.P)]
    bad_cases = [
        dict(q=d["q"][:-1]),                                                  # one shard short
        dict(q=[x[:, :-1] for x in d["q"]]),                                  # a row short
        dict(q=[x.float() for x in d["q"]]),                                  # wrong element type
        dict(q=[x.cpu() for x in d["q"]]),                                    # host memory
        dict(q=[x.transpose(2, 1).contiguous().transpose(2, 1) for x in d["q"]]),  # not contiguous
        dict(o=[x.float() for x in o]),                                       # f32 output
        dict(key_mask=d["key_mask"][:, :-1]),                                 # mask a key short
        dict(key_ranges=torch.zeros((w.B, 2, 3), dtype=torch.int32, device="cuda")),
        dict(lse=[torch.empty((w.B, plan.shard_rows(p), w.Hq - 1), device="cuda") for p in range(w.P)]),
    ]
    for case in bad_cases:
        args = dict(q=d["q"], k=d["k"], v=d["v"], o=o, key_mask=d["key_mask"])
        args.update(case)
        with pytest.raises(ValueError):
            plan.sp_attention(args["q"], args["k"], args["v"], args["o"], key_mask=args["key_mask"],
                              key_ranges=args.get("key_ranges"), lse=args.get("lse"))
    qh, kh, vh = H.empty_heads(plan, w, H.in_dtype(w))
    with pytest.raises(ValueError):
        plan.to_heads(d["q"], d["k"], d["v"], qh[:-1], kh, vh)
    with pytest.raises(ValueError):
        plan.to_seq([x[:, :-1] for x in qh], o)
    # nothing reached the GPU: the good call still works
    plan.sp_attention(d["q"], d["k"], d["v"], o, key_mask=d["key_mask"])
    torch.cuda.synchronize()
    assert plan.sync_status() == 0
