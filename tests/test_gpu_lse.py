"""Log-sum-exp output and the ring-attention merge on the GPU, against the
oracle: LSE of the staged and fused paths, the merge kernel itself, and ring
attention over virtual ring ranks (one key chunk each, merged in ring order)
equal to attention over every key."""
import numpy as np
import pytest

import oracle
import synth
from tests import _helpers as H

pytestmark = pytest.mark.gpu

LSE_TOL = 1e-3

W_MASKED = synth.Workload("lse-prefix", B=2, P=4, S_l=300, R=200, mode="prefix", Hq=8, Hkv=4, D=128, dtype="bf16",
                          std_q=1.0, std_kv=1.0, seed=31, valid=((0, 77), (200, 1400)))
W_FP8 = synth.Workload("lse-fp8", B=1, P=2, S_l=260, R=64, mode="suffix", Hq=4, Hkv=4, D=128, dtype="e4m3",
                       std_q=1.0, std_kv=1.0, seed=32, valid=((0, 520 + 30),))
W_D64 = synth.Workload("lse-d64", B=1, P=2, S_l=333, R=0, mode="none", Hq=4, Hkv=2, D=64, dtype="bf16",
                       std_q=1.0, std_kv=1.0, seed=33)


def _oracle_rank_lse(w, data, heads, r, key_mask):
    qh, kh, vh = heads
    Hl, Hkl = w.Hq // w.P, w.Hkv // w.P
    sl = lambda a, n: None if a is None else np.ascontiguousarray(a[r * n:(r + 1) * n])
    koff = w.R if w.mode == "kv_prefix" else 0
    return oracle.attention_lse(qh[r], kh[r], vh[r], key_mask, data["scale"], sl(data["q_scale"], Hl),
                                sl(data["k_scale"], Hkl), sl(data["v_scale"], Hkl), q_key_offset=koff)


def _lse_within(got, ref, tol=LSE_TOL):
    both_inf = np.isneginf(got) & np.isneginf(ref)
    fin = ~both_inf
    assert np.array_equal(np.isneginf(got), np.isneginf(ref))
    err = np.abs(got[fin].astype(np.float64) - ref[fin])
    ok = err <= tol * (1 + np.abs(ref[fin]))
    assert ok.all(), "max lse err %g" % err.max()


@pytest.mark.parametrize("w", [W_MASKED, W_FP8, W_D64], ids=lambda w: w.name)
def test_lse_staged_and_fused(w):
    import torch
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    qh, kh, vh = H.empty_heads(plan, w, H.in_dtype(w))
    plan.to_heads(d["q"], d["k"], d["v"], qh, kh, vh)
    oh = [torch.empty((w.B, plan.heads_rows_q, w.Hq // w.P, w.D), dtype=torch.bfloat16, device="cuda") for _ in range(w.P)]
    lh = [torch.full((w.B, plan.heads_rows_q, w.Hq // w.P), float("nan"), device="cuda") for _ in range(w.P)]
    plan.attention(qh, kh, vh, oh, key_mask=d["key_mask"], q_scale=d["q_scale"], k_scale=d["k_scale"],
                   v_scale=d["v_scale"], lse=lh)
    o = [torch.empty((w.B, plan.shard_rows_q, w.Hq, w.D), dtype=torch.bfloat16, device="cuda") for _ in range(w.P)]
    ls = [torch.full((w.B, plan.shard_rows_q, w.Hq), float("nan"), device="cuda") for _ in range(w.P)]
    plan.sp_attention(d["q"], d["k"], d["v"], o, key_mask=d["key_mask"], q_scale=d["q_scale"], k_scale=d["k_scale"],
                      v_scale=d["v_scale"], lse=ls)
    torch.cuda.synchronize()
    heads = H.oracle_heads(w, data)
    for r in range(w.P):
        _, want = _oracle_rank_lse(w, data, heads, r, data["key_mask"])
        _lse_within(lh[r].cpu().numpy(), want)
    # the fused LSE is the staged LSE moved back to the shards, bit for bit
    s1 = oracle.Shape(w.B, w.P, w.S_l, w.R, w.rep_mode, w.Hq, w.Hkv, 1)
    back = oracle.to_seq(s1, [x.cpu().numpy()[..., None] for x in lh])
    for p in range(w.P):
        np.testing.assert_array_equal(ls[p].cpu().numpy(), back[p][..., 0])


def test_merge_kernel_matches_oracle():
    import torch
    import ulysses_sequence_attention_uly_gb300 as uly
    rng = np.random.default_rng(40)
    rows, D = 777, 128
    oa = torch.from_numpy(rng.standard_normal((rows, D)).astype(np.float32)).to(torch.bfloat16).cuda()
    ob = torch.from_numpy(rng.standard_normal((rows, D)).astype(np.float32)).to(torch.bfloat16).cuda()
    la = rng.standard_normal(rows).astype(np.float32) * 5
    lb = rng.standard_normal(rows).astype(np.float32) * 5
    la[::17] = -np.inf
    lb[::13] = -np.inf
    la_t, lb_t = torch.from_numpy(la).cuda(), torch.from_numpy(lb).cuda()
    out = torch.empty_like(oa)
    lout = torch.empty_like(la_t)
    uly.lse_merge(oa, la_t, ob, lb_t, out, lout)
    torch.cuda.synchronize()
    want_o, want_l = oracle.lse_merge(oa.double().cpu().numpy(), la.astype(np.float64), ob.double().cpu().numpy(),
                                      lb.astype(np.float64))
    ok, err, _ = H.within(H.host_f64(out), want_o, 1e-2)
    assert ok, err
    _lse_within(lout.cpu().numpy(), want_l, 1e-5)
    # in place gives the same bytes
    uly.lse_merge(oa, la_t, ob, lb_t)
    torch.cuda.synchronize()
    assert torch.equal(oa.view(torch.int16), out.view(torch.int16))
    assert torch.equal(la_t, lout)


@pytest.mark.parametrize("w,chunks", [(W_MASKED, 3), (W_D64, 4), (W_FP8, 2)], ids=lambda x: getattr(x, "name", str(x)))
def test_ring_over_key_chunks_equals_whole(w, chunks):
    """Ring attention over virtual ring ranks: rank c attends to key chunk c
    (key mask restricted to the chunk); merging the partial (O, LSE) in ring
    order gives attention over every key."""
    import torch
    import ulysses_sequence_attention_uly_gb300 as uly
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    qh, kh, vh = H.empty_heads(plan, w, H.in_dtype(w))
    plan.to_heads(d["q"], d["k"], d["v"], qh, kh, vh)
    nk = plan.heads_rows_kv
    base = data["key_mask"] if data["key_mask"] is not None else np.ones((w.B, nk), np.uint8)
    bounds = np.linspace(0, nk, chunks + 1).astype(int)
    acc_o = acc_l = None
    for c in range(chunks):
        m = np.zeros_like(base)
        m[:, bounds[c]:bounds[c + 1]] = base[:, bounds[c]:bounds[c + 1]]
        oh = [torch.empty((w.B, plan.heads_rows_q, w.Hq // w.P, w.D), dtype=torch.bfloat16, device="cuda")
              for _ in range(w.P)]
        lh = [torch.empty((w.B, plan.heads_rows_q, w.Hq // w.P), device="cuda") for _ in range(w.P)]
        plan.attention(qh, kh, vh, oh, key_mask=torch.from_numpy(m).cuda(), q_scale=d["q_scale"],
                       k_scale=d["k_scale"], v_scale=d["v_scale"], lse=lh)
        if acc_o is None:
            acc_o, acc_l = oh, lh
        else:
            for r in range(w.P):
                uly.lse_merge(acc_o[r], acc_l[r], oh[r], lh[r])
    torch.cuda.synchronize()
    heads = H.oracle_heads(w, data)
    for r in range(w.P):
        want_o, want_l = _oracle_rank_lse(w, data, heads, r, data["key_mask"])
        ok, err, nbad = H.within(H.host_f64(acc_o[r]), want_o, H.TOL[w.dtype])
        assert ok, "rank %d: max err %g (%d)" % (r, err, nbad)
        _lse_within(acc_l[r].cpu().numpy(), want_l)


def _chunk_mask(base, lo, hi):
    m = np.zeros_like(base)
    m[:, lo:hi] = base[:, lo:hi]
    return m


# key chunks in ring order: W_MASKED admits keys [0, 77) and [200, 1400), so
# its chunk [77, 200) admits none -- first (both parts empty), then a chunk
# that fills the empty rows, a regular merge, and the empty chunk again
# (every row keeps its running values)
RING_CHUNKS = {
    "lse-prefix": [(77, 200), (0, 77), (200, 700), (700, 1400), (77, 200)],
    "lse-fp8": [(0, 300), (300, 520 + 30)],
    "lse-d64": [(0, 222), (222, 500), (500, 666)],
}


@pytest.mark.parametrize("w", [W_MASKED, W_FP8, W_D64], ids=lambda w: w.name)
def test_ring_with_fused_merge_equals_whole(w):
    """uly_attention_merge step by step over key chunks (the merge in the
    attention's epilogue) gives attention over every key, and matches the
    ring built from separate uly_lse_merge passes."""
    import torch
    import ulysses_sequence_attention_uly_gb300 as uly
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    qh, kh, vh = H.empty_heads(plan, w, H.in_dtype(w))
    plan.to_heads(d["q"], d["k"], d["v"], qh, kh, vh)
    nk = plan.heads_rows_kv
    base = data["key_mask"] if data["key_mask"] is not None else np.ones((w.B, nk), np.uint8)
    sc = dict(q_scale=d["q_scale"], k_scale=d["k_scale"], v_scale=d["v_scale"])
    shape_o = (w.B, plan.heads_rows_q, w.Hq // w.P, w.D)
    shape_l = (w.B, plan.heads_rows_q, w.Hq // w.P)
    # running result starts empty: lse -inf, O never read (NaN would show)
    oh = [torch.full(shape_o, float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(w.P)]
    lh = [torch.full(shape_l, float("-inf"), device="cuda") for _ in range(w.P)]
    # the same ring through separate merges
    acc_o = acc_l = None
    for lo, hi in RING_CHUNKS[w.name]:
        m = torch.from_numpy(_chunk_mask(base, lo, hi)).cuda()
        plan.attention_merge(qh, kh, vh, oh, lh, key_mask=m, **sc)
        o_c = [torch.empty(shape_o, dtype=torch.bfloat16, device="cuda") for _ in range(w.P)]
        l_c = [torch.empty(shape_l, device="cuda") for _ in range(w.P)]
        plan.attention(qh, kh, vh, o_c, key_mask=m, lse=l_c, **sc)
        if acc_o is None:
            acc_o, acc_l = o_c, l_c
        else:
            for r in range(w.P):
                uly.lse_merge(acc_o[r], acc_l[r], o_c[r], l_c[r])
    torch.cuda.synchronize()
    assert plan.sync_status() == 0
    heads = H.oracle_heads(w, data)
    for r in range(w.P):
        want_o, want_l = _oracle_rank_lse(w, data, heads, r, data["key_mask"])
        got = H.host_f64(oh[r])
        ok, err, nbad = H.within(got, want_o, H.TOL[w.dtype])
        assert ok, "rank %d: max err %g (%d)" % (r, err, nbad)
        _lse_within(lh[r].cpu().numpy(), want_l)
        # fused and separate merges agree to within the bf16 rounding of the steps
        ok, err, nbad = H.within(got, H.host_f64(acc_o[r]), H.TOL[w.dtype])
        assert ok, "rank %d vs separate merges: max err %g (%d)" % (r, err, nbad)
        _lse_within(lh[r].cpu().numpy(), acc_l[r].cpu().numpy().astype(np.float64))


def test_attention_merge_needs_lse_and_staged_layout():
    import torch
    import ulysses_sequence_attention_uly_gb300 as uly
    w = W_D64
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    qh, kh, vh = H.empty_heads(plan, w, H.in_dtype(w))
    oh = [torch.empty((w.B, plan.heads_rows_q, w.Hq // w.P, w.D), dtype=torch.bfloat16, device="cuda")
          for _ in range(w.P)]
    with pytest.raises(ValueError):
        plan.attention_merge(qh, kh, vh, oh, None)
    import ctypes
    from ulysses_sequence_attention_uly_gb300 import _ptr_array
    rc = uly.lib().uly_attention_merge(plan._h, _ptr_array(qh), _ptr_array(kh), _ptr_array(vh), None, None, 0,
                                       ctypes.c_float(0.125), 0, None, None, None, _ptr_array(oh), None, None)
    assert rc == uly.ULY_ERR_INVALID


# one-launch ring: chunk bounds per workload (P + 1 entries), including empty
# chunks and a bound inside a 128-key tile
RING_BOUNDS = {
    "lse-prefix": lambda nk: [0, 77, 200, 700, nk],       # P = 4; rank 1's chunk admits no key
    "lse-fp8": lambda nk: [0, 300, nk],                   # P = 2
    "lse-d64": lambda nk: [0, 0, nk],                     # P = 2; rank 0's chunk empty
}


@pytest.mark.parametrize("w", [W_MASKED, W_FP8, W_D64], ids=lambda w: w.name)
def test_ring_one_launch_equals_whole(w):
    """uly_ring_attention (every rank's queries walk the key chunks from
    their own rank's on, in one launch) gives attention over every key, O and
    LSE, and agrees with the chunk-by-chunk ring of uly_attention_merge to
    within rounding.  A rank whose walk starts at key 0 takes the keys in
    the order uly_attention does and is bit-identical to it."""
    import torch
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    qh, kh, vh = H.empty_heads(plan, w, H.in_dtype(w))
    plan.to_heads(d["q"], d["k"], d["v"], qh, kh, vh)
    nk = plan.heads_rows_kv
    bounds = RING_BOUNDS[w.name](nk)
    sc = dict(q_scale=d["q_scale"], k_scale=d["k_scale"], v_scale=d["v_scale"])
    km = None if data["key_mask"] is None else torch.from_numpy(data["key_mask"]).cuda()
    shape_o = (w.B, plan.heads_rows_q, w.Hq // w.P, w.D)
    shape_l = (w.B, plan.heads_rows_q, w.Hq // w.P)
    oh = [torch.full(shape_o, float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(w.P)]
    lh = [torch.full(shape_l, float("nan"), device="cuda") for _ in range(w.P)]
    plan.ring_attention(qh, kh, vh, oh, bounds, key_mask=km, lse=lh, **sc)
    # the plain call (ascending key order) and the chunk-by-chunk ring
    op = [torch.empty(shape_o, dtype=torch.bfloat16, device="cuda") for _ in range(w.P)]
    lp = [torch.empty(shape_l, device="cuda") for _ in range(w.P)]
    plan.attention(qh, kh, vh, op, key_mask=km, lse=lp, **sc)
    base = data["key_mask"] if data["key_mask"] is not None else np.ones((w.B, nk), np.uint8)
    oc = [torch.full(shape_o, float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(w.P)]
    lc = [torch.full(shape_l, float("-inf"), device="cuda") for _ in range(w.P)]
    for c in range(w.P):
        m = torch.from_numpy(_chunk_mask(base, bounds[c], bounds[c + 1])).cuda()
        plan.attention_merge(qh, kh, vh, oc, lc, key_mask=m, **sc)
    torch.cuda.synchronize()
    assert plan.sync_status() == 0
    heads = H.oracle_heads(w, data)
    for r in range(w.P):
        want_o, want_l = _oracle_rank_lse(w, data, heads, r, data["key_mask"])
        got = H.host_f64(oh[r])
        ok, err, nbad = H.within(got, want_o, H.TOL[w.dtype])
        assert ok, "rank %d: max err %g (%d)" % (r, err, nbad)
        _lse_within(lh[r].cpu().numpy(), want_l)
        ok, err, nbad = H.within(got, H.host_f64(oc[r]), H.TOL[w.dtype])
        assert ok, "rank %d vs chunk-by-chunk ring: max err %g (%d)" % (r, err, nbad)
        if bounds[r] == 0:
            # the walk starts at the first admitted tile: the plain order
            assert torch.equal(oh[r].view(torch.int16), op[r].view(torch.int16)), "rank %d" % r
            assert torch.equal(lh[r], lp[r]), "rank %d" % r


def test_ring_attention_rejects_bad_bounds():
    import ctypes
    import torch
    import ulysses_sequence_attention_uly_gb300 as uly
    from ulysses_sequence_attention_uly_gb300 import _ptr_array
    w = W_D64
    data = synth.generate(w)
    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    qh, kh, vh = H.empty_heads(plan, w, H.in_dtype(w))
    oh = [torch.empty((w.B, plan.heads_rows_q, w.Hq // w.P, w.D), dtype=torch.bfloat16, device="cuda")
          for _ in range(w.P)]
    nk = plan.heads_rows_kv
    with pytest.raises(ValueError):
        plan.ring_attention(qh, kh, vh, oh, [0, nk])
    for bad in ([1, 100, nk], [0, 100, nk - 1], [0, 300, 200], [0, 100, nk + 1]):
        cb = (ctypes.c_int32 * 3)(*bad)
        rc = uly.lib().uly_ring_attention(plan._h, _ptr_array(qh), _ptr_array(kh), _ptr_array(vh), None, None, 0,
                                          cb, ctypes.c_float(0.125), 0, None, None, None, _ptr_array(oh), None, None)
        assert rc == uly.ULY_ERR_INVALID, bad
    rc = uly.lib().uly_ring_attention(plan._h, _ptr_array(qh), _ptr_array(kh), _ptr_array(vh), None, None, 0,
                                      None, ctypes.c_float(0.125), 0, None, None, None, _ptr_array(oh), None, None)
    assert rc == uly.ULY_ERR_INVALID


W_UNEVEN = synth.Workload("ring-uneven", B=2, P=4, S_l=0, R=96, mode="prefix", Hq=8, Hkv=4, D=128, dtype="bf16",
                          std_q=1.0, std_kv=1.0, seed=35, valid=((0, 40), (96, 96 + 700)), lens=(300, 45, 257, 129))


@pytest.mark.parametrize("w,masked_rows", [(W_MASKED, "self"), (W_UNEVEN, "sdpa"), (W_UNEVEN, "zero")],
                         ids=["self-rows", "uneven", "uneven-zero-rows"])
def test_ring_one_launch_other_plans(w, masked_rows):
    """The one-launch ring under the other masked-row conventions (the
    'self' rows walk the complement key sets, rotated alike) and on uneven
    shards: every rank within tolerance of the plain call, rank 0 (whose walk
    starts at key 0) equal to it bit for bit."""
    import torch
    data = synth.generate(w)
    plan = H.make_plan(w, masked_rows=masked_rows)
    d = H.dev_inputs(w, data)
    qh, kh, vh = H.empty_heads(plan, w, H.in_dtype(w))
    plan.to_heads(d["q"], d["k"], d["v"], qh, kh, vh)
    nk = plan.heads_rows_kv
    bounds = [int(x) for x in np.linspace(0, nk, w.P + 1)]
    sc = dict(q_scale=d["q_scale"], k_scale=d["k_scale"], v_scale=d["v_scale"])
    km = torch.from_numpy(data["key_mask"]).cuda()
    shape_o = (w.B, plan.heads_rows_q, w.Hq // w.P, w.D)
    shape_l = (w.B, plan.heads_rows_q, w.Hq // w.P)
    op = [torch.full(shape_o, float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(w.P)]
    lp = [torch.full(shape_l, float("nan"), device="cuda") for _ in range(w.P)]
    plan.attention(qh, kh, vh, op, key_mask=km, lse=lp, **sc)
    orng = [torch.full(shape_o, float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(w.P)]
    lrng = [torch.full(shape_l, float("nan"), device="cuda") for _ in range(w.P)]
    plan.ring_attention(qh, kh, vh, orng, bounds, key_mask=km, lse=lrng, **sc)
    torch.cuda.synchronize()
    assert plan.sync_status() == 0
    H.assert_written(orng)
    assert torch.equal(orng[0].view(torch.int16), op[0].view(torch.int16))
    assert torch.equal(lrng[0], lp[0])
    for r in range(w.P):
        ok, err, nbad = H.within(H.host_f64(orng[r]), H.host_f64(op[r]), H.TOL[w.dtype])
        assert ok, "rank %d: max err %g (%d)" % (r, err, nbad)
        _lse_within(lrng[r].cpu().numpy(), lp[r].cpu().numpy().astype(np.float64))
