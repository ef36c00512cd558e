"""Pins for the oracle's fp64 attention (CPU only).

Each check rests on something other than the oracle's own formula: a
hand-worked case (tests/golden/hand_2x2.txt), closed forms (uniform V,
one-hot scores), invariants (masked keys do not matter, key order does not
matter, which is what lets the replicated suffix be rotated to the front in
sglang layer.py USPAttention._forward_with_replicated_suffix), torch's fp64
scaled_dot_product_attention as an independent library routine, and torch's
own float8/bfloat16 decoders for the input formats.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_2x2.txt")


def _golden_cases():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            name, q0, q1, scale, m0, m1, o0, o1 = line.split()
            rows.append((name, [float(q0), float(q1)], float(scale), [int(m0), int(m1)], [float(o0), float(o1)]))
    return rows


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c[0])
def test_hand_worked(case):
    _, qv, scale, mask, want = case
    q = np.array(qv, dtype=np.float64).reshape(1, 1, 1, 2)
    k = np.array([[1.0, 0.0], [0.0, 1.0]]).reshape(1, 2, 1, 2)
    v = np.array([[1.0, 2.0], [3.0, 4.0]]).reshape(1, 2, 1, 2)
    km = np.array(mask, dtype=np.uint8).reshape(1, 2)
    o = oracle.attention(q, k, v, km, scale)
    np.testing.assert_allclose(o.reshape(2), want, rtol=0, atol=1e-15)


def _rand(shape, rng, std=1.0):
    return rng.standard_normal(shape) * std


def test_uniform_v_returns_that_row():
    rng = np.random.default_rng(0)
    B, Nq, Nk, H, D = 2, 7, 11, 3, 8
    row = rng.standard_normal(D)
    v = np.broadcast_to(row, (B, Nk, H, D)).copy()
    o = oracle.attention(_rand((B, Nq, H, D), rng), _rand((B, Nk, H, D), rng), v, None, 0.3)
    np.testing.assert_allclose(o, np.broadcast_to(row, o.shape), rtol=0, atol=1e-14)


def test_one_hot_scores_pick_that_value():
    # q orthogonal to every key but one; that key is c*q with large c, so
    # its weight is 1 - O(N e^{-c|q|^2 scale}).
    rng = np.random.default_rng(1)
    D, Nk = 8, 6
    q = np.zeros((1, 1, 1, D)); q[0, 0, 0, 0] = 1.0
    k = np.zeros((1, Nk, 1, D))
    for m in range(Nk):
        k[0, m, 0, 1 + (m % (D - 1))] = rng.standard_normal()
    hot = 4
    k[0, hot, 0, :] = 0.0
    k[0, hot, 0, 0] = 40.0
    v = _rand((1, Nk, 1, D), rng)
    o = oracle.attention(q, k, v, None, 1.0)
    bound = (Nk - 1) * np.exp(-40.0) * 2 * np.abs(v).max()
    np.testing.assert_allclose(o[0, 0, 0], v[0, hot, 0], rtol=0, atol=bound)


def test_masked_keys_do_not_matter():
    rng = np.random.default_rng(2)
    B, Nq, Nk, H, D = 2, 5, 13, 2, 4
    q, k, v = _rand((B, Nq, H, D), rng), _rand((B, Nk, H, D), rng), _rand((B, Nk, H, D), rng)
    km = (rng.random((B, Nk)) < 0.6).astype(np.uint8)
    km[:, 0] = 1
    o1 = oracle.attention(q, k, v, km, 0.5)
    k2, v2 = k.copy(), v.copy()
    dead = km == 0
    k2[dead] = 1e3 * rng.standard_normal((dead.sum(), H, D))
    v2[dead] = 1e3 * rng.standard_normal((dead.sum(), H, D))
    o2 = oracle.attention(q, k2, v2, km, 0.5)
    np.testing.assert_array_equal(o1, o2)


def test_key_order_does_not_matter():
    rng = np.random.default_rng(3)
    B, Nq, Nk, H, D = 1, 6, 17, 2, 8
    q, k, v = _rand((B, Nq, H, D), rng), _rand((B, Nk, H, D), rng), _rand((B, Nk, H, D), rng)
    km = (rng.random((B, Nk)) < 0.7).astype(np.uint8)
    perm = rng.permutation(Nk)
    o1 = oracle.attention(q, k, v, km, 0.4)
    o2 = oracle.attention(q, k[:, perm], v[:, perm], km[:, perm], 0.4)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-12)


def test_fully_masked_key_set_gives_zero():
    rng = np.random.default_rng(4)
    q, k, v = _rand((2, 3, 1, 4), rng), _rand((2, 5, 1, 4), rng), _rand((2, 5, 1, 4), rng)
    km = np.ones((2, 5), dtype=np.uint8)
    km[1] = 0
    o = oracle.attention(q, k, v, km, 1.0)
    assert np.all(o[1] == 0.0)
    assert np.all(np.abs(o[0]) > 0)


def _sdpa(q, k, v, km, scale):
    """torch fp64 SDPA with boolean key mask and GQA by repeat_interleave."""
    G = q.shape[2] // k.shape[2]
    qt = torch.from_numpy(q).transpose(1, 2)
    kt = torch.from_numpy(k).transpose(1, 2).repeat_interleave(G, dim=1)
    vt = torch.from_numpy(v).transpose(1, 2).repeat_interleave(G, dim=1)
    mask = None if km is None else torch.from_numpy(km.astype(bool))[:, None, None, :]
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    return o.transpose(1, 2).numpy()


@pytest.mark.parametrize("G", [1, 2, 4])
@pytest.mark.parametrize("masked", [False, True])
def test_matches_torch_sdpa_fp64(G, masked):
    rng = np.random.default_rng(10 + G)
    B, Nq, Nk, Hkv, D = 2, 9, 23, 2, 16
    Hq = Hkv * G
    q, k, v = _rand((B, Nq, Hq, D), rng), _rand((B, Nk, Hkv, D), rng), _rand((B, Nk, Hkv, D), rng)
    km = None
    if masked:
        km = (rng.random((B, Nk)) < 0.5).astype(np.uint8)
        km[:, 3] = 1
    scale = 1 / np.sqrt(D)
    np.testing.assert_allclose(oracle.attention(q, k, v, km, scale), _sdpa(q, k, v, km, scale),
                               rtol=1e-12, atol=1e-12)


def test_selected_rows_match_full():
    rng = np.random.default_rng(6)
    B, Nq, Nk, Hq, Hkv, D = 2, 8, 10, 4, 2, 8
    q, k, v = _rand((B, Nq, Hq, D), rng), _rand((B, Nk, Hkv, D), rng), _rand((B, Nk, Hkv, D), rng)
    full = oracle.attention(q, k, v, None, 0.3)
    sel = np.array([[1, 7, 3], [0, 0, 0], [1, 2, 1]], dtype=np.int32)
    part = oracle.attention(q, k, v, None, 0.3, sel=sel)
    for i, (b, n, h) in enumerate(sel):
        np.testing.assert_array_equal(part[i], full[b, n, h])


def test_zero_masked_rows():
    rng = np.random.default_rng(8)
    B, N, H, D = 1, 6, 2, 4
    q, k, v = _rand((B, N, H, D), rng), _rand((B, N + 2, H, D), rng), _rand((B, N + 2, H, D), rng)
    km = np.array([[1, 1, 0, 1, 1, 0, 1, 0]], dtype=np.uint8)
    a = oracle.attention(q, k, v, km, 0.5)
    z = oracle.attention(q, k, v, km, 0.5, zero_masked_rows=True, q_key_offset=2)
    for n in range(N):
        if km[0, n + 2]:
            np.testing.assert_array_equal(z[0, n], a[0, n])
        else:
            assert np.all(z[0, n] == 0)


def test_bf16_decode_matches_torch():
    bits = np.arange(0, 1 << 16, 37, dtype=np.uint16)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_f64(int(b)) for b in bits])
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(got[ok], want[ok])


def test_e4m3_decode_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_f64(int(c)) for c in codes])
    np.testing.assert_array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    np.testing.assert_array_equal(got[ok], want[ok])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


def test_storage_types_decode_with_scales():
    # bf16 / e4m3 attention equals fp64 attention on the decoded, scaled values
    rng = np.random.default_rng(9)
    B, Nq, Nk, Hq, Hkv, D = 1, 5, 9, 4, 2, 16
    qf, kf, vf = (rng.standard_normal(s).astype(np.float32) for s in
                  ((B, Nq, Hq, D), (B, Nk, Hkv, D), (B, Nk, Hkv, D)))
    to_bf = lambda x: torch.from_numpy(x).to(torch.bfloat16)
    qb, kb, vb = (to_bf(x) for x in (qf, kf, vf))
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    o_bits = oracle.attention(bits(qb), bits(kb), bits(vb), None, 0.25)
    o_f64 = oracle.attention(*(t.to(torch.float64).numpy() for t in (qb, kb, vb)), None, 0.25)
    np.testing.assert_array_equal(o_bits, o_f64)
    sq, sk, sv = (rng.uniform(0.01, 0.1, n).astype(np.float32) for n in (Hq, Hkv, Hkv))
    q8, k8, v8 = (torch.from_numpy(x / s[None, None, :, None]).to(torch.float8_e4m3fn)
                  for x, s in ((qf, sq), (kf, sk), (vf, sv)))
    o8 = oracle.attention(*(t.view(torch.uint8).numpy() for t in (q8, k8, v8)), None, 0.25,
                          q_scale=sq, k_scale=sk, v_scale=sv)
    deq = lambda t, s: t.to(torch.float64).numpy() * s.astype(np.float64)[None, None, :, None]
    o8_f64 = oracle.attention(deq(q8, sq), deq(k8, sk), deq(v8, sv), None, 0.25)
    np.testing.assert_allclose(o8, o8_f64, rtol=1e-13, atol=1e-13)


def test_within_rejects_nan():
    from tests import _helpers as H
    ok, _, nbad = H.within(np.array([1.0, np.nan]), np.array([1.0, 2.0]), 0.5)
    assert not ok and nbad == 1
    ok, _, _ = H.within(np.array([1.0, 2.2]), np.array([1.0, 2.0]), 0.1)
    assert ok


# ---- log-sum-exp output and the ring merge ---------------------------------

def test_lse_matches_logsumexp_definition():
    rng = np.random.default_rng(21)
    B, Nq, Nk, Hq, Hkv, D = 2, 5, 13, 4, 2, 8
    q, k, v = _rand((B, Nq, Hq, D), rng), _rand((B, Nk, Hkv, D), rng), _rand((B, Nk, Hkv, D), rng)
    km = (rng.random((B, Nk)) < 0.6).astype(np.uint8)
    km[0, :] = 0  # batch 0: no admitted key
    km[1, 2] = 1
    o, lse = oracle.attention_lse(q, k, v, km, 0.7)
    np.testing.assert_array_equal(o, oracle.attention(q, k, v, km, 0.7))
    assert np.all(np.isneginf(lse[0]))
    # torch's logsumexp of the admitted scores, GQA by repeat_interleave
    kt = torch.from_numpy(k).repeat_interleave(Hq // Hkv, dim=2)
    s = 0.7 * torch.einsum("bnhd,bmhd->bhnm", torch.from_numpy(q), kt)
    s = s.masked_fill(~torch.from_numpy(km.astype(bool))[:, None, None, :], float("-inf"))
    want = torch.logsumexp(s, dim=-1).permute(0, 2, 1).numpy()
    np.testing.assert_allclose(lse[1], want[1], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("split", [1, 6, 12])
def test_ring_merge_of_key_chunks_equals_whole(split):
    # attention over keys [0, split) and [split, Nk) merged by the page's
    # sigmoid / logsigmoid update equals attention over every key
    rng = np.random.default_rng(22)
    B, Nq, Nk, H, D = 1, 4, 13, 2, 8
    q, k, v = _rand((B, Nq, H, D), rng), _rand((B, Nk, H, D), rng), _rand((B, Nk, H, D), rng)
    whole, lse_w = oracle.attention_lse(q, k, v, None, 0.5)
    m1 = np.zeros((B, Nk), np.uint8); m1[:, :split] = 1
    m2 = 1 - m1
    o1, l1 = oracle.attention_lse(q, k, v, m1, 0.5)
    o2, l2 = oracle.attention_lse(q, k, v, m2, 0.5)
    om, lm = oracle.lse_merge(o1, l1, o2, l2)
    np.testing.assert_allclose(om, whole, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lm, lse_w, rtol=0, atol=1e-13)
    # merging in the other order gives the same result
    om2, lm2 = oracle.lse_merge(o2, l2, o1, l1)
    np.testing.assert_allclose(om2, whole, rtol=0, atol=1e-13)


def test_ring_merge_with_empty_part():
    rng = np.random.default_rng(23)
    o = rng.standard_normal((3, 4))
    lse = rng.standard_normal(3)
    ninf = np.full(3, -np.inf)
    zero = np.zeros((3, 4))
    a, la = oracle.lse_merge(o, lse, zero, ninf)
    np.testing.assert_array_equal(a, o); np.testing.assert_array_equal(la, lse)
    b, lb = oracle.lse_merge(zero, ninf, o, lse)
    np.testing.assert_array_equal(b, o); np.testing.assert_array_equal(lb, lse)


def test_masked_rows_as_own_segment_matches_sdpa():
    # convention "self": a query whose own token is masked attends to the
    # masked keys only, an admitted one to the admitted keys only; checked
    # against torch fp64 SDPA with the equivalent per-row boolean mask
    rng = np.random.default_rng(24)
    B, N, Hq, Hkv, D = 2, 11, 4, 2, 8
    q, k, v = _rand((B, N, Hq, D), rng), _rand((B, N + 3, Hkv, D), rng), _rand((B, N + 3, Hkv, D), rng)
    km = (rng.random((B, N + 3)) < 0.6).astype(np.uint8)
    km[:, 4] = 0
    km[:, 5] = 1
    off = 3
    got = oracle.attention(q, k, v, km, 0.4, zero_masked_rows=2, q_key_offset=off)
    rowv = km[:, off:off + N].astype(bool)                       # [B, N]
    allowed = (km.astype(bool)[:, None, :] == rowv[:, :, None])   # [B, N, Nk]
    G = Hq // Hkv
    o = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q).transpose(1, 2), torch.from_numpy(k).transpose(1, 2).repeat_interleave(G, 1),
        torch.from_numpy(v).transpose(1, 2).repeat_interleave(G, 1),
        attn_mask=torch.from_numpy(allowed)[:, None], scale=0.4).transpose(1, 2).numpy()
    np.testing.assert_allclose(got, o, rtol=1e-12, atol=1e-12)
    # admitted rows are the same under every convention
    sdpa = oracle.attention(q, k, v, km, 0.4)
    np.testing.assert_array_equal(got[rowv], sdpa[rowv])
