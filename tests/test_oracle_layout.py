"""Pins for the oracle's sequence<->head exchange (CPU only).

The oracle writes the exchange as an explicit per-element index map.  These
tests check it against facts that do not come from that map:

* the round trip to_seq(to_heads(x)) is the identity and P=1 is the identity;
* an "iota" fill (every element carries its own coordinates) shows every
  element lands exactly once, in sender-rank-major order, with rank r holding
  heads [r*H/P, (r+1)*H/P) and taking replicated rows from its own shard;
* an independent formulation with torch chunk/cat and with the
  reshape/permute chain of flashdreams cp.py ContextParallelAttention.
  _impl_ulysses, over P virtual ranks, and of the replicated-row recipes of
  sglang layer.py USPAttention._forward_with_replicated_prefix / _suffix /
  _kv_prefix.
"""
import itertools

import numpy as np
import pytest
import torch

import oracle
from oracle import Shape, REP_NONE, REP_PREFIX, REP_SUFFIX, REP_KV_PREFIX

MODES = [REP_NONE, REP_PREFIX, REP_SUFFIX, REP_KV_PREFIX]


def _shape(B, P, S_l, R, mode, Hq, Hkv, D):
    return Shape(B, P, S_l, R if mode != REP_NONE else 0, mode, Hq, Hkv, D)


def _consistent_shards(s: Shape, is_kv: bool, rng, dtype=np.int32):
    """Random shards whose replicated rows agree across shards."""
    H = s.Hkv if is_kv else s.Hq
    rs = oracle.shard_rows(s, is_kv)
    rep_rows = rs - s.S_l
    rep = rng.integers(-2**30, 2**30, size=(s.B, rep_rows, H, s.D)).astype(dtype)
    out = []
    for _ in range(s.P):
        img = rng.integers(-2**30, 2**30, size=(s.B, s.S_l, H, s.D)).astype(dtype)
        if rep_rows == 0:
            out.append(img)
        elif s.mode == REP_SUFFIX:
            out.append(np.ascontiguousarray(np.concatenate([img, rep], axis=1)))
        else:
            out.append(np.ascontiguousarray(np.concatenate([rep, img], axis=1)))
    return out


CASES = [(B, P, S_l, R, mode) for B in (1, 2) for P in (1, 2, 3, 4) for (S_l, R) in ((5, 3), (7, 1))
         for mode in MODES]


@pytest.mark.parametrize("B,P,S_l,R,mode", CASES)
def test_round_trip_is_identity(B, P, S_l, R, mode):
    s = _shape(B, P, S_l, R, mode, Hq=2 * P, Hkv=P, D=3)
    rng = np.random.default_rng(7)
    x = _consistent_shards(s, False, rng)
    back = oracle.to_seq(s, oracle.to_heads(s, False, x))
    for a, b in zip(x, back):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("is_kv", [False, True])
def test_single_rank_is_identity(mode, is_kv):
    s = _shape(2, 1, 9, 4, mode, Hq=4, Hkv=2, D=5)
    rng = np.random.default_rng(3)
    x = _consistent_shards(s, is_kv, rng)
    y = oracle.to_heads(s, is_kv, x)
    np.testing.assert_array_equal(x[0], y[0])


def _iota(s: Shape, is_kv: bool):
    """Shard p element (b,row,h,d) holds the int64 code of its coordinates."""
    H = s.Hkv if is_kv else s.Hq
    rs = oracle.shard_rows(s, is_kv)
    out = []
    for p in range(s.P):
        b, row, h, d = np.meshgrid(np.arange(s.B), np.arange(rs), np.arange(H), np.arange(s.D), indexing="ij")
        out.append(np.ascontiguousarray((((p * 100 + b) * 10000 + row) * 100 + h) * 100 + d, dtype=np.int64))
    return out


def _decode(code):
    d = code % 100
    h = (code // 100) % 100
    row = (code // 10000) % 10000
    b = (code // 100000000) % 100
    p = code // 10000000000
    return p, b, row, h, d


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("is_kv", [False, True])
def test_iota_image(mode, is_kv):
    s = _shape(2, 3, 4, 2, mode, Hq=6, Hkv=3, D=2)
    H = s.Hkv if is_kv else s.Hq
    Hl = H // s.P
    x = _iota(s, is_kv)
    y = oracle.to_heads(s, is_kv, x)
    rs = oracle.shard_rows(s, is_kv)
    rep_rows = rs - s.S_l
    rep_first = s.mode in (REP_PREFIX, REP_KV_PREFIX)
    seen = {}
    for r in range(s.P):
        p, b, row, h, d = _decode(y[r])
        # rank r holds exactly its own heads, d and b unchanged
        assert np.all(h // Hl == r)
        assert np.array_equal(h % Hl, np.broadcast_to(np.arange(Hl)[None, None, :, None], h.shape))
        assert np.array_equal(d, np.broadcast_to(np.arange(s.D), d.shape))
        assert np.array_equal(b, np.broadcast_to(np.arange(s.B)[:, None, None, None], b.shape))
        n_rows = y[r].shape[1]
        for n in range(n_rows):
            pp, rr = int(p[0, n, 0, 0]), int(row[0, n, 0, 0])
            is_rep = (rr < rep_rows) if rep_first else (rr >= s.S_l)
            if is_rep:
                assert pp == r, "replicated rows come from the rank's own shard"
                key = ("rep", rr)
            else:
                key = ("img", pp, rr)
            seen.setdefault(key, []).append((r, n))
    img_keys = [k for k in seen if k[0] == "img"]
    rep_keys = [k for k in seen if k[0] == "rep"]
    # every image row of every shard appears once per rank, rows are
    # sender-rank-major and in shard order; replicated rows once per rank
    assert len(img_keys) == s.P * s.S_l
    assert all(len(seen[k]) == s.P for k in img_keys)
    assert len(rep_keys) == rep_rows
    assert all(len(seen[k]) == s.P for k in rep_keys)
    for r in range(s.P):
        img_order = [(k[1], k[2]) for k in sorted(img_keys, key=lambda k: [n for (rr, n) in seen[k] if rr == r][0])]
        assert img_order == sorted(img_order)
        rep_pos = sorted(n for k in rep_keys for (rr, n) in seen[k] if rr == r)
        if rep_rows:
            if rep_first:
                assert rep_pos == list(range(rep_rows))
            else:
                assert rep_pos == list(range(s.P * s.S_l, s.P * s.S_l + rep_rows))


# ---- an independent formulation: torch over P virtual ranks ------------------

def _a2a_chunks(xs):
    """all_to_all with scatter on heads, gather on sequence (sender-major)."""
    P = len(xs)
    parts = [x.chunk(P, dim=2) for x in xs]
    return [torch.cat([parts[p][r] for p in range(P)], dim=1) for r in range(P)]


def _a2a_reshape(xs):
    """The same exchange through the reshape/permute + all_to_all_single
    chain of cp.py (there in bhsd; here the bshd equivalent): every sender
    lays out [P_dst, S, B, H_l, D], the exchange hands block r of every
    sender to rank r, and the receiver flattens (sender, S) and returns to
    [B, P*S, H_l, D]."""
    P = len(xs)
    B, S, H, D = xs[0].shape
    send = [x.reshape(B, S, P, H // P, D).permute(2, 1, 0, 3, 4).contiguous() for x in xs]
    recv = [torch.stack([send[p][r] for p in range(P)]) for r in range(P)]  # [P_src, S, B, H_l, D]
    return [y.flatten(0, 1).permute(1, 0, 2, 3).contiguous() for y in recv]


def _a2a_back(ys, S):
    """Inverse exchange: scatter on sequence, gather on heads."""
    P = len(ys)
    parts = [y.split(S, dim=1) for y in ys]
    return [torch.cat([parts[r][p] for r in range(P)], dim=2) for p in range(P)]


def _torch_to_heads(s: Shape, is_kv, xs):
    P, R = s.P, s.R
    H = s.Hkv if is_kv else s.Hq
    Hl = H // P
    if s.mode == REP_NONE or (s.mode == REP_KV_PREFIX and not is_kv):
        return _a2a_chunks(xs)
    if s.mode in (REP_PREFIX, REP_KV_PREFIX):
        shard = _a2a_chunks([x[:, R:] for x in xs])
        return [torch.cat([xs[r][:, :R, r * Hl:(r + 1) * Hl], shard[r]], dim=1) for r in range(P)]
    # suffix: rotate to a prefix, run the prefix recipe, rotate back
    rot = [torch.cat([x[:, -R:], x[:, :-R]], dim=1) for x in xs]
    pre = _torch_to_heads(Shape(s.B, P, s.S_l, R, REP_PREFIX, s.Hq, s.Hkv, s.D), is_kv, rot)
    return [torch.cat([y[:, R:], y[:, :R]], dim=1) for y in pre]


def _torch_to_seq(s: Shape, ys):
    P, R = s.P, s.R
    if s.mode in (REP_NONE, REP_KV_PREFIX):
        return _a2a_back(ys, s.S_l)
    if s.mode == REP_PREFIX:
        rep = torch.cat([y[:, :R] for y in ys], dim=2)  # all-gather over heads
        back = _a2a_back([y[:, R:] for y in ys], s.S_l)
        return [torch.cat([rep, b], dim=1) for b in back]
    rot = [torch.cat([y[:, -R:], y[:, :-R]], dim=1) for y in ys]
    pre = _torch_to_seq(Shape(s.B, P, s.S_l, R, REP_PREFIX, s.Hq, s.Hkv, s.D), rot)
    return [torch.cat([x[:, R:], x[:, :R]], dim=1) for x in pre]


@pytest.mark.parametrize("B,P,mode", list(itertools.product((1, 2), (2, 4), MODES)))
def test_matches_torch_formulation(B, P, mode):
    s = _shape(B, P, 6, 3, mode, Hq=2 * P, Hkv=P, D=4)
    rng = np.random.default_rng(11)
    for is_kv in (False, True):
        x = _consistent_shards(s, is_kv, rng, dtype=np.int64)
        want = _torch_to_heads(s, is_kv, [torch.from_numpy(a) for a in x])
        got = oracle.to_heads(s, is_kv, x)
        for a, b in zip(got, want):
            np.testing.assert_array_equal(a, b.numpy())
    y = [rng.integers(0, 2**40, size=(B, oracle.heads_rows(s, False), s.Hq // P, s.D)) for _ in range(P)]
    want = _torch_to_seq(s, [torch.from_numpy(a) for a in y])
    got = oracle.to_seq(s, y)
    for a, b in zip(got, want):
        np.testing.assert_array_equal(a, b.numpy())


@pytest.mark.parametrize("P", [2, 4])
def test_reshape_chain_agrees_with_chunks(P):
    rng = np.random.default_rng(5)
    xs = [torch.from_numpy(rng.integers(0, 1000, size=(2, 5, 2 * P, 3))) for _ in range(P)]
    for a, b in zip(_a2a_chunks(xs), _a2a_reshape(xs)):
        assert torch.equal(a, b)
    s = Shape(2, P, 5, 0, REP_NONE, 2 * P, 2 * P, 3)
    got = oracle.to_heads(s, False, [x.numpy() for x in xs])
    for a, b in zip(got, _a2a_reshape(xs)):
        np.testing.assert_array_equal(a, b.numpy())


@pytest.mark.parametrize("bad", [
    dict(Hq=6, Hkv=6, P=4),      # heads not divisible by ranks
    dict(Hq=8, Hkv=3, P=1),      # q heads not a multiple of kv heads
    dict(Hq=8, Hkv=8, P=2, mode=REP_NONE, R=4),   # rows replicated without a mode
    dict(Hq=8, Hkv=8, P=2, mode=REP_PREFIX, R=0),  # a mode without rows
])
def test_check_rejects(bad):
    kw = dict(B=1, P=2, S_l=4, R=0, mode=REP_NONE, Hq=8, Hkv=8, D=4)
    kw.update(bad)
    assert not oracle.check(Shape(**kw))
    assert oracle.check(Shape(**dict(kw, Hq=8, Hkv=8, P=2, mode=REP_PREFIX, R=2)))


# ---- uneven shards (seq_lens) ------------------------------------------------

def _uneven_shards(s: Shape, is_kv: bool, rng, dtype=np.int64):
    H = s.Hkv if is_kv else s.Hq
    rep_rows = oracle.shard_rows(s, is_kv, 0) - s.lens[0]
    rep = rng.integers(-2**40, 2**40, size=(s.B, rep_rows, H, s.D)).astype(dtype)
    out = []
    for p in range(s.P):
        img = rng.integers(-2**40, 2**40, size=(s.B, s.lens[p], H, s.D)).astype(dtype)
        if rep_rows == 0:
            out.append(img)
        elif s.mode == REP_SUFFIX:
            out.append(np.ascontiguousarray(np.concatenate([img, rep], axis=1)))
        else:
            out.append(np.ascontiguousarray(np.concatenate([rep, img], axis=1)))
    return out


UNEVEN = [(mode, lens) for mode in MODES for lens in ((5, 1, 7), (3, 3, 9, 1), (2, 11))]


@pytest.mark.parametrize("mode,lens", UNEVEN)
def test_uneven_round_trip_and_torch_formulation(mode, lens):
    P = len(lens)
    s = Shape(2, P, 0, 3 if mode != REP_NONE else 0, mode, 2 * P, P, 3, lens=lens)
    rng = np.random.default_rng(sum(lens) + mode)
    x = _uneven_shards(s, False, rng)
    y = oracle.to_heads(s, False, x)
    back = oracle.to_seq(s, y)
    for a, b in zip(x, back):
        np.testing.assert_array_equal(a, b)
    # the varlen all-to-all: rank r gets its head slice of every shard's
    # rows, concatenated in sender order (torch chunk/cat, uneven sizes)
    for is_kv in (False, True):
        xs = _uneven_shards(s, is_kv, rng)
        got = oracle.to_heads(s, is_kv, xs)
        H = s.Hkv if is_kv else s.Hq
        Hl = H // P
        R = s.R
        t = [torch.from_numpy(a) for a in xs]
        rep_first = mode == REP_PREFIX or (mode == REP_KV_PREFIX and is_kv)
        rep_last = mode == REP_SUFFIX
        for r in range(P):
            if rep_first:
                parts = [t[r][:, :R, r * Hl:(r + 1) * Hl]] + [a[:, R:, r * Hl:(r + 1) * Hl] for a in t]
            elif rep_last:
                parts = [a[:, :lens[p], r * Hl:(r + 1) * Hl] for p, a in enumerate(t)] + \
                        [t[r][:, lens[r]:, r * Hl:(r + 1) * Hl]]
            else:
                parts = [a[:, :, r * Hl:(r + 1) * Hl] for a in t]
            np.testing.assert_array_equal(got[r], torch.cat(parts, dim=1).numpy())


@pytest.mark.parametrize("lens", [(4, 1, 6), (1, 1), (9, 2, 2, 5)])
def test_uneven_iota_exactly_once(lens):
    P = len(lens)
    s = Shape(1, P, 0, 2, REP_PREFIX, 2 * P, 2 * P, 2, lens=lens)
    xs = []
    for p in range(P):
        rs = oracle.shard_rows(s, False, p)
        b, row, h, d = np.meshgrid(np.arange(1), np.arange(rs), np.arange(2 * P), np.arange(2), indexing="ij")
        xs.append(np.ascontiguousarray((((p * 100 + b) * 10000 + row) * 100 + h) * 100 + d, dtype=np.int64))
    ys = oracle.to_heads(s, False, xs)
    seen = {}
    for r, y in enumerate(ys):
        codes = y.reshape(-1)
        for c in codes:
            seen[int(c)] = seen.get(int(c), 0) + 1
    # every image element of every shard once; replicated rows once per rank
    for p, x in enumerate(xs):
        for c in x[:, 2:].reshape(-1):
            assert seen.pop(int(c)) == 1
    assert all(v == 1 for v in seen.values())  # rank r's copy of the prefix, its own head slice


@pytest.mark.parametrize("mode", MODES)
def test_equal_lengths_reduce_to_even(mode):
    # lens = (S_l, ..., S_l) must give the even oracle's result exactly
    P, S = 3, 5
    even = Shape(2, P, S, 4 if mode != REP_NONE else 0, mode, 2 * P, P, 3)
    lens = Shape(2, P, 0, even.R, mode, 2 * P, P, 3, lens=(S,) * P)
    rng = np.random.default_rng(mode + 40)
    for is_kv in (False, True):
        xs = _uneven_shards(lens, is_kv, rng)
        a = oracle.to_heads(even, is_kv, xs)
        b = oracle.to_heads(lens, is_kv, xs)
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)
        if not is_kv:  # to_seq takes the q-shaped (output) tensors
            for x, y in zip(oracle.to_seq(even, a), oracle.to_seq(lens, b)):
                np.testing.assert_array_equal(x, y)
