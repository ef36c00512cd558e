"""The oracle's whole path (to_heads -> per-rank attention -> to_seq) against
torch fp64 SDPA over the global layout with every head at once -- the check
sglang PR #43521 applies to its pipelined exchange ("Accuracy Tests": each
case byte for byte against attention over the global layout).  CPU only."""
import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import Shape


def _oracle_path(w, data, zero_rows=False):
    s = Shape(w.B, w.P, w.S_l, w.R, w.rep_mode, w.Hq, w.Hkv, w.D, lens=w.lens)
    qh = oracle.to_heads(s, False, data["q"])
    kh = oracle.to_heads(s, True, data["k"])
    vh = oracle.to_heads(s, True, data["v"])
    Hl, Hkl = w.Hq // w.P, w.Hkv // w.P
    oh = []
    for r in range(w.P):
        sl = lambda a, n: None if a is None else a[r * n:(r + 1) * n]
        koff = w.R if w.mode == "kv_prefix" else 0
        oh.append(oracle.attention(qh[r], kh[r], vh[r], data["key_mask"], data["scale"],
                                   sl(data["q_scale"], Hl), sl(data["k_scale"], Hkl), sl(data["v_scale"], Hkl),
                                   zero_masked_rows=zero_rows, q_key_offset=koff))
    return oracle.to_seq(s, oh)


def _global(w, shards, is_kv):
    """Global sequence in key order, rebuilt from the shards with numpy."""
    has_rep = w.rows_global(is_kv) != w.n_img
    if not has_rep:
        return np.concatenate(shards, axis=1)
    if w.mode == "suffix":
        return np.concatenate([x[:, :w.shard_len(p)] for p, x in enumerate(shards)] +
                              [shards[0][:, w.shard_len(0):]], axis=1)
    return np.concatenate([shards[0][:, :w.R]] + [x[:, w.R:] for x in shards], axis=1)


def _decode(a, scale):
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(torch.float64)
    t = torch.from_numpy(a).view(torch.float8_e4m3fn).to(torch.float64)
    return t * torch.from_numpy(scale.astype(np.float64))[None, None, :, None]


SMALL = {
    "tiny": synth.WORKLOADS["tiny"],
    "wan14b-small": synth.WORKLOADS["wan14b"].scaled(S_l=40, R=24, valid=((0, 9), (24, 24 + 160)), Hq=8, Hkv=8),
    "gqa-small": synth.WORKLOADS["gqa"].scaled(S_l=24, R=16, Hq=8, Hkv=4),
    "fp8-small": synth.WORKLOADS["fp8"].scaled(P=4, S_l=30, R=20, Hq=8, Hkv=8, valid=((0, 120 + 7),)),
    "wan1.3b-small": synth.WORKLOADS["wan1.3b"].scaled(S_l=33, Hq=8, Hkv=8),
    "uneven-prefix": synth.WORKLOADS["wan14b"].scaled(S_l=0, lens=(41, 7, 30), P=3, R=20, Hq=6, Hkv=6,
                                                    valid=((0, 9), (20, 98))),
    "uneven-suffix": synth.WORKLOADS["fp8"].scaled(P=2, S_l=0, lens=(25, 61), R=9, Hq=4, Hkv=4, valid=((0, 90),)),
    "uneven-kvprefix": synth.WORKLOADS["gqa"].scaled(S_l=0, lens=(13, 31, 5, 20), R=8, Hq=8, Hkv=4),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_path_matches_global_sdpa(name):
    w = SMALL[name]
    data = synth.generate(w)
    outs = _oracle_path(w, data)
    qg = _decode(_global(w, data["q"], False), data["q_scale"])
    kg = _decode(_global(w, data["k"], True), data["k_scale"])
    vg = _decode(_global(w, data["v"], True), data["v_scale"])
    G = w.Hq // w.Hkv
    mask = None if data["key_mask"] is None else torch.from_numpy(data["key_mask"].astype(bool))[:, None, None, :]
    og = torch.nn.functional.scaled_dot_product_attention(
        qg.transpose(1, 2), kg.transpose(1, 2).repeat_interleave(G, 1), vg.transpose(1, 2).repeat_interleave(G, 1),
        attn_mask=mask, scale=data["scale"]).transpose(1, 2).numpy()
    # split the global output back into shards the way the inputs were split
    for p in range(w.P):
        a, b = w.img_off(p), w.img_off(p + 1)
        if w.mode in ("prefix",):
            want = np.concatenate([og[:, :w.R], og[:, w.R + a:w.R + b]], axis=1)
        elif w.mode == "suffix":
            want = np.concatenate([og[:, a:b], og[:, w.n_img:]], axis=1)
        else:
            want = og[:, a:b]
        np.testing.assert_allclose(outs[p], want, rtol=1e-12, atol=1e-12)


def test_zero_rows_path():
    w = SMALL["tiny"]
    data = synth.generate(w)
    a = _oracle_path(w, data)
    z = _oracle_path(w, data, zero_rows=True)
    for p in range(w.P):
        # prefix rows 10..15 are masked keys, so those query rows read zero
        assert np.all(z[p][:, 10:16] == 0)
        np.testing.assert_array_equal(z[p][:, :10], a[p][:, :10])
        np.testing.assert_array_equal(z[p][:, 16:], a[p][:, 16:])
