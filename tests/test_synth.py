"""Seeded input generation: shapes, determinism, replicated rows, fp8 scales."""
import numpy as np
import pytest

import synth


def test_workload_table():
    w = synth.WORKLOADS
    assert w["wan14b"].n_img == 27280 and w["wan14b"].rows_global(True) == 27792
    assert w["wan1.3b"].n_img == 32760
    assert w["gqa"].n_img == 16384 and w["gqa"].rows_global(False) == 16384 and w["gqa"].rows_global(True) == 16640
    assert w["fp8"].n_img == 75600 and w["fp8"].rows_global(True) == 76112
    assert w["tiny"].rows_shard(False) == 72 and w["tiny"].P * w["tiny"].rows_shard(False) == 144


@pytest.mark.parametrize("name", ["tiny"])
def test_deterministic_and_replicated(name):
    w = synth.WORKLOADS[name]
    a, b = synth.generate(w), synth.generate(w)
    for t in ("q", "k", "v"):
        for x, y in zip(a[t], b[t]):
            np.testing.assert_array_equal(x, y)
        # replicated prefix rows are the same bytes on every shard
        for x in a[t][1:]:
            np.testing.assert_array_equal(x[:, :w.R], a[t][0][:, :w.R])
    m = a["key_mask"]
    assert m.shape == (1, 128) and m[0, :10].all() and not m[0, 10:16].any() and m[0, 16:].all()


def test_fp8_scales():
    w = synth.WORKLOADS["fp8"].scaled(P=2, S_l=20, R=8, Hq=4, Hkv=4, valid=((0, 45),))
    d = synth.generate(w)
    import torch
    for t in ("q", "k", "v"):
        s = d[t + "_scale"]
        assert s.shape == (4,) and np.all(s > 0)
        vals = np.concatenate([torch.from_numpy(x).view(torch.float8_e4m3fn).float().numpy() for x in d[t]], axis=1)
        assert np.all(np.abs(vals) <= 448.0)
        assert np.allclose(np.abs(vals).max(axis=(0, 1, 3)), 448.0)
    rs = d["workload"].rows_shard(False)
    assert d["q"][0].shape == (1, rs, 4, 128) and d["q"][0].dtype == np.uint8
    # suffix rows replicated
    for x in d["k"][1:]:
        np.testing.assert_array_equal(x[:, w.S_l:], d["k"][0][:, w.S_l:])
