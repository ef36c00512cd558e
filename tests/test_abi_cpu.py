"""C ABI on the CPU: the library builds and exports every declared symbol;
argument validation and the automatic head-group rule need no GPU."""
import ctypes
import os
import re

import pytest

import ulysses_sequence_attention_uly_gb300 as uly

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    text = open(os.path.join(ROOT, "include", "uly.h")).read()
    return sorted(set(re.findall(r"^\s*[\w\s\*]+?\b(uly_\w+)\s*\(", text, flags=re.M)))


def test_library_exports_every_declared_symbol():
    L = uly.lib()
    decl = _declared()
    assert len(decl) >= 13
    for name in decl:
        assert hasattr(L, name), name
    assert sorted(uly.EXPORTS) == decl


def _create(**kw):
    d = dict(B=1, P=4, S_l=64, R=0, rep_mode=0, Hq=8, Hkv=8, D=128, dtype=0, masked_rows=0)
    d.update(kw)
    desc = uly._Desc(*[d[n] for n in ("B", "P", "S_l", "R", "rep_mode", "Hq", "Hkv", "D", "dtype", "masked_rows")])
    h = ctypes.c_void_p()
    rc = uly.lib().uly_plan_create(ctypes.byref(desc), 0, ctypes.byref(h))
    if rc == 0:
        uly.lib().uly_plan_destroy(h)
    return rc


@pytest.mark.parametrize("kw,want", [
    (dict(Hq=6, Hkv=6), uly.ULY_ERR_INVALID),                 # heads not divisible by P
    (dict(Hq=8, Hkv=3, P=1), uly.ULY_ERR_INVALID),            # Hq not a multiple of Hkv
    (dict(R=16), uly.ULY_ERR_INVALID),                         # replicated rows without a mode
    (dict(rep_mode=1, R=0), uly.ULY_ERR_INVALID),             # a mode without rows
    (dict(rep_mode=7, R=4), uly.ULY_ERR_INVALID),             # unknown mode
    (dict(B=0), uly.ULY_ERR_INVALID),
    (dict(S_l=0), uly.ULY_ERR_INVALID),
    (dict(dtype=5), uly.ULY_ERR_INVALID),
    (dict(masked_rows=3), uly.ULY_ERR_INVALID),
    (dict(D=96), uly.ULY_ERR_UNSUPPORTED),
    (dict(D=64, dtype=1), uly.ULY_ERR_UNSUPPORTED),           # e4m3 needs D = 128
    (dict(P=32, Hq=64, Hkv=64), uly.ULY_ERR_UNSUPPORTED),     # more ranks than the ABI holds
    (dict(P=17, Hq=17, Hkv=17), uly.ULY_ERR_UNSUPPORTED),     # one rank past the limit (16)
])
def test_plan_create_rejects(kw, want):
    assert _create(**kw) == want


def _create_varlen(lens, **kw):
    d = dict(B=1, P=len(lens), S_l=0, R=0, rep_mode=0, Hq=8, Hkv=8, D=128, dtype=0, masked_rows=0)
    d.update(kw)
    desc = uly._Desc(*[d[n] for n in ("B", "P", "S_l", "R", "rep_mode", "Hq", "Hkv", "D", "dtype", "masked_rows")])
    arr = (ctypes.c_int32 * len(lens))(*lens)
    h = ctypes.c_void_p()
    rc = uly.lib().uly_plan_create_varlen(ctypes.byref(desc), arr, 0, ctypes.byref(h))
    if rc == 0:
        uly.lib().uly_plan_destroy(h)
    return rc


@pytest.mark.parametrize("lens,kw,want", [
    ((5, 0, 7, 9), {}, uly.ULY_ERR_INVALID),                    # an empty shard
    ((5, -3, 7, 9), {}, uly.ULY_ERR_INVALID),
    ((1 << 26, 1 << 26, 1, 1), {}, uly.ULY_ERR_UNSUPPORTED),    # rows beyond the int32 tile indexing
    ((5, 6, 7), {}, uly.ULY_ERR_INVALID),                       # 8 heads over 3 ranks
])
def test_plan_create_varlen_rejects(lens, kw, want):
    assert _create_varlen(lens, **kw) == want


def test_plan_create_varlen_ignores_s_l():
    # S_l = 0 is invalid for an even plan but ignored with shard lengths: the
    # shape passes validation and only the device query fails without a GPU
    rc = _create_varlen((5, 6, 7, 8))
    import torch
    assert rc == (uly.ULY_OK if torch.cuda.is_available() else uly.ULY_ERR_CUDA)
    assert uly.lib().uly_plan_create_varlen(None, None, 0, None) == uly.ULY_ERR_INVALID


def test_null_arguments():
    L = uly.lib()
    assert L.uly_plan_create(None, 0, None) == uly.ULY_ERR_INVALID
    assert L.uly_plan_rows(None, 0) == -1
    assert L.uly_to_seq(None, None, None, None) == uly.ULY_ERR_INVALID
    assert L.uly_sync_status(None, None) == uly.ULY_ERR_INVALID
    bounds = (ctypes.c_int32 * 3)(0, 1, 2)
    assert L.uly_ring_attention(None, None, None, None, None, None, 0, bounds, ctypes.c_float(0.125), 0, None, None,
                                None, None, None, None) == uly.ULY_ERR_INVALID
    L.uly_plan_destroy(None)


@pytest.mark.parametrize("args,want", [
    # (hq_local, hkv_local, q_rows, B*P, SMs): the source page's automatic group count
    ((10, 10, 27792, 4, 152), 5),   # Wan2.1 14B-like, P=4: 5 groups of 2 heads per rank
    ((3, 3, 32760, 4, 152), 3),     # Wan2.1 1.3B-like, P=4: three one-head groups
    ((8, 2, 16384, 8, 152), 2),     # GQA: 4 q heads + 1 kv head per group
    ((5, 5, 76112, 8, 152), 5),     # 40 heads over 8 ranks
    ((2, 2, 128, 2, 152), 1),       # too short to fill four waves: whole call
    ((7, 7, 10 ** 6, 1, 1), 7),     # largest candidate first
    ((6, 6, 10 ** 6, 1, 1), 3),     # 7, 5, 4 do not divide 6
    ((4, 2, 10 ** 6, 1, 1), 2),     # must also divide the kv heads
    ((11, 11, 10 ** 6, 1, 1), 1),   # prime: nothing divides
    ((0, 1, 1, 1, 1), -1),
])
def test_pick_head_groups(args, want):
    assert uly.pick_head_groups(*args) == want


def test_pick_head_groups_waves_threshold():
    # exactly four waves qualifies, one tile fewer does not
    sm = 152
    tiles_needed = 4 * sm  # batch_ranks * (hq/g) * tiles >= 4 * sm with hq/g = 1, batch_ranks = 1
    assert uly.pick_head_groups(2, 2, tiles_needed * 128, 1, sm) == 2
    assert uly.pick_head_groups(2, 2, (tiles_needed - 1) * 128, 1, sm) == 1


def test_status_strings():
    L = uly.lib()
    for st in range(5):
        assert L.uly_status_string(st)
    assert L.uly_status_string(99) == b"unknown status"
