"""CPU oracle for the Ulysses attention hot path (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product library never does, and this
package imports nothing from it: the two share only the seeded synthetic
inputs of ``synth``.

The arithmetic lives in ``uly_oracle.c`` (plain C, fp64, OpenMP over query
rows); this module compiles it with gcc on first use and marshals numpy
arrays through ctypes.  See ``uly_oracle.c`` for what each function computes
and which passage of the source pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "uly_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

REP_NONE, REP_PREFIX, REP_SUFFIX, REP_KV_PREFIX = 0, 1, 2, 3
BF16, E4M3, F64 = 0, 1, 2


class _Shape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "P", "S_l", "R", "mode", "Hq", "Hkv", "D")] + [
        ("lens", ctypes.POINTER(ctypes.c_int32))]


@dataclass(frozen=True)
class Shape:
    """One exchange: B batches, P ranks, S_l image rows per shard, R
    replicated rows in ``mode``, Hq/Hkv heads, head dim D; ``lens`` (a
    tuple of P row counts) makes the shards uneven and replaces S_l."""

    B: int
    P: int
    S_l: int
    R: int
    mode: int
    Hq: int
    Hkv: int
    D: int
    lens: tuple | None = None

    def c(self) -> _Shape:
        st = _Shape(self.B, self.P, self.S_l, self.R, self.mode, self.Hq, self.Hkv, self.D, None)
        if self.lens is not None:
            arr = (ctypes.c_int32 * self.P)(*self.lens)
            st.lens = ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32))
            st._keep = arr  # keeps the array alive as long as the struct
        return st


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp64, no fast-math) into oracle/_build."""
    with _lock:
        if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
            return _LIB_PATH
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.POINTER(_Shape)
        L.orc_shard_rows.restype = ctypes.c_int64
        L.orc_shard_rows.argtypes = [P, ctypes.c_int]
        L.orc_shard_rows_p.restype = ctypes.c_int64
        L.orc_shard_rows_p.argtypes = [P, ctypes.c_int, ctypes.c_int]
        L.orc_heads_rows.restype = ctypes.c_int64
        L.orc_heads_rows.argtypes = [P, ctypes.c_int]
        L.orc_check.argtypes = [P]
        L.orc_src_row.argtypes = [P, ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                  ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)]
        L.orc_out_row.restype = ctypes.c_int64
        L.orc_out_row.argtypes = [P, ctypes.c_int, ctypes.c_int64]
        vpp = ctypes.POINTER(ctypes.c_void_p)
        L.orc_to_heads.argtypes = [P, ctypes.c_int, ctypes.c_int, vpp, vpp]
        L.orc_to_seq.argtypes = [P, ctypes.c_int, vpp, vpp]
        L.orc_bf16_to_f64.restype = ctypes.c_double
        L.orc_bf16_to_f64.argtypes = [ctypes.c_uint16]
        L.orc_e4m3_to_f64.restype = ctypes.c_double
        L.orc_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        L.orc_attention.argtypes = [ctypes.c_int] * 7 + [ctypes.c_void_p] * 4 + [
            ctypes.c_double] + [ctypes.c_void_p] * 3 + [ctypes.c_int, ctypes.c_int, ctypes.c_int64,
                                                        ctypes.c_void_p, ctypes.c_void_p]
        L.orc_attention_lse.argtypes = L.orc_attention.argtypes + [ctypes.c_void_p]
        L.orc_lse_merge.argtypes = [ctypes.c_int64, ctypes.c_int] + [ctypes.c_void_p] * 6
        L.orc_lse_merge.restype = None
        L.orc_max_threads.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _ptrs(arrs):
    return (ctypes.c_void_p * len(arrs))(*[a.ctypes.data for a in arrs])


def check(s: Shape) -> bool:
    return lib().orc_check(ctypes.byref(s.c())) == 0


def shard_rows(s: Shape, is_kv: bool, p: int = 0) -> int:
    return int(lib().orc_shard_rows_p(ctypes.byref(s.c()), p, int(is_kv)))


def heads_rows(s: Shape, is_kv: bool) -> int:
    return int(lib().orc_heads_rows(ctypes.byref(s.c()), int(is_kv)))


def src_row(s: Shape, is_kv: bool, r: int, n: int) -> tuple[int, int]:
    sh, rw = ctypes.c_int32(), ctypes.c_int64()
    lib().orc_src_row(ctypes.byref(s.c()), int(is_kv), r, n, ctypes.byref(sh), ctypes.byref(rw))
    return sh.value, rw.value


def out_row(s: Shape, p: int, row: int) -> int:
    return int(lib().orc_out_row(ctypes.byref(s.c()), p, row))


def to_heads(s: Shape, is_kv: bool, shards: list[np.ndarray]) -> list[np.ndarray]:
    """Shards [B, rows_shard, H, D] -> per-rank [B, rows_heads, H/P, D] (same dtype)."""
    H = s.Hkv if is_kv else s.Hq
    assert len(shards) == s.P
    dt = shards[0].dtype
    src = [np.ascontiguousarray(x) for x in shards]
    for p, x in enumerate(src):
        assert x.shape == (s.B, shard_rows(s, is_kv, p), H, s.D) and x.dtype == dt
    out = [np.empty((s.B, heads_rows(s, is_kv), H // s.P, s.D), dtype=dt) for _ in range(s.P)]
    rc = lib().orc_to_heads(ctypes.byref(s.c()), int(is_kv), dt.itemsize, _ptrs(src), _ptrs(out))
    if rc:
        raise ValueError("oracle rejected shape %r" % (s,))
    return out


def to_seq(s: Shape, ranks: list[np.ndarray]) -> list[np.ndarray]:
    """Per-rank outputs [B, rows_heads(q), Hq/P, D] -> shards [B, rows_shard(q), Hq, D]."""
    assert len(ranks) == s.P
    dt = ranks[0].dtype
    src = [np.ascontiguousarray(x) for x in ranks]
    for x in src:
        assert x.shape == (s.B, heads_rows(s, False), s.Hq // s.P, s.D) and x.dtype == dt
    out = [np.empty((s.B, shard_rows(s, False, p), s.Hq, s.D), dtype=dt) for p in range(s.P)]
    rc = lib().orc_to_seq(ctypes.byref(s.c()), dt.itemsize, _ptrs(src), _ptrs(out))
    if rc:
        raise ValueError("oracle rejected shape %r" % (s,))
    return out


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return BF16
    if a.dtype == np.uint8:
        return E4M3
    if a.dtype == np.float64:
        return F64
    raise TypeError("oracle attention takes bf16 bits (uint16), e4m3 bytes (uint8) or float64")


def attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, key_mask: np.ndarray | None,
              scale: float, q_scale=None, k_scale=None, v_scale=None,
              zero_masked_rows: bool | int = False, q_key_offset: int = 0,
              sel: np.ndarray | None = None) -> np.ndarray:
    """fp64 attention of q [B,Nq,Hq,D] over k/v [B,Nk,Hkv,D].

    ``zero_masked_rows``: 0/False every row attends to the admitted keys,
    1/True rows whose own token is masked are zero, 2 masked rows attend
    only to the masked keys (a segment of their own).
    ``sel`` (int32 [n,3] of (b, n, h)) restricts the output to those query
    rows and returns [n, D]; otherwise returns [B, Nq, Hq, D] float64."""
    B, Nq, Hq, D = q.shape
    _, Nk, Hkv, _ = k.shape
    assert k.shape == v.shape == (B, Nk, Hkv, D) and Hq % Hkv == 0
    code = _dtype_code(q)
    assert _dtype_code(k) == code == _dtype_code(v)
    q, k, v = (np.ascontiguousarray(x) for x in (q, k, v))
    km = None if key_mask is None else np.ascontiguousarray(key_mask, dtype=np.uint8)
    if km is not None:
        assert km.shape == (B, Nk)
    scl = [None if x is None else np.ascontiguousarray(x, dtype=np.float32) for x in (q_scale, k_scale, v_scale)]
    if sel is None:
        out = np.zeros((B, Nq, Hq, D), dtype=np.float64)
        n_sel = 0
    else:
        sel = np.ascontiguousarray(sel, dtype=np.int32).reshape(-1, 3)
        n_sel = sel.shape[0]
        out = np.zeros((n_sel, D), dtype=np.float64)
    lib().orc_attention(B, Nq, Nk, Hq, Hkv, D, code, _ptr(q), _ptr(k), _ptr(v), _ptr(km),
                        float(scale), _ptr(scl[0]), _ptr(scl[1]), _ptr(scl[2]),
                        int(zero_masked_rows), int(q_key_offset), n_sel, _ptr(sel), _ptr(out))
    return out


def attention_lse(q, k, v, key_mask, scale, q_scale=None, k_scale=None, v_scale=None,
                  zero_masked_rows=False, q_key_offset=0, sel=None):
    """As attention(), plus the per-row log-sum-exp of the admitted scores
    (-inf where no key is admitted).  Returns (out, lse)."""
    B, Nq, Hq, D = q.shape
    _, Nk, Hkv, _ = k.shape
    code = _dtype_code(q)
    q, k, v = (np.ascontiguousarray(x) for x in (q, k, v))
    km = None if key_mask is None else np.ascontiguousarray(key_mask, dtype=np.uint8)
    scl = [None if x is None else np.ascontiguousarray(x, dtype=np.float32) for x in (q_scale, k_scale, v_scale)]
    if sel is None:
        out = np.zeros((B, Nq, Hq, D)); lse = np.zeros((B, Nq, Hq)); n_sel = 0
    else:
        sel = np.ascontiguousarray(sel, dtype=np.int32).reshape(-1, 3)
        n_sel = sel.shape[0]
        out = np.zeros((n_sel, D)); lse = np.zeros(n_sel)
    lib().orc_attention_lse(B, Nq, Nk, Hq, Hkv, D, code, _ptr(q), _ptr(k), _ptr(v), _ptr(km), float(scale),
                            _ptr(scl[0]), _ptr(scl[1]), _ptr(scl[2]), int(zero_masked_rows), int(q_key_offset),
                            n_sel, _ptr(sel), _ptr(out), _ptr(lse))
    return out, lse


def lse_merge(prev_out, prev_lse, out, lse):
    """Ring-attention merge of two partial results (see uly_oracle.c)."""
    D = prev_out.shape[-1]
    po = np.ascontiguousarray(prev_out, dtype=np.float64).reshape(-1, D)
    pl = np.ascontiguousarray(prev_lse, dtype=np.float64).reshape(-1)
    o = np.ascontiguousarray(out, dtype=np.float64).reshape(-1, D)
    l = np.ascontiguousarray(lse, dtype=np.float64).reshape(-1)
    ro, rl = np.empty_like(po), np.empty_like(pl)
    lib().orc_lse_merge(po.shape[0], D, _ptr(po), _ptr(pl), _ptr(o), _ptr(l), _ptr(ro), _ptr(rl))
    return ro.reshape(np.shape(prev_out)), rl.reshape(np.shape(prev_lse))


def max_threads() -> int:
    return int(lib().orc_max_threads())


def bf16_to_f64(bits: int) -> float:
    return float(lib().orc_bf16_to_f64(bits))


def e4m3_to_f64(byte: int) -> float:
    return float(lib().orc_e4m3_to_f64(byte))
