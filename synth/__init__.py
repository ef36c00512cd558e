"""Seeded synthetic inputs for the Ulysses attention hot path.

This module is shared by the tests, the benchmark and the CPU oracle's
callers.  It holds none of the method's arithmetic: it draws seeded normal
values, rounds them to the storage type (bf16, or e4m3 with a per-head absmax
scale as the fp8 configuration prescribes), lays out each shard's
seq-sharded tensor (its image rows plus, where the workload has them, a copy
of the replicated text rows) and writes the key-validity mask.

Workloads (the shapes the source pages benchmark; values are synthetic):

* ``tiny``     B=1, P=2, 56 image rows per shard + 16-row replicated prefix
               (keys 0..9 valid, 10..15 masked), H=4, D=64, bf16 N(0,1).
* ``wan1.3b``  B=1, P=4, 8190 rows per shard, no text, H=12, D=128,
               bf16 0.5*N(0,1); unmasked.
* ``wan14b``   B=1, P=4, 6820 rows per shard + 512-row replicated prefix of
               which the first 226 keys are valid, H=40, D=128, bf16 N(0,1).
* ``gqa``      B=2, P=4, 4096 rows per shard, Hq=32, Hkv=8, D=128, a 256-row
               K/V-only replicated prefix; Q N(0,1), K/V 0.7*N(0,1).
* ``fp8``      B=1, P=8, 9450 rows per shard + 512-row replicated suffix with
               300 valid keys, H=40, D=128; e4m3 from N(0,1) with per-head
               absmax scales; bf16 output.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np

REP_MODES = {"none": 0, "prefix": 1, "suffix": 2, "kv_prefix": 3}


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    P: int
    S_l: int
    R: int
    mode: str
    Hq: int
    Hkv: int
    D: int
    dtype: str  # "bf16" or "e4m3"
    std_q: float
    std_kv: float
    seed: int
    # valid keys per batch as half-open ranges in global key order; None = all
    valid: tuple | None = None
    head_groups: int = 1
    notes: str = field(default="", compare=False)
    # uneven shards: image rows of each shard (replaces S_l), or None
    lens: tuple | None = None

    @property
    def rep_mode(self) -> int:
        return REP_MODES[self.mode]

    def shard_len(self, p: int) -> int:
        return self.S_l if self.lens is None else self.lens[p]

    def img_off(self, p: int) -> int:
        return sum(self.shard_len(q) for q in range(p))

    @property
    def n_img(self) -> int:
        return self.img_off(self.P)

    def rows_shard(self, is_kv: bool, p: int = 0) -> int:
        if self.mode == "none":
            return self.shard_len(p)
        if self.mode == "kv_prefix" and not is_kv:
            return self.shard_len(p)
        return self.shard_len(p) + self.R

    def rows_global(self, is_kv: bool) -> int:
        if self.mode == "none":
            return self.n_img
        if self.mode == "kv_prefix" and not is_kv:
            return self.n_img
        return self.n_img + self.R

    @property
    def elem_size(self) -> int:
        return 1 if self.dtype == "e4m3" else 2

    def scaled(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    "tiny": Workload("tiny", B=1, P=2, S_l=56, R=16, mode="prefix", Hq=4, Hkv=4, D=64, dtype="bf16",
                     std_q=1.0, std_kv=1.0, seed=0, valid=((0, 10), (16, 128)), head_groups=1),
    "wan1.3b": Workload("wan1.3b", B=1, P=4, S_l=8190, R=0, mode="none", Hq=12, Hkv=12, D=128, dtype="bf16",
                        std_q=0.5, std_kv=0.5, seed=1, valid=None, head_groups=3),
    "wan14b": Workload("wan14b", B=1, P=4, S_l=6820, R=512, mode="prefix", Hq=40, Hkv=40, D=128, dtype="bf16",
                       std_q=1.0, std_kv=1.0, seed=2, valid=((0, 226), (512, 512 + 27280)), head_groups=5),
    "gqa": Workload("gqa", B=2, P=4, S_l=4096, R=256, mode="kv_prefix", Hq=32, Hkv=8, D=128, dtype="bf16",
                    std_q=1.0, std_kv=0.7, seed=3, valid=None, head_groups=2),
    "fp8": Workload("fp8", B=1, P=8, S_l=9450, R=512, mode="suffix", Hq=40, Hkv=40, D=128, dtype="e4m3",
                    std_q=1.0, std_kv=1.0, seed=4, valid=((0, 75600 + 300),), head_groups=5),
}


def _round_bf16(x: np.ndarray) -> np.ndarray:
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def _quant_e4m3(x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Per-head absmax scaling of a [B, N, H, D] float32 tensor to e4m3 bytes.
    scale_h = max(absmax_h, 1e-12) / 448 so that |x / scale_h| <= 448."""
    import torch
    amax = np.abs(x).max(axis=(0, 1, 3)).astype(np.float32)
    scale = (np.maximum(amax, np.float32(1e-12)) / np.float32(448.0)).astype(np.float32)
    y = torch.from_numpy(np.ascontiguousarray(x / scale[None, None, :, None], dtype=np.float32))
    y8 = y.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    return y8, scale


def _draw(w: Workload, which: int, rows: int, heads: int, std: float) -> np.ndarray:
    rng = np.random.default_rng([w.seed, which])
    x = rng.standard_normal((w.B, rows, heads, w.D), dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def shard_rows_index(w: Workload, p: int, is_kv: bool) -> np.ndarray:
    """Global row indices of shard p's rows, in the shard's row order.  The
    global tensor holds replicated rows first (prefix / kv-prefix) or last
    (suffix), image rows in between; every shard holds the replicated rows
    (before its image rows, or after them for a suffix)."""
    a, b = w.img_off(p), w.img_off(p + 1)
    if w.rows_global(is_kv) == w.n_img:
        return np.arange(a, b)
    if w.mode == "suffix":
        return np.concatenate([np.arange(a, b), np.arange(w.n_img, w.n_img + w.R)])
    return np.concatenate([np.arange(w.R), np.arange(w.R + a, w.R + b)])


def _split_shards(w: Workload, g: np.ndarray, is_kv: bool) -> list[np.ndarray]:
    """Global rows -> per-shard tensors (see shard_rows_index)."""
    return [np.ascontiguousarray(g[:, shard_rows_index(w, p, is_kv)]) for p in range(w.P)]


def key_mask(w: Workload) -> np.ndarray | None:
    """[B, Nk] uint8 validity of every key in global key order, or None."""
    if w.valid is None:
        return None
    nk = w.rows_global(True)
    m = np.zeros((w.B, nk), dtype=np.uint8)
    for (a, b) in w.valid:
        m[:, a:b] = 1
    return m


def key_ranges(w: Workload) -> np.ndarray | None:
    """[B, n, 2] int32 half-open valid key ranges, or None."""
    if w.valid is None:
        return None
    r = np.array(w.valid, dtype=np.int32).reshape(1, -1, 2)
    return np.ascontiguousarray(np.repeat(r, w.B, axis=0))


def generate(w: Workload) -> dict:
    """Seeded shard inputs of workload ``w``.

    Returns a dict with ``q``, ``k``, ``v`` (lists of P numpy arrays
    [B, rows_shard, H, D]; uint16 bf16 bits or uint8 e4m3 bytes),
    ``q_scale``/``k_scale``/``v_scale`` (float32 per head, e4m3 only, else
    None), ``key_mask`` and ``key_ranges`` (see above) and ``scale``
    (1/sqrt(D))."""
    out = {"workload": w, "scale": float(1.0 / np.sqrt(w.D))}
    for which, (name, is_kv, heads, std) in enumerate(
            (("q", False, w.Hq, w.std_q), ("k", True, w.Hkv, w.std_kv), ("v", True, w.Hkv, w.std_kv))):
        g = _draw(w, which, w.rows_global(is_kv), heads, std)
        if w.dtype == "e4m3":
            g, s = _quant_e4m3(g)
            out[name + "_scale"] = s
        else:
            g = _round_bf16(g)
            out[name + "_scale"] = None
        out[name] = _split_shards(w, g, is_kv)
        del g
    out["key_mask"] = key_mask(w)
    out["key_ranges"] = key_ranges(w)
    return out
