"""Shared test helpers: seeded inputs to device tensors, the CUDA path through
the C ABI, and the oracle's reference for the same inputs."""
from __future__ import annotations

import numpy as np

import oracle
import synth

TOL = {"bf16": 2e-2, "e4m3": 6e-2}


def oracle_shape(w: synth.Workload) -> oracle.Shape:
    return oracle.Shape(w.B, w.P, w.S_l, w.R, w.rep_mode, w.Hq, w.Hkv, w.D, lens=w.lens)


def oracle_heads(w, data):
    s = oracle_shape(w)
    return (oracle.to_heads(s, False, data["q"]), oracle.to_heads(s, True, data["k"]),
            oracle.to_heads(s, True, data["v"]))


def _slice(a, r, n):
    return None if a is None else np.ascontiguousarray(a[r * n:(r + 1) * n])


def oracle_rank_attention(w, data, heads, r, zero_rows=False, sel=None):
    qh, kh, vh = heads
    Hl, Hkl = w.Hq // w.P, w.Hkv // w.P
    koff = w.R if w.mode == "kv_prefix" else 0
    return oracle.attention(qh[r], kh[r], vh[r], data["key_mask"], data["scale"],
                            _slice(data["q_scale"], r, Hl), _slice(data["k_scale"], r, Hkl),
                            _slice(data["v_scale"], r, Hkl), zero_masked_rows=zero_rows, q_key_offset=koff, sel=sel)


def oracle_path(w, data, zero_rows=False):
    """Oracle to_heads -> per-rank attention -> to_seq; returns (per-rank
    gathered outputs, per-shard outputs), float64."""
    heads = oracle_heads(w, data)
    oh = [oracle_rank_attention(w, data, heads, r, zero_rows) for r in range(w.P)]
    return oh, oracle.to_seq(oracle_shape(w), oh)


def within(got: np.ndarray, ref: np.ndarray, tol: float):
    err = np.abs(got.astype(np.float64) - ref)
    bound = tol * (1.0 + np.abs(ref))
    bad = ~(err <= bound)  # NaN in either operand counts as a failure
    return (not bad.any()), float(np.nanmax(err)) if err.size else 0.0, int(bad.sum())


# ------------------------------------------------------------------ device --
def dev(arrs, w):
    import torch
    out = []
    for a in arrs:
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).cuda()
        out.append(t.view(torch.bfloat16) if a.dtype == np.uint16 else t)
    return out


def dev_inputs(w, data):
    import torch
    d = {"q": dev(data["q"], w), "k": dev(data["k"], w), "v": dev(data["v"], w)}
    for n in ("q_scale", "k_scale", "v_scale"):
        d[n] = None if data[n] is None else torch.from_numpy(data[n]).cuda()
    d["key_mask"] = None if data["key_mask"] is None else torch.from_numpy(data["key_mask"]).cuda()
    d["key_ranges"] = None if data["key_ranges"] is None else torch.from_numpy(data["key_ranges"]).cuda()
    return d


def make_plan(w, masked_rows="sdpa"):
    from ulysses_sequence_attention_uly_gb300 import Plan
    return Plan(w.B, w.P, w.S_l, w.R, w.mode, w.Hq, w.Hkv, w.D, dtype=w.dtype, masked_rows=masked_rows,
                shard_lens=w.lens)


def empty_heads(plan, w, elem_dtype):
    import torch
    qh = [torch.empty((w.B, plan.heads_rows_q, w.Hq // w.P, w.D), dtype=elem_dtype, device="cuda") for _ in range(w.P)]
    kh = [torch.empty((w.B, plan.heads_rows_kv, w.Hkv // w.P, w.D), dtype=elem_dtype, device="cuda") for _ in range(w.P)]
    vh = [torch.empty_like(x) for x in kh]
    return qh, kh, vh


def in_dtype(w):
    import torch
    return torch.uint8 if w.dtype == "e4m3" else torch.bfloat16


def run_staged(plan, w, d, head_groups=0, mask="mask"):
    """to_heads -> attention -> to_seq through the C ABI; returns (oh, o)."""
    import torch
    qh, kh, vh = empty_heads(plan, w, in_dtype(w))
    plan.to_heads(d["q"], d["k"], d["v"], qh, kh, vh)
    oh = [torch.full((w.B, plan.heads_rows_q, w.Hq // w.P, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
          for _ in range(w.P)]
    km, kr = _mask_args(d, mask)
    plan.attention(qh, kh, vh, oh, key_mask=km, key_ranges=kr, head_groups=head_groups,
                   q_scale=d["q_scale"], k_scale=d["k_scale"], v_scale=d["v_scale"])
    o = [torch.full((w.B, plan.shard_rows(p), w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
         for p in range(w.P)]
    plan.to_seq(oh, o)
    return oh, o


def run_fused(plan, w, d, head_groups=0, mask="mask"):
    import torch
    o = [torch.full((w.B, plan.shard_rows(p), w.Hq, w.D), float("nan"), dtype=torch.bfloat16, device="cuda")
         for p in range(w.P)]
    km, kr = _mask_args(d, mask)
    plan.sp_attention(d["q"], d["k"], d["v"], o, key_mask=km, key_ranges=kr, head_groups=head_groups,
                      q_scale=d["q_scale"], k_scale=d["k_scale"], v_scale=d["v_scale"])
    return o


def _mask_args(d, mask):
    if mask == "mask":
        return d["key_mask"], None
    if mask == "ranges":
        return None, d["key_ranges"]
    return None, None


def assert_written(ts):
    """Outputs start NaN-filled: every element must have been written."""
    import torch
    for t in ts:
        assert not torch.isnan(t.float()).any(), "output elements left unwritten"


def host_f64(t):
    import torch
    return t.float().cpu().numpy().astype(np.float64) if t.dtype == torch.bfloat16 else t.cpu().numpy()


def bits(t):
    import torch
    return t.view(torch.int16).cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()
