"""GB300 (sm_103a) Ulysses sequence-parallel attention: Python binding.

A thin ctypes layer over the C ABI of ``include/uly.h`` (``libuly.so``):
it marshals torch CUDA tensors into device pointers and the current stream
and raises on a non-zero status.  Every step of the path runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback -- importing the
binding without the compiled library raises.

    plan = Plan(B=1, P=4, S_l=6820, R=512, rep_mode="prefix", Hq=40, Hkv=40, D=128)
    plan.sp_attention(q_shards, k_shards, v_shards, o_shards, key_ranges=r)

With ULY_CHECKED=1 in the environment the binding loads the checked build
of the library (index checks in every kernel; see checked_violations).
"""
from __future__ import annotations

import ctypes
import math
import os

from . import _build

ULY_OK, ULY_ERR_INVALID, ULY_ERR_UNSUPPORTED, ULY_ERR_CUDA, ULY_ERR_TIMEOUT = 0, 1, 2, 3, 4
REP_MODES = {"none": 0, "prefix": 1, "suffix": 2, "kv_prefix": 3}
DTYPES = {"bf16": 0, "e4m3": 1}
MASKED_ROWS = {"sdpa": 0, "zero": 1, "self": 2}
MAX_RANKS = 16

# every symbol include/uly.h declares
EXPORTS = ("uly_plan_create", "uly_plan_destroy", "uly_plan_set_wait_limit", "uly_plan_test_withhold_fill",
           "uly_plan_rows", "uly_pick_head_groups", "uly_to_heads", "uly_attention", "uly_to_seq",
           "uly_sp_attention", "uly_sync_status", "uly_status_string", "uly_device_sm_count",
           "uly_sp_attention_noalloc", "uly_lse_merge", "uly_pipelined_attention", "uly_plan_create_varlen",
           "uly_plan_shard_rows", "uly_sp_attention_host", "uly_checked_violations",
           "uly_plan_test_check_narrow", "uly_attention_merge", "uly_noalloc_sync_status", "uly_ring_attention")


class UlyError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what, _status_string(status), status))


class _Desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("B", "P", "S_l", "R", "rep_mode", "Hq", "Hkv", "D", "dtype", "masked_rows")]


_lib = None


def checked() -> bool:
    """Whether this process uses the checked build (ULY_CHECKED=1)."""
    return os.environ.get("ULY_CHECKED", "") == "1"


def build(force: bool = False, verbose: bool = False, checked_build: bool | None = None) -> str:
    """Compile libuly.so (or libuly_checked.so) with nvcc for sm_103a, in-tree."""
    return _build.build(force=force, verbose=verbose, checked=checked() if checked_build is None else checked_build)


def lib():
    """Load the library, compiling it first if the sources are newer."""
    global _lib
    if _lib is None:
        path = _build.build(checked=checked())
        L = ctypes.CDLL(path)
        vp, vpp = ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)
        i32, i64, u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
        L.uly_plan_create.argtypes = [ctypes.POINTER(_Desc), ctypes.c_int, ctypes.POINTER(vp)]
        L.uly_plan_create_varlen.argtypes = [ctypes.POINTER(_Desc), ctypes.POINTER(i32), ctypes.c_int,
                                             ctypes.POINTER(vp)]
        L.uly_plan_shard_rows.argtypes = [vp, i32, i32]
        L.uly_plan_shard_rows.restype = i64
        L.uly_plan_destroy.argtypes = [vp]
        L.uly_plan_destroy.restype = None
        L.uly_plan_set_wait_limit.argtypes = [vp, u64]
        L.uly_plan_test_withhold_fill.argtypes = [vp, i32]
        L.uly_plan_rows.argtypes = [vp, ctypes.c_int]
        L.uly_plan_rows.restype = i64
        L.uly_pick_head_groups.argtypes = [i32, i32, i64, i64, i32]
        L.uly_to_heads.argtypes = [vp, vpp, vpp, vpp, vpp, vpp, vpp, vp]
        attn = [vp, vpp, vpp, vpp, vp, vp, i32, ctypes.c_float, i32, vp, vp, vp, vpp, vpp, vp]
        L.uly_attention.argtypes = attn
        L.uly_attention_merge.argtypes = attn
        L.uly_sp_attention.argtypes = attn
        L.uly_ring_attention.argtypes = [vp, vpp, vpp, vpp, vp, vp, i32, ctypes.POINTER(i32), ctypes.c_float, i32,
                                         vp, vp, vp, vpp, vpp, vp]
        L.uly_to_seq.argtypes = [vp, vpp, vpp, vp]
        L.uly_sync_status.argtypes = [vp, vp]
        L.uly_status_string.argtypes = [ctypes.c_int]
        L.uly_status_string.restype = ctypes.c_char_p
        L.uly_sp_attention_noalloc.argtypes = [ctypes.POINTER(_Desc)] + attn[1:]
        L.uly_noalloc_sync_status.argtypes = [vp]
        L.uly_lse_merge.argtypes = [i64, i32, vp, vp, vp, vp, vp, vp, vp]
        L.uly_pipelined_attention.argtypes = [vp, vpp, vpp, vpp, vpp, vpp, vpp, vpp, vp, vp, i32, ctypes.c_float,
                                              i32, vp, vp, vp, vpp, vp, vp]
        L.uly_sp_attention_host.argtypes = [vp, vpp, vpp, vpp, vpp, vpp, vpp, vp, vp, i32, ctypes.c_float, i32,
                                            vp, vp, vp, vpp, vpp, vp]
        L.uly_device_sm_count.argtypes = [ctypes.c_int]
        L.uly_device_sm_count.restype = i32
        L.uly_checked_violations.argtypes = [i32]
        L.uly_checked_violations.restype = i64
        L.uly_plan_test_check_narrow.argtypes = [vp, i32]
        _lib = L
    return _lib


def _status_string(st: int) -> str:
    try:
        return lib().uly_status_string(st).decode()
    except Exception:  # noqa: BLE001 - only used for messages
        return "status"


def _check(st: int, what: str):
    if st != ULY_OK:
        raise UlyError(st, what)


# ---- argument checks: the C ABI sees only pointers, so shapes, element
# types, devices and contiguity are checked here against the plan before a
# call (a short pointer list or a small tensor would otherwise be read or
# written past its end on the GPU).
_ELEM = {"bf16": ("torch.bfloat16",), "e4m3": ("torch.uint8", "torch.float8_e4m3fn")}


def _want(t, shape, dtypes, what, device):
    import torch
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda" or t.device.index != device:
        raise ValueError("%s: expected a CUDA tensor on device %d" % (what, device))
    if str(t.dtype) not in dtypes:
        raise ValueError("%s: element type %s, expected one of %s" % (what, t.dtype, ", ".join(dtypes)))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s: shape %s, expected %s" % (what, tuple(t.shape), tuple(shape)))
    if not t.is_contiguous():
        raise ValueError("%s: must be contiguous" % what)


def _want_list(ts, shapes, dtypes, what, device):
    if ts is None or len(ts) != len(shapes):
        raise ValueError("%s: expected %d tensors, got %s" % (what, len(shapes), None if ts is None else len(ts)))
    for i, (t, shp) in enumerate(zip(ts, shapes)):
        _want(t, shp, dtypes, "%s[%d]" % (what, i), device)


def _want_mask(key_mask, key_ranges, B, Nk, device):
    if key_mask is not None:
        _want(key_mask, (B, Nk), ("torch.uint8", "torch.bool"), "key_mask", device)
    if key_ranges is not None:
        if key_ranges.dim() != 3 or key_ranges.shape[0] != B or key_ranges.shape[2] != 2 or key_ranges.shape[1] < 1:
            raise ValueError("key_ranges: shape %s, expected (%d, n >= 1, 2)" % (tuple(key_ranges.shape), B))
        _want(key_ranges, tuple(key_ranges.shape), ("torch.int32",), "key_ranges", device)


def _want_scales(dtype, q_scale, k_scale, v_scale, Hq, Hkv, device):
    # only an e4m3 shape uses scales; a bf16 call that passes some is left
    # to the C ABI, which rejects it with ULY_ERR_INVALID
    if dtype != "e4m3":
        return
    for t, n, what in ((q_scale, Hq, "q_scale"), (k_scale, Hkv, "k_scale"), (v_scale, Hkv, "v_scale")):
        if t is None:
            raise ValueError("%s: e4m3 inputs need per-head scales" % what)
        _want(t, (n,), ("torch.float32",), what, device)


def _ptr(t) -> int | None:
    if t is None:
        return None
    return t.data_ptr()


def _ptr_array(ts):
    if ts is None:
        return None
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def pick_head_groups(hq_local: int, hkv_local: int, q_rows: int, batch_ranks: int, sm_count: int) -> int:
    """Automatic head-group count (see uly_pick_head_groups in include/uly.h)."""
    return int(lib().uly_pick_head_groups(hq_local, hkv_local, q_rows, batch_ranks, sm_count))


def sp_attention_noalloc(B, P, S_l, R, rep_mode, Hq, Hkv, D, q, k, v, o, dtype="bf16", masked_rows="sdpa",
                         key_mask=None, key_ranges=None, scale=None, head_groups=0, q_scale=None, k_scale=None,
                         v_scale=None, lse=None, stream=None):
    """Fused attention without a plan and without any device allocation
    (uly_sp_attention_noalloc): for callers whose device memory belongs to
    their own pool and who therefore cannot let the library cudaMalloc.  Its
    scratch is a fixed array inside the library shared by every call, so
    calls must not overlap on the GPU."""
    d = _Desc(B, P, S_l, R, REP_MODES[rep_mode], Hq, Hkv, D, DTYPES[dtype], MASKED_ROWS[masked_rows])
    import torch
    dev = torch.cuda.current_device()
    rq = S_l + (R if rep_mode in ("prefix", "suffix") else 0)
    rk = S_l + (R if rep_mode != "none" else 0)
    el = _ELEM[dtype]
    _want_list(q, [(B, rq, Hq, D)] * P, el, "q", dev)
    _want_list(k, [(B, rk, Hkv, D)] * P, el, "k", dev)
    _want_list(v, [(B, rk, Hkv, D)] * P, el, "v", dev)
    _want_list(o, [(B, rq, Hq, D)] * P, ("torch.bfloat16",), "o", dev)
    if lse is not None:
        _want_list(lse, [(B, rq, Hq)] * P, ("torch.float32",), "lse", dev)
    _want_mask(key_mask, key_ranges, B, P * S_l + (R if rep_mode != "none" else 0), dev)
    _want_scales(dtype, q_scale, k_scale, v_scale, Hq, Hkv, dev)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    n_ranges = 0 if key_ranges is None else int(key_ranges.shape[1])
    _check(lib().uly_sp_attention_noalloc(ctypes.byref(d), _ptr_array(q), _ptr_array(k), _ptr_array(v),
                                          _ptr(key_mask), _ptr(key_ranges), n_ranges, ctypes.c_float(scale),
                                          int(head_groups), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
                                          _ptr_array(o), _ptr_array(lse), _stream(stream)),
           "uly_sp_attention_noalloc")


def noalloc_sync_status(stream=None) -> int:
    """Synchronize the stream, then read and clear the status word of the
    allocation-free call (uly_noalloc_sync_status): 0, or ULY_ERR_TIMEOUT
    when one of its device waits expired."""
    return int(lib().uly_noalloc_sync_status(_stream(stream)))


def lse_merge(o_a, lse_a, o_b, lse_b, o_out=None, lse_out=None, stream=None):
    """Ring-attention merge (uly_lse_merge) of two bf16 [..., D] results and
    their f32 [...] log-sum-exps; in place into (o_a, lse_a) by default."""
    if o_out is None:
        o_out, lse_out = o_a, lse_a
    dev = o_a.device.index if o_a.device.type == "cuda" else -1
    for t, what in ((o_a, "o_a"), (o_b, "o_b"), (o_out, "o_out")):
        _want(t, tuple(o_a.shape), ("torch.bfloat16",), what, dev)
    for t, what in ((lse_a, "lse_a"), (lse_b, "lse_b"), (lse_out, "lse_out")):
        _want(t, tuple(o_a.shape[:-1]), ("torch.float32",), what, dev)
    D = o_a.shape[-1]
    rows = o_a.numel() // D
    _check(lib().uly_lse_merge(rows, D, _ptr(o_a), _ptr(lse_a), _ptr(o_b), _ptr(lse_b), _ptr(o_out), _ptr(lse_out),
                               _stream(stream)), "uly_lse_merge")
    return o_out, lse_out


def checked_violations(reset: bool = False) -> int:
    """Index-check violations counted on the current device since the last
    reset (uly_checked_violations); -1 when the library is the normal build."""
    return int(lib().uly_checked_violations(1 if reset else 0))


def device_sm_count(device: int = 0) -> int:
    return int(lib().uly_device_sm_count(device))


class Plan:
    """One Ulysses attention shape (include/uly.h, uly_plan_create)."""

    def __init__(self, B: int, P: int, S_l: int, R: int, rep_mode: str, Hq: int, Hkv: int, D: int,
                 dtype: str = "bf16", masked_rows: str = "sdpa", device: int | None = None,
                 shard_lens=None):
        import torch
        if device is None:
            device = torch.cuda.current_device()
        self.device = device
        self.desc = dict(B=B, P=P, S_l=S_l, R=R, rep_mode=rep_mode, Hq=Hq, Hkv=Hkv, D=D, dtype=dtype,
                         masked_rows=masked_rows)
        d = _Desc(B, P, S_l, R, REP_MODES[rep_mode], Hq, Hkv, D, DTYPES[dtype], MASKED_ROWS[masked_rows])
        h = ctypes.c_void_p()
        if shard_lens is None:
            _check(lib().uly_plan_create(ctypes.byref(d), device, ctypes.byref(h)), "uly_plan_create")
        else:
            lens = (ctypes.c_int32 * P)(*shard_lens)
            _check(lib().uly_plan_create_varlen(ctypes.byref(d), lens, device, ctypes.byref(h)),
                   "uly_plan_create_varlen")
        self.shard_lens = None if shard_lens is None else tuple(shard_lens)
        self._h = h
        self.P, self.B, self.Hq, self.Hkv, self.D = P, B, Hq, Hkv, D
        self.dtype = dtype

    def close(self):
        if getattr(self, "_h", None):
            lib().uly_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # noqa: BLE001 - interpreter shutdown
            pass

    # ---- sizes
    def rows(self, which: int) -> int:
        return int(lib().uly_plan_rows(self._h, which))

    def shard_rows(self, shard: int, is_kv: bool = False) -> int:
        return int(lib().uly_plan_shard_rows(self._h, shard, int(is_kv)))

    @property
    def shard_rows_q(self):
        return self.rows(0)

    @property
    def shard_rows_kv(self):
        return self.rows(1)

    @property
    def heads_rows_q(self):
        return self.rows(2)

    @property
    def heads_rows_kv(self):
        return self.rows(3)

    def set_wait_limit(self, ns: int):
        _check(lib().uly_plan_set_wait_limit(self._h, int(ns)), "uly_plan_set_wait_limit")

    def test_withhold_fill(self, fill: int):
        _check(lib().uly_plan_test_withhold_fill(self._h, int(fill)), "uly_plan_test_withhold_fill")

    def test_check_narrow(self, rows: int):
        _check(lib().uly_plan_test_check_narrow(self._h, int(rows)), "uly_plan_test_check_narrow")

    # ---- argument checks against the plan's shape
    def _check_seq(self, q=None, k=None, v=None, o=None, lse=None):
        B, D, dev, P = self.B, self.D, self.device, self.P
        el = _ELEM[self.dtype]
        if q is not None:
            _want_list(q, [(B, self.shard_rows(p), self.Hq, D) for p in range(P)], el, "q", dev)
        for t, what in ((k, "k"), (v, "v")):
            if t is not None:
                _want_list(t, [(B, self.shard_rows(p, True), self.Hkv, D) for p in range(P)], el, what, dev)
        if o is not None:
            _want_list(o, [(B, self.shard_rows(p), self.Hq, D) for p in range(P)], ("torch.bfloat16",), "o", dev)
        if lse is not None:
            _want_list(lse, [(B, self.shard_rows(p), self.Hq) for p in range(P)], ("torch.float32",), "lse", dev)

    def _check_heads(self, qh=None, kh=None, vh=None, oh=None, lse=None):
        B, D, dev, P = self.B, self.D, self.device, self.P
        el = _ELEM[self.dtype]
        hq, hkv = self.Hq // P, self.Hkv // P
        if qh is not None:
            _want_list(qh, [(B, self.heads_rows_q, hq, D)] * P, el, "qh", dev)
        for t, what in ((kh, "kh"), (vh, "vh")):
            if t is not None:
                _want_list(t, [(B, self.heads_rows_kv, hkv, D)] * P, el, what, dev)
        if oh is not None:
            _want_list(oh, [(B, self.heads_rows_q, hq, D)] * P, ("torch.bfloat16",), "oh", dev)
        if lse is not None:
            _want_list(lse, [(B, self.heads_rows_q, hq)] * P, ("torch.float32",), "lse", dev)

    def _check_call(self, key_mask, key_ranges, q_scale, k_scale, v_scale):
        _want_mask(key_mask, key_ranges, self.B, self.heads_rows_kv, self.device)
        _want_scales(self.dtype, q_scale, k_scale, v_scale, self.Hq, self.Hkv, self.device)

    # ---- the path
    def to_heads(self, q, k, v, qh, kh, vh, stream=None):
        self._check_seq(q, k, v)
        self._check_heads(qh, kh, vh)
        _check(lib().uly_to_heads(self._h, _ptr_array(q), _ptr_array(k), _ptr_array(v),
                                  _ptr_array(qh), _ptr_array(kh), _ptr_array(vh), _stream(stream)),
               "uly_to_heads")

    def to_seq(self, oh, o, stream=None):
        self._check_heads(oh=oh)
        self._check_seq(o=o)
        _check(lib().uly_to_seq(self._h, _ptr_array(oh), _ptr_array(o), _stream(stream)), "uly_to_seq")

    def _attn(self, fn, name, q, k, v, o, key_mask, key_ranges, scale, head_groups, q_scale, k_scale, v_scale,
              lse, stream, fused):
        if fused:
            self._check_seq(q, k, v, o, lse)
        else:
            self._check_heads(q, k, v, o, lse)
        self._check_call(key_mask, key_ranges, q_scale, k_scale, v_scale)
        if scale is None:
            scale = 1.0 / math.sqrt(self.D)
        n_ranges = 0
        if key_ranges is not None:
            n_ranges = int(key_ranges.shape[1])
        _check(fn(self._h, _ptr_array(q), _ptr_array(k), _ptr_array(v), _ptr(key_mask), _ptr(key_ranges),
                  n_ranges, ctypes.c_float(scale), int(head_groups), _ptr(q_scale), _ptr(k_scale), _ptr(v_scale),
                  _ptr_array(o), _ptr_array(lse), _stream(stream)), name)

    def attention(self, qh, kh, vh, oh, key_mask=None, key_ranges=None, scale=None, head_groups=0,
                  q_scale=None, k_scale=None, v_scale=None, lse=None, stream=None):
        self._attn(lib().uly_attention, "uly_attention", qh, kh, vh, oh, key_mask, key_ranges, scale, head_groups,
                   q_scale, k_scale, v_scale, lse, stream, fused=False)

    def attention_merge(self, qh, kh, vh, oh, lse, key_mask=None, key_ranges=None, scale=None, head_groups=0,
                        q_scale=None, k_scale=None, v_scale=None, stream=None):
        """One ring step (uly_attention_merge): attention over the admitted
        keys merged into the running (oh, lse), both read and written."""
        if lse is None:
            raise ValueError("attention_merge needs the running lse tensors")
        self._attn(lib().uly_attention_merge, "uly_attention_merge", qh, kh, vh, oh, key_mask, key_ranges, scale,
                   head_groups, q_scale, k_scale, v_scale, lse, stream, fused=False)

    def ring_attention(self, qh, kh, vh, oh, chunk_bounds, key_mask=None, key_ranges=None, scale=None,
                       head_groups=0, q_scale=None, k_scale=None, v_scale=None, lse=None, stream=None):
        """Ring attention over P virtual ring ranks in one launch
        (uly_ring_attention): rank r's key chunk is [chunk_bounds[r],
        chunk_bounds[r + 1]) of the global key order (P + 1 ints, 0 to
        heads_rows_kv); each rank's queries take the chunks from its own on."""
        self._check_heads(qh, kh, vh, oh, lse)
        self._check_call(key_mask, key_ranges, q_scale, k_scale, v_scale)
        if scale is None:
            scale = 1.0 / math.sqrt(self.D)
        bounds = [int(x) for x in chunk_bounds]
        if len(bounds) != self.P + 1:
            raise ValueError("chunk_bounds needs P + 1 = %d entries" % (self.P + 1))
        cb = (ctypes.c_int32 * len(bounds))(*bounds)
        n_ranges = 0 if key_ranges is None else int(key_ranges.shape[1])
        _check(lib().uly_ring_attention(self._h, _ptr_array(qh), _ptr_array(kh), _ptr_array(vh), _ptr(key_mask),
                                        _ptr(key_ranges), n_ranges, cb, ctypes.c_float(scale), int(head_groups),
                                        _ptr(q_scale), _ptr(k_scale), _ptr(v_scale), _ptr_array(oh),
                                        _ptr_array(lse), _stream(stream)), "uly_ring_attention")

    def sp_attention(self, q, k, v, o, key_mask=None, key_ranges=None, scale=None, head_groups=0,
                     q_scale=None, k_scale=None, v_scale=None, lse=None, stream=None):
        self._attn(lib().uly_sp_attention, "uly_sp_attention", q, k, v, o, key_mask, key_ranges, scale,
                   head_groups, q_scale, k_scale, v_scale, lse, stream, fused=True)

    def pipelined_attention(self, q, k, v, qh, kh, vh, oh, o, key_mask=None, key_ranges=None, scale=None,
                            head_groups=0, q_scale=None, k_scale=None, v_scale=None, stream=None,
                            copy_stream=None):
        """Staged path with the exchange pipelined against the attention
        (uly_pipelined_attention): per-chunk gather kernels on copy_stream;
        qh/kh/vh/oh are the staging buffers."""
        import torch
        self._check_seq(q, k, v, o)
        self._check_heads(qh, kh, vh, oh)
        self._check_call(key_mask, key_ranges, q_scale, k_scale, v_scale)
        if scale is None:
            scale = 1.0 / math.sqrt(self.D)
        if stream is None:
            stream = torch.cuda.current_stream()
        if copy_stream is None:
            copy_stream = self._copy_stream()
        n_ranges = 0 if key_ranges is None else int(key_ranges.shape[1])
        _check(lib().uly_pipelined_attention(self._h, _ptr_array(q), _ptr_array(k), _ptr_array(v), _ptr_array(qh),
                                             _ptr_array(kh), _ptr_array(vh), _ptr_array(oh), _ptr(key_mask),
                                             _ptr(key_ranges), n_ranges, ctypes.c_float(scale), int(head_groups),
                                             _ptr(q_scale), _ptr(k_scale), _ptr(v_scale), _ptr_array(o),
                                             _stream(stream), _stream(copy_stream)), "uly_pipelined_attention")

    def sp_attention_host(self, q_host, k_host, v_host, q, k, v, o, o_host, key_mask=None, key_ranges=None,
                          scale=None, head_groups=0, q_scale=None, k_scale=None, v_scale=None, stream=None):
        """Fused call with the shards in (page-locked) host memory
        (uly_sp_attention_host): q_host/k_host/v_host are copied into the
        device shard tensors q/k/v, the output goes to o and then o_host,
        copies overlapped with the attention of other ranks' heads."""
        if scale is None:
            scale = 1.0 / math.sqrt(self.D)
        self._check_seq(q, k, v, o)
        self._check_call(key_mask, key_ranges, q_scale, k_scale, v_scale)
        for hs, ds in ((q_host, q), (k_host, k), (v_host, v), (o_host, o)):
            if len(hs) != self.P or len(ds) != self.P:
                raise ValueError("expected %d shard tensors" % self.P)
            for h, d in zip(hs, ds):
                if h.device.type != "cpu" or h.shape != d.shape or h.dtype != d.dtype or not h.is_contiguous():
                    raise ValueError("host tensors must be contiguous CPU tensors shaped like the device ones")
        n_ranges = 0 if key_ranges is None else int(key_ranges.shape[1])
        _check(lib().uly_sp_attention_host(self._h, _ptr_array(q_host), _ptr_array(k_host), _ptr_array(v_host),
                                           _ptr_array(q), _ptr_array(k), _ptr_array(v), _ptr(key_mask),
                                           _ptr(key_ranges), n_ranges, ctypes.c_float(scale), int(head_groups),
                                           _ptr(q_scale), _ptr(k_scale), _ptr(v_scale), _ptr_array(o),
                                           _ptr_array(o_host), _stream(stream)), "uly_sp_attention_host")

    def _copy_stream(self):
        import torch
        if getattr(self, "_cs", None) is None:
            self._cs = torch.cuda.Stream()
        return self._cs

    def sync_status(self, stream=None) -> int:
        return int(lib().uly_sync_status(self._h, _stream(stream)))
