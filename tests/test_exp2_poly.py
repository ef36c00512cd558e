"""The software 2^x of the e4m3 softmax (tc.cuh exp2_poly_f2): its
constants are the minimax cubic that csrc/exp2_poly.py derives, and the
float32 evaluation the kernel performs stays within the bound the P operand
needs (relative error far below e4m3's and bf16's own rounding)."""
import os
import re
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "ulysses_sequence_attention_uly_gb300", "csrc")
sys.path.insert(0, CSRC)
import exp2_poly  # noqa: E402


def _kernel_constants():
    src = open(os.path.join(CSRC, "tc.cuh")).read()
    body = src[src.index("exp2_poly_f2(uint64_t x)"):]
    body = body[:body.index("\n}\n")]
    vals = [float(v) for v in re.findall(r"f2\(([0-9.e+-]+)f, \1f\)", body)]
    vals = [v for v in vals if 0.0 < v < 1.0]  # drop the shifter and the -1 of the reduction
    # c3 first, then c2, c1, c0 in the Horner chain
    return vals


def test_constants_match_derivation():
    c, err = exp2_poly.coefficients_f32()
    got = [np.float32(v) for v in _kernel_constants()]  # the kernel's literals, as float32
    assert got == [np.float32(c[3]), np.float32(c[2]), np.float32(c[1]), np.float32(c[0])]
    assert err < 1e-4


def test_float32_evaluation_error():
    c, _ = exp2_poly.coefficients_f32()
    x = np.linspace(-120, 8, 400001).astype(np.float32)
    y = (x + np.float32(12582912.0)).astype(np.float32)          # shifter
    n = (y - np.float32(12582912.0)).astype(np.float32)          # rint(x)
    f = (x - n).astype(np.float32)
    assert np.all(np.abs(f) <= 0.5)
    p = np.float32(c[3])
    for k in (2, 1, 0):  # fma: one rounding per step
        p = (p.astype(np.float64) * f + np.float64(np.float32(c[k]))).astype(np.float32)
    r = np.ldexp(p.astype(np.float64), n.astype(np.int64))
    rel = np.abs(r / np.exp2(x.astype(np.float64)) - 1.0)
    assert rel.max() < 1.2e-4
    # the exponent add of the kernel: bits(p) + (bits(y) << 23) == p * 2^n
    bits_y = y.view(np.uint32).astype(np.uint64)
    bits_p = p.view(np.uint32).astype(np.uint64)
    out = ((bits_p + (bits_y << np.uint64(23))) & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.float32)
    np.testing.assert_array_equal(out.astype(np.float64), r)
