"""The checked build (library compiled with -DULY_CHECKED=1): every index the
kernels compute into a global tensor is checked against its extent.  The
whole GPU suite runs against it in a child process and must see no
violation and the same results as with the normal build; and a narrowed row
check, through a test
hook that leaves every access inside the real tensors, is counted and its
runs are left unwritten."""
import os
import re
import subprocess
import sys

import pytest

import synth
from tests import _helpers as H

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
# every GPU test but this file
SUITES = ["tests", "--ignore=tests/test_gpu_checked.py"]


def test_gpu_suites_under_the_checked_build():
    if os.environ.get("ULY_CHECKED", "") == "1":
        pytest.skip("already running under the checked build")
    env = dict(os.environ, ULY_CHECKED="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider"] + SUITES,
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1500)
    assert r.returncode == 0, r.stdout[-4000:] + r.stderr[-2000:]
    m = re.search(r"(\d+) passed", r.stdout)
    assert m and int(m.group(1)) >= 100, r.stdout[-2000:]  # the whole suite ran, not a stray subset
    print(r.stdout.strip().splitlines()[-1])


_W = synth.Workload("checked-prefix", B=2, P=4, S_l=300, R=200, mode="prefix", Hq=8, Hkv=4, D=128, dtype="bf16",
                    std_q=1.0, std_kv=1.0, seed=101, valid=((0, 77), (200, 1400)))


def test_narrowed_row_check_is_counted():
    """Prefix mode: narrowing the row check by one row refuses the last image
    row of every shard (replicated rows come from rows < R): one run per
    (tensor, batch, rank, shard), counted once by the lane that would have
    copied it and left holding the fill value; without the hook the same
    call is clean and bit exact."""
    code = r'''
import sys, numpy as np, torch
sys.path.insert(0, %r)
import synth
from tests import _helpers as H
import ulysses_sequence_attention_uly_gb300 as uly
w = synth.Workload(%r, B=%d, P=%d, S_l=%d, R=%d, mode=%r, Hq=%d, Hkv=%d, D=%d, dtype="bf16",
                   std_q=1.0, std_kv=1.0, seed=%d, valid=%r)
data = synth.generate(w)
plan = H.make_plan(w)
d = H.dev_inputs(w, data)
assert uly.checked()
assert uly.checked_violations(reset=True) == 0
qh, kh, vh = H.empty_heads(plan, w, torch.bfloat16)
for t in qh + kh + vh:
    t.fill_(7.0)
plan.test_check_narrow(1)
plan.to_heads(d["q"], d["k"], d["v"], qh, kh, vh)
n = uly.checked_violations(reset=True)
plan.test_check_narrow(0)
runs = 3 * w.B * w.P * w.P
assert n == runs, (n, runs)
want = H.oracle_heads(w, data)
bad = 0
for got_list, want_list in zip((qh, kh, vh), want):
    for g, wnt in zip(got_list, want_list):
        gb = H.bits(g).view(np.uint16)
        diff = ~(gb == wnt).all(axis=(-1, -2))
        bad += int(diff.sum())
        assert (gb[diff] == 0x40E0).all()  # bf16 7.0: the refused rows were not written
assert bad == runs, (bad, runs)
plan.to_heads(d["q"], d["k"], d["v"], qh, kh, vh)
assert uly.checked_violations(reset=True) == 0
for got_list, want_list in zip((qh, kh, vh), want):
    for g, wnt in zip(got_list, want_list):
        np.testing.assert_array_equal(H.bits(g).view(np.uint16), wnt)
print("ok", n)
''' % (ROOT, _W.name, _W.B, _W.P, _W.S_l, _W.R, _W.mode, _W.Hq, _W.Hkv, _W.D, _W.seed, _W.valid)
    env = dict(os.environ, ULY_CHECKED="1")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]


def test_normal_build_reports_no_checks():
    import ulysses_sequence_attention_uly_gb300 as uly
    if uly.checked():
        pytest.skip("running under the checked build")
    assert uly.checked_violations() == -1
    plan = H.make_plan(_W)
    with pytest.raises(uly.UlyError) as e:
        plan.test_check_narrow(1)
    assert e.value.status == uly.ULY_ERR_UNSUPPORTED
