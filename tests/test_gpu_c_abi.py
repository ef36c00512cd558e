"""The C ABI driven by a plain C program (tests/c_abi/uly_c_example.c, no
Python or PyTorch in the call path): built with the system C compiler
against include/uly.h and the in-tree library, run on seeded shards, its
output bit-identical to the binding's fused call and within tolerance of the
oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import synth
from tests import _helpers as H

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "uly_c_example.c")

CASES = [
    synth.WORKLOADS["tiny"],
    synth.Workload("c-prefix-masked", B=2, P=4, S_l=300, R=200, mode="prefix", Hq=8, Hkv=4, D=128, dtype="bf16",
                   std_q=1.0, std_kv=1.0, seed=91, valid=((0, 77), (200, 1400))),
    synth.Workload("c-suffix-d64", B=1, P=3, S_l=129, R=40, mode="suffix", Hq=6, Hkv=6, D=64, dtype="bf16",
                   std_q=1.0, std_kv=1.0, seed=92),
]


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    import ulysses_sequence_attention_uly_gb300 as uly
    libdir = os.path.dirname(uly.build(checked_build=False))
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path_factory.mktemp("c_abi") / "uly_c_example")
    rpath = "-Wl,-rpath," + libdir + ":" + os.path.join(cuda, "lib64")
    subprocess.run([cc, "-std=c11", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda, "include"), SRC, "-o", exe, "-L", libdir, "-luly",
                    "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm", rpath], check=True)
    return exe


def _bf16_to_f64(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_c_program_matches_binding_and_oracle(program, w, tmp_path):
    data = synth.generate(w)
    for p in range(w.P):
        for n in ("q", "k", "v"):
            np.ascontiguousarray(data[n][p]).tofile(str(tmp_path / ("%s%d.bin" % (n, p))))
    ranges = data["key_ranges"]
    n_ranges = 0 if ranges is None else int(ranges.shape[1])
    if ranges is not None:
        np.ascontiguousarray(ranges, dtype=np.int32).tofile(str(tmp_path / "ranges.bin"))
    args = [program, str(tmp_path), str(w.B), str(w.P), str(w.S_l), str(w.R), str(w.rep_mode), str(w.Hq),
            str(w.Hkv), str(w.D), str(n_ranges)]
    r = subprocess.run(args, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr

    plan = H.make_plan(w)
    d = H.dev_inputs(w, data)
    via_binding = H.run_fused(plan, w, d, mask="ranges" if ranges is not None else "none")
    _, want = H.oracle_path(w, data)
    for p in range(w.P):
        got = np.fromfile(str(tmp_path / ("o%d.bin" % p)), dtype=np.uint16)
        assert got.size == via_binding[p].numel()
        assert np.array_equal(got.view(np.int16), H.bits(via_binding[p]).reshape(-1)), p
        ok, err, nbad = H.within(_bf16_to_f64(got).reshape(want[p].shape), want[p], H.TOL["bf16"])
        assert ok, "shard %d: max err %g (%d)" % (p, err, nbad)
