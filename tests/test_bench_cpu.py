"""bench.py's host-side pieces that need no GPU: the digest that keys the
recorded ncu traffic to the kernel's code."""
import os
import shutil

import bench

CSRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                    "ulysses_sequence_attention_uly_gb300", "csrc")


def _copy(tmp_path):
    d = tmp_path / "csrc"
    d.mkdir()
    for name in bench.KERNEL_SOURCES:
        shutil.copy(os.path.join(CSRC, name), d / name)
    return d


def test_digest_ignores_comments_and_whitespace(tmp_path):
    d = _copy(tmp_path)
    base = bench.kernel_code_digest(str(d))
    assert base == bench.kernel_code_digest()
    src = (d / "attn.cu").read_text()
    (d / "attn.cu").write_text("// a new comment\n" + src.replace("\n", "\n  ", 3) + "\n/* and another */\n")
    assert bench.kernel_code_digest(str(d)) == base


def test_digest_follows_code(tmp_path):
    d = _copy(tmp_path)
    base = bench.kernel_code_digest(str(d))
    src = (d / "tc.cuh").read_text()
    (d / "tc.cuh").write_text(src.replace("ex2.approx.ftz.f32", "ex2.approx.f32", 1))
    assert bench.kernel_code_digest(str(d)) != base


def test_p90_nearest_rank():
    import bench
    assert bench.p90([5.0]) == 5.0
    assert bench.p90(list(range(1, 11))) == 9
    assert bench.p90(list(range(20, 0, -1))) == 18  # order of the samples does not matter


def test_reference_arm_reports_measured_step_time():
    """The reference arm's ms_per_step is the wall time of one sampled step
    (so K steps fit in the run's wall time); the full workload's
    extrapolated time is reported apart, and the config names the same
    workload string as the GPU arm (head groups included)."""
    import time

    import synth
    args = type("A", (), {"workload": "tiny", "steps": 1, "warmup": 0})()
    t0 = time.perf_counter()
    out = bench.run_reference(args, 0, 1)
    wall_ms = 1e3 * (time.perf_counter() - t0)
    assert out["impl"] == "reference"
    assert 0 < out["ms_per_step"] <= wall_ms
    assert out["extrapolated_full_step_ms"] > 0
    assert out["config"]["workload"] == bench.workload_string(synth.WORKLOADS["tiny"])
    assert "head_groups=" in out["config"]["workload"]
