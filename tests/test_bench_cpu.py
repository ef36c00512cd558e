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
