"""bench.py's roofline traffic comes from a committed ncu summary and must be dropped (reported as
null) as soon as the measured kernel's source changes. These CPU tests check the fingerprint that
decides it: it follows the per-element arithmetic, the work-division section of the common header
and the double-buffered kernel's own text, and ignores edits elsewhere in those files."""
import os
import shutil

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join("fsdp_sharded_mixed_ss_gb300", "csrc")


def _record():
    ent = {}
    with open(os.path.join(ROOT, "profiles", "adam_traffic.txt")) as f:
        for line in f:
            if "=" in line and not line.lstrip().startswith("#"):
                k, v = line.split("=", 1)
                ent[k.strip()] = v.strip()
    return ent


ELEMS = int(_record()["elements"])


@pytest.fixture()
def tree(tmp_path, monkeypatch):
    """A copy of the sources and the traffic record, with bench.py pointed at it."""
    shutil.copytree(os.path.join(ROOT, CSRC), tmp_path / CSRC)
    shutil.copytree(os.path.join(ROOT, "profiles"), tmp_path / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def _edit(path, old, new):
    text = path.read_text()
    assert old in text, old
    path.write_text(text.replace(old, new, 1))


def test_committed_record_matches_the_committed_kernel():
    rec = bench.profile_traffic("adam_pipe_kernel", ELEMS)
    assert rec is not None and rec > 0
    assert bench.profile_traffic("some_other_kernel", ELEMS) is None
    assert bench.profile_traffic("adam_pipe_kernel", ELEMS + 8) is None     # a record for another shard length


def test_edits_to_the_measured_kernel_drop_the_record(tree):
    base = bench.kernel_fingerprint()
    assert bench.profile_traffic("adam_pipe_kernel", ELEMS) is not None
    # the double-buffered kernel's text
    _edit(tree / CSRC / "ss_step.cu", "constexpr bool kPrefetch = F || NR <= kPipePrefetchRanks;",
          "constexpr bool kPrefetch = F || NR <= kPipePrefetchRanks + 1;")
    assert bench.kernel_fingerprint() != base
    assert bench.profile_traffic("adam_pipe_kernel", ELEMS) is None


def test_edits_to_the_work_division_drop_the_record(tree):
    base = bench.kernel_fingerprint()
    _edit(tree / CSRC / "ss_common.cuh", "return static_cast<int64_t>(j) * gridDim.x + blockIdx.x;",
          "return static_cast<int64_t>(j) * gridDim.x + (gridDim.x - 1 - blockIdx.x);")
    assert bench.kernel_fingerprint() != base
    assert bench.profile_traffic("adam_pipe_kernel", ELEMS) is None


def test_edits_to_the_arithmetic_drop_the_record(tree):
    base = bench.kernel_fingerprint()
    _edit(tree / CSRC / "ss_math.cuh", "float e = fmaf(a, b, -p);", "float e = fmaf(a, b, -p) * 1.0f;")
    assert bench.kernel_fingerprint() != base


def test_edits_elsewhere_keep_the_record(tree):
    base = bench.kernel_fingerprint()
    # another kernel in the same file, and a part of the common header outside the work division
    _edit(tree / CSRC / "ss_step.cu", "adam_scalar_kernel(const __grid_constant__ StepArgs<MAXR> a) {",
          "adam_scalar_kernel(const __grid_constant__ StepArgs<MAXR> a) {  // edited")
    _edit(tree / CSRC / "ss_common.cuh", "constexpr int kThreads = 256;", "constexpr int kThreads = 256;  // edited")
    assert bench.kernel_fingerprint() == base
    assert bench.profile_traffic("adam_pipe_kernel", ELEMS) is not None
