"""Host logic of the decode's work split: the cost-weighted cut that the
split kernel and the merge kernel both compute (each (sequence, KV head)
piece counts a fixed extra cost, and the warps' ranges are equal in cost)
must partition the units in order, name the range of every unit, and give
every cut (sequence, KV head) consecutive, non-empty ranges -- the merge
counts its pieces as the number of ranges it spans.  The cut is
__host__ __device__ code, compiled here for the host with nvcc and checked on
random length mixes with empty sequences (no GPU needed)."""

import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_work_cut_partitions_the_units(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "work_cut_check")
    r = subprocess.run([nvcc, "-std=c++20", "-O1", "-I", os.path.join(ROOT, "include"),
                        "-I", os.path.join(ROOT, "paged_kv_cache_68_gb300", "csrc"),
                        os.path.join(HERE, "work_cut_check.cu"), "-o", exe],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr[-2000:]
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout + r.stderr
