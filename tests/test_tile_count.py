"""Host logic of the ring kernels' work decomposition (no GPU): the
closed-form tile count over the whole ring, the per-step counts and the walk
itself agree, and both unit numberings cover every query tile exactly once."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_ring_tile_count_closed_form(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    exe = str(tmp_path / "tile_count_check")
    subprocess.run([cxx, "-std=c++17", "-O2", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "context_parallelism_02_gb300", "csrc"),
                    os.path.join(HERE, "tile_count_check.cpp"), "-o", exe], check=True)
    res = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "0 mismatches" in res.stdout
