"""The grouped FFN's tile order (grouped_ffn_gb300/csrc/tile_order.cuh): the
proportional hot/cold merge is a bijection that keeps each stream's order
and the hot:cold mix at every position, and the incremental walk each CTA
uses visits the same tiles.  Checked by a host program built with nvcc from
the same header the kernel uses.  CPU only."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_tile_order_is_a_bijection_and_the_walk_matches(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not available")
    exe = tmp_path / "tile_order_check"
    subprocess.run([nvcc, "-O2", "-std=c++17", "-I", os.path.join(ROOT, "grouped_ffn_gb300", "csrc"),
                    "-o", str(exe), os.path.join(ROOT, "tests", "tile_order_check.cu")],
                   check=True, capture_output=True, timeout=300)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "tile order ok" in r.stdout
