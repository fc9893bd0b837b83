"""The attention kernel's tile ranges (TileDeal in csrc/common.cuh) checked on
the host: tests/tile_deal_check.cu, compiled with nvcc as host code, walks
every deal the planner can make for up to 70 queries, 40 tiles a query and
160 CTAs (balanced, balanced with a per-query start cost, query-aligned), and
deals near 2^31 units at their range ends."""
import os
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


@pytest.mark.skipif(not (os.path.exists(NVCC) or shutil.which("nvcc")), reason="nvcc not found")
def test_tile_deal_ranges_and_owners_agree():
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "tile_deal_check")
        subprocess.run([NVCC, "-std=c++17", "-x", "cu", os.path.join(ROOT, "tests", "tile_deal_check.cu"),
                        "-I" + os.path.join(ROOT, "long_context_compressed_17_b300", "csrc"),
                        "-I" + os.path.join(ROOT, "include"), "-o", exe], check=True)
        out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0, out.stdout
    cases, bad = out.stdout.split()[1], out.stdout.split()[3]
    assert int(cases) > 100000 and int(bad) == 0
