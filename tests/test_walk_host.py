"""The launch-time token walk (walk_grid / set_walk / TokenWalk in
kimi_k3_attention_gb300/csrc) checked on the CPU: tests/walk_check.cu includes
the library's launch header, is built with nvcc and enumerates grids for many
token counts and resident-cluster counts.  Every token must be taken exactly
once and no cluster left idle while tokens remain."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "kimi_k3_attention_gb300", "csrc")


def test_walk_covers_every_token_once(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "walk_check")
    r = subprocess.run([nvcc, "-std=c++17", "-O2", "-I", CSRC, "-I", os.path.join(ROOT, "include"),
                        "-gencode", "arch=compute_103a,code=sm_103a",
                        os.path.join(ROOT, "tests", "walk_check.cu"), "-o", exe],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout[-2000:] + r.stderr[-2000:]
