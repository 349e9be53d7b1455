"""The tcgen05 CTA-pair behaviour the dense attention kernel is built on.

`probes/pair_mma.cu` allocates TMEM collectively in a two-CTA cluster, issues
256-row MMAs from the even CTA in the shared-memory (QK^T) and TMEM (P V)
forms and a multicast commit, and compares each CTA's TMEM rows with products
computed on the host. The kernel relies on each CTA supplying 128 rows of A
and the even CTA the first half of B's N columns (the "hypothesis 0" line).
"""
import os
import shutil
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_pair_mma_semantics():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "pair_mma")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                        "-o", exe, os.path.join(HERE, "probes", "pair_mma.cu")], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    lines = out.stdout.splitlines()
    assert any(l.startswith("tmem addr") and l.endswith("status 0 0") for l in lines), out.stdout
    tm = next(l for l in lines if l.startswith("tmem addr"))
    assert tm.split()[3] == tm.split()[5].rstrip(";"), f"pair TMEM addresses differ: {tm}"
    assert "hypothesis 0: SS mismatches 0, TS mismatches 0 of 32768" in lines, out.stdout
