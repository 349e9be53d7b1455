"""The MMA shape costs the block-sparse kernel's design rests on.

`probes/mma_shapes.cu` times tcgen05.mma kind::f16 on one CTA. An M = 64 MMA
takes as many cycles as an M = 128 MMA of the same N (SS and TS), so giving
each 64-row query tile its own MMAs would double the tensor time per useful
score; the block-sparse kernel instead runs 128-row MMAs over the union of
two query tiles' key lists (about 97 key tiles for two tiles that keep 80
each, against 160 half-used ones). The probe also shows the N = 64 floor
(~50-55 cycles, against 64 for N = 128) that makes head-dim-64 P V MMAs run
at about 60% of the N = 128 rate.
"""
import os
import re
import shutil
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_m64_mma_costs_as_much_as_m128():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "mma_shapes")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                        "-o", exe, os.path.join(HERE, "probes", "mma_shapes.cu")], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    cyc = {}
    for line in out.stdout.splitlines():
        m = re.match(r"(SS|TS) M=(\d+) N=(\d+) K=16: ([\d.]+) cycles per MMA .* done=(\d)", line)
        if m:
            assert m.group(5) == "1", line
            cyc[(m.group(1), int(m.group(2)), int(m.group(3)))] = float(m.group(4))
    assert len(cyc) == 10, out.stdout
    for (form, M, N), c in cyc.items():
        if M == 64:
            assert c >= 0.8 * cyc[(form, 128, N)], (form, N, c, cyc[(form, 128, N)])
