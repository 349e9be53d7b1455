"""What an MMA-issuing thread's own waits cost the tensor core.

`probes/mma_issue.cu` issues groups of tcgen05.mma from one thread and adds,
between groups, a fence or a wait on an mbarrier phase that has already
completed. The fence is free. The wait holds back the thread's next MMA by
about 200 cycles (a 4-MMA QK^T group goes from ~256 to ~470 cycles), even
though it returns at once, and so does a poll of a shared-memory word that is
already set. With the same waits spread over two issuing threads in different
warps, the tensor core runs one thread's MMAs in the other's gap.

These figures explain the attention kernels' MMA loop: each of its waits (K
converted, V landed, each stage's P) costs the tensor core about as much as
three N = 128 MMAs. In those kernels the variants that act on this (waits
folded into other threads' signals, a second issuing thread) measured slower
than the single issuer, so it stays.
"""
import os
import re
import shutil
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def _run_probe():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "mma_issue")
        subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                        "-o", exe, os.path.join(HERE, "probes", "mma_issue.cu")], check=True)
        out = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    cyc = {}
    for line in out.stdout.splitlines():
        m = re.match(r"case (\d+) (\S+): ([\d.]+) cycles per group, done=(\d)", line)
        if m:
            assert m.group(4) == "1", line
            cyc[int(m.group(1))] = float(m.group(3))
    assert sorted(cyc) == list(range(11)), out.stdout
    return cyc


def test_issuer_waits_cost_the_tensor_core():
    cyc = _run_probe()
    # 4 SS MMAs of 128 x 128 x 16 run at ~64 cycles each
    assert 200.0 < cyc[0] < 330.0, cyc
    # a commit and a fence between groups are (nearly) free
    assert cyc[1] < 1.15 * cyc[0], cyc
    # a wait on a completed phase is not
    assert cyc[2] > cyc[0] + 100.0, cyc
    assert cyc[3] > cyc[0] + 100.0, cyc
    # the kernel-shaped group: two waits per group cost a large share ...
    assert cyc[5] > 1.3 * cyc[4], cyc
    # ... which a second issuing thread in another warp recovers
    assert cyc[6] < 0.75 * cyc[5], cyc
    # polling a shared-memory word that is already set, with an acquire or a
    # volatile load, costs the same as the mbarrier wait: any shared-memory
    # result the issuing thread waits on does, while the MMAs read their
    # operands from shared memory
    assert cyc[7] > cyc[0] + 100.0 and cyc[8] > cyc[0] + 100.0, cyc
    assert cyc[9] > 1.3 * cyc[4] and cyc[10] > 1.3 * cyc[4], cyc
