"""The kernels' mbarrier waits are bounded: a wait on a phase that nothing
completes gives up after its iteration limit, the kernel reports it and
returns, and the next launch runs normally (no fault, no hang)."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "context_paged_decode_gb300", "csrc")


def test_bounded_wait_gives_up_and_the_context_stays_usable(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    exe = str(tmp_path / "wait_bound")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
                    "-I", CSRC, "-o", exe, os.path.join(HERE, "wait_bound.cu")],
                   check=True, capture_output=True, timeout=300)
    out = subprocess.run([exe], check=True, capture_output=True, text=True, timeout=300).stdout
    print(out.strip())
    f = out.split()
    errors = [int(x) for x in f[1:4]]
    status = [int(x) for x in f[5:7]]
    seconds = float(f[8])
    assert errors == [0, 0, 0], out
    assert status == [2, 1], out          # gave up; then a completed wait
    assert seconds < 120.0, out           # bounded well below a stuck launch
