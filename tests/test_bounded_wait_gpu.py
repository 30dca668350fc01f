"""Failure detection on the GPU without a fault: a kernel waits on an
mbarrier that nothing arrives at, through the same bounded wait every libpa
kernel uses (tests/bounded_wait/wait_timeout.cu).  The wait must end by
itself within about a second with PA_DEVERR_TIMEOUT in the device error word,
and the context must stay usable for the next kernel."""
import json
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PA_DEVERR_TIMEOUT = 4


def test_wait_that_never_completes_times_out(cuda_device, tmp_path):
    nvcc = shutil.which("nvcc") or os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "wait_timeout")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-std=c++17",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(ROOT, "paged_kv_flashattention_gb300", "csrc"),
           os.path.join(ROOT, "tests", "bounded_wait", "wait_timeout.cu"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    line = r.stdout.strip().splitlines()[-1] if r.stdout.strip() else "{}"
    res = json.loads(line)
    assert r.returncode == 0, r.stdout + r.stderr
    assert res["first"] == "no error" and res["first_wait_completed"] == 0
    assert res["error_word"] & PA_DEVERR_TIMEOUT
    assert 10.0 < res["first_wait_ms"] < 5000.0
    assert res["second"] == "no error" and res["second_wait_completed"] == 1
