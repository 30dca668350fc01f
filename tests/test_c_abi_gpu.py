"""The C ABI from plain C: tests/c_abi/abi_closed_form.c includes only
include/pa.h, links libpa.so and the CUDA runtime, stores tokens and runs split
decode (pa_decode and pa_decode_noalloc) and causal extend (pa_prefill) on
cases with closed-form answers (equal keys: the output is the mean of the
visible V rows), and exits 0 when every element matches."""
import glob
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home():
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def test_c_program_abi_closed_form(cuda_device, tmp_path):
    import paged_kv_flashattention_gb300 as pa     # the in-tree libpa.so is built
    assert pa.abi_version() == 3
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    cuda = _cuda_home()
    libdirs = [d for d in [os.path.join(cuda, "lib64")] + glob.glob(os.path.join(cuda, "targets", "*", "lib"))
               if os.path.exists(os.path.join(d, "libcudart.so"))]
    assert libdirs, f"libcudart.so not found under {cuda}"
    pkg = os.path.join(ROOT, "paged_kv_flashattention_gb300")
    exe = str(tmp_path / "abi_closed_form")
    cmd = [gcc, "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
           os.path.join(ROOT, "tests", "c_abi", "abi_closed_form.c"),
           "-L", pkg, "-lpa", "-L", libdirs[0], "-lcudart", "-lm",
           f"-Wl,-rpath,{pkg}", f"-Wl,-rpath,{libdirs[0]}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.startswith("ok")
