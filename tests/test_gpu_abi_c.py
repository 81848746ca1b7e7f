"""The C ABI from plain C: tests/native/abi_from_c.c is compiled by gcc (no
CUDA compiler, no Python in the program) against include/rr.h, linked with
librr.so and the CUDA runtime, and run; it calls every collective entry
point and checks the results exactly."""
import os
import shutil
import subprocess

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime_api.h")):
            return cand
    pytest.fail("CUDA toolkit headers not found")


def test_abi_from_plain_c(tmp_path):
    if not torch.cuda.is_available():
        pytest.fail("this test needs a CUDA GPU")
    from allgather_rr_allreduce_gb300 import build
    lib = build.build()
    gcc = shutil.which("gcc")
    assert gcc, "gcc not found"
    cuda = _cuda_home()
    libdir = os.path.dirname(lib)
    cudalib = next(d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"),
                               os.path.join(cuda, "targets", "sbsa-linux", "lib"))
                   if os.path.exists(os.path.join(d, "libcudart.so")))
    exe = tmp_path / "abi_from_c"
    subprocess.run([gcc, "-std=c11", "-O1", "-Wall", "-Wextra", "-Werror",
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"),
                    os.path.join(ROOT, "tests", "native", "abi_from_c.c"),
                    "-L", libdir, "-lrr", "-L", cudalib, "-lcudart",
                    f"-Wl,-rpath,{libdir}:{cudalib}", "-o", str(exe)], check=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "abi_from_c ok" in res.stdout
