"""The C ABI from plain C: a program that includes only grpo.h and the CUDA
runtime header, links libgrpo.so and runs a whole step (advantages, mask,
forward, forward+backward) on its own cudaMalloc'd buffers, then the same
batch as two data-parallel shards; it checks its own statuses, the bitwise
equality of the two losses, and that the shards add up to the batch; two runs
print the same bits."""
import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def test_plain_c_program_runs_a_step(tmp_path):
    from rl_fine_tuning_gb300 import build
    build.build()
    cuda = _cuda_home()
    libdirs = [p for p in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib")) if os.path.isdir(p)]
    exe = tmp_path / "grpo_step"
    cmd = ["gcc", "-O2", "-std=c11", "-o", str(exe), os.path.join(ROOT, "tests", "c_abi", "grpo_step.c"),
           "-I" + os.path.join(ROOT, "include"), "-I" + os.path.join(cuda, "include"),
           "-L" + os.path.dirname(build.LIB), "-Wl,-rpath," + os.path.dirname(build.LIB)]
    for d in libdirs:
        cmd += ["-L" + d, "-Wl,-rpath," + d]
    cmd += ["-lgrpo", "-lcudart", "-lm"]
    subprocess.check_call(cmd)
    out1 = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out1.returncode == 0, out1.stderr
    out2 = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out2.returncode == 0, out2.stderr
    assert out1.stdout.startswith("ok ") and out1.stdout == out2.stdout
