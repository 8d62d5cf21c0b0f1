"""The C ABI from plain C: tests/c_abi_consumer.c includes only include/ss.h, links libss.so and
checks host calls (layout, accounting, argument errors before any launch) and, on a GPU, device
calls on cudaMalloc'd buffers (an exact rank-ordered reduce, the first AdamW step against its
closed form, an unshard/reshard round trip). No Python or PyTorch is on that path."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi_consumer.c")


def _cuda_home():
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp_path, gpu: bool) -> str:
    import fsdp_sharded_mixed_ss_gb300 as ss

    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib_dir = os.path.dirname(os.path.abspath(ss.LIB_PATH))
    exe = str(tmp_path / ("consumer_gpu" if gpu else "consumer"))
    cmd = [cc, "-std=c99", "-O1", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), SRC, "-o", exe,
           "-L", lib_dir, "-lss", "-Wl,-rpath," + lib_dir, "-lm"]
    if gpu:
        home = _cuda_home()
        cmd[1:1] = ["-DSS_WITH_CUDA", "-I", os.path.join(home, "include")]
        cmd += ["-L", os.path.join(home, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(home, "lib64")]
    p = subprocess.run(cmd, capture_output=True, text=True)
    assert p.returncode == 0, p.stderr
    return exe


def test_c_consumer_host_calls(tmp_path):
    exe = _build(tmp_path, gpu=False)
    p = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert p.returncode == 0 and p.stdout.strip() == "OK", p.stdout + p.stderr


@pytest.mark.gpu
def test_c_consumer_device_calls(tmp_path):
    exe = _build(tmp_path, gpu=True)
    p = subprocess.run([exe, "gpu"], capture_output=True, text=True, timeout=300)
    assert p.returncode == 0 and p.stdout.strip() == "OK", p.stdout + p.stderr
