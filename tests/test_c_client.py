"""The C ABI from plain C: tests/c_client/ep_client.c is built with gcc against
include/ep_gb300.h and libep_gb300.so alone (no Python or PyTorch in the
process).  Its query mode needs no GPU; its GPU mode runs a small batch through
ep_dispatch_with_layout and ep_combine and checks combine(dispatch(x)) = d_t x
exactly."""
import os
import shutil
import subprocess

import pytest

from combine_ep_dispatch_gb300 import _build, _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_client", "ep_client.c")


def _compile(out, gpu):
    if shutil.which("gcc") is None:
        pytest.skip("gcc is not installed")
    _build.build_library()
    libdir = os.path.dirname(_lib.LIB_PATH)
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), SRC,
           "-o", out, "-L", libdir, "-l:" + os.path.basename(_lib.LIB_PATH),
           "-Wl,-rpath," + libdir]
    if gpu:
        cuda = _build.cuda_home()
        cmd[1:1] = ["-DEP_CLIENT_GPU", "-I", os.path.join(cuda, "include")]
        cmd += ["-L", os.path.join(cuda, "lib64"), "-lcudart", "-Wl,-rpath," + os.path.join(cuda, "lib64")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_client_query_mode(tmp_path):
    exe = str(tmp_path / "ep_client")
    _compile(exe, gpu=False)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert "query mode ok" in r.stdout


@pytest.mark.gpu
def test_c_client_gpu_mode(tmp_path):
    exe = str(tmp_path / "ep_client_gpu")
    _compile(exe, gpu=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "gpu mode ok" in r.stdout
