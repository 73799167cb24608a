"""Build step of the CUDA library: compiles csrc/*.cu for sm_103a with nvcc and
links libep_gb300.so into this package directory (in-tree, no install step).

The translation units compile in parallel; ptxas register / spill / shared
memory reports land in _build/ptxas.log beside the objects."""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libep_gb300.so")
HEADERS = [os.path.join(ROOT, "include", "ep_gb300.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler",
              "-fvisibility=hidden", "-Xptxas", "-v", "--expt-relaxed-constexpr"]


def cuda_home() -> str:
    env = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if env:
        return env
    nvcc = shutil.which("nvcc")
    if nvcc:
        return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    return "/usr/local/cuda"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + HEADERS + [__file__]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build_library(force: bool = False, verbose: bool = False, out: str | None = None,
                  build_dir: str | None = None) -> str:
    """Compile and link the library; with ``out`` the result goes to that path
    instead of the package's libep_gb300.so."""
    if not force and out is None and up_to_date():
        return LIB
    lib_path = out or LIB
    build = build_dir or BUILD
    nvcc = os.path.join(cuda_home(), "bin", "nvcc")
    if not os.path.exists(nvcc):
        nvcc = "nvcc"
    os.makedirs(build, exist_ok=True)
    srcs = _sources()

    def compile_one(src):
        obj = os.path.join(build, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), "-c", src,
               "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(compile_one, srcs))
    with open(os.path.join(build, "ptxas.log"), "w") as f:
        for (obj, log) in results:
            f.write(f"== {os.path.basename(obj)}\n{log}\n")
    if verbose:
        for _, log in results:
            print(log)
    lib64 = os.path.join(cuda_home(), "lib64")
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *[o for o, _ in results],
           "-Xlinker", f"-rpath,{lib64}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build_library(force=True, verbose=True))
