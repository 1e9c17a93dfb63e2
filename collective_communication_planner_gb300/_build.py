"""Builds libtccl.so in place: host C++ with g++, kernels with nvcc for sm_103a.

Translation units compile in parallel; the result is linked with the static
CUDA runtime so the library has no run-time path requirements.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
LIB = PKG / "libtccl.so"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]

HOST_SOURCES = ["api.cpp", "plan.cpp", "reshard.cpp", "copy_out_host.cpp"]
CUDA_SOURCES = ["kernels_bulk.cu", "kernels_small_ar.cu", "kernels_small_rs.cu",
                "kernels_small_ag.cu", "kernels_reshard.cu", "kernels_rmsnorm.cu",
                "no_alloc.cu", "kernels_copy_out.cu"]


def _cuda_home() -> Path:
    env = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if env:
        return Path(env)
    nvcc = shutil.which("nvcc")
    if nvcc:
        return Path(nvcc).resolve().parent.parent
    return Path("/usr/local/cuda")


def _sources():
    return ([CSRC / s for s in HOST_SOURCES + CUDA_SOURCES] +
            list(CSRC.glob("*.h")) + list(CSRC.glob("*.cuh")) + [INCLUDE / "tccl.h"])


def up_to_date() -> bool:
    if not LIB.exists():
        return False
    t = LIB.stat().st_mtime
    return all(p.stat().st_mtime <= t for p in _sources())


def build(force: bool = False, verbose: bool = False) -> Path:
    if not force and up_to_date():
        return LIB
    cuda = _cuda_home()
    nvcc = str(cuda / "bin" / "nvcc")
    obj_dir = PKG / "_build"
    obj_dir.mkdir(exist_ok=True)
    inc = [f"-I{INCLUDE}", f"-I{CSRC}", f"-I{cuda / 'include'}"]
    jobs = []
    for s in HOST_SOURCES:
        jobs.append(["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-Wno-unused-function",
                     *inc, "-c", str(CSRC / s), "-o", str(obj_dir / (s + ".o"))])
    for s in CUDA_SOURCES:
        jobs.append([nvcc, *ARCH, "-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC",
                     *inc, "-c", str(CSRC / s), "-o", str(obj_dir / (s + ".o"))])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        for cmd, r in ex.map(run, jobs):
            if r.returncode != 0:
                raise RuntimeError("build failed: " + " ".join(cmd) + "\n" + r.stdout + r.stderr)
            if verbose and (r.stdout or r.stderr):
                print(r.stdout + r.stderr)
    tmp = LIB.with_suffix(f".{os.getpid()}.tmp")
    link = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", str(tmp),
            *[str(obj_dir / (s + ".o")) for s in HOST_SOURCES + CUDA_SOURCES]]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed: " + " ".join(link) + "\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
