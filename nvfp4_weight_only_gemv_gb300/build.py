"""Builds the CUDA library ``libnvfp4gemv.so`` in-tree for sm_103a with nvcc."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
SRC = os.path.join(PKG_DIR, "csrc", "nvfp4_gemv.cu")
HEADER = os.path.join(ROOT, "include", "nvfp4_gemv.h")
LIB_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(LIB_DIR, "libnvfp4gemv.so")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the NVFP4 GEMV library needs the CUDA toolkit to build")


def nvcc_command(out: str = LIB_PATH, extra: tuple = ()) -> list:
    return [nvcc_path(), ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xptxas=-warn-spills",
            "-I", os.path.join(ROOT, "include"), "-shared", "-Xcompiler", "-fPIC",
            *extra, "-o", out, SRC]


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in (SRC, HEADER))


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the library if it is missing or older than its sources; return its path."""
    if not force and not is_stale():
        return LIB_PATH
    os.makedirs(LIB_DIR, exist_ok=True)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = nvcc_command(tmp)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    if verbose and (res.stdout or res.stderr):
        print(res.stdout + res.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


def variant_path(name: str) -> str:
    return os.path.join(LIB_DIR, f"libnvfp4gemv_{name}.so")


def build_variant(name: str, defines: dict, force: bool = False) -> str:
    """Builds the same source with extra preprocessor definitions (the phase-trace diagnostic,
    planner experiments) into _build/libnvfp4gemv_<name>.so and returns its path. Load it by
    setting NVFP4_GEMV_LIBRARY to that path before the package first loads its library."""
    out = variant_path(name)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= max(os.path.getmtime(f) for f in (SRC, HEADER)):
        return out
    os.makedirs(LIB_DIR, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = nvcc_command(tmp, tuple(f"-D{k}={v}" for k, v in sorted(defines.items())))
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force=True, verbose=True))
