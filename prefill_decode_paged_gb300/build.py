"""Build the in-tree CUDA library ``_build/libkv_relayout.so`` for sm_103a with nvcc."""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libkv_relayout.so")
# the same library with device-side address checks (KVR_DEVICE_CHECKS; tests only)
LIB_CHECKED = os.path.join(BUILD, "libkv_relayout_checked.so")
SOURCES = ["plan.cpp", "relayout.cu", "sm_stream.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    home = os.environ.get("CUDA_HOME") or os.environ.get("CUDA_PATH")
    if home and os.path.exists(os.path.join(home, "bin", "nvcc")):
        return os.path.join(home, "bin", "nvcc")
    found = shutil.which("nvcc")
    if found:
        return found
    raise RuntimeError("nvcc not found: set CUDA_HOME or put nvcc on PATH")


def _cuda_libdir(nvcc: str) -> str:
    home = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    for cand in ("lib64", "lib"):
        if os.path.isdir(os.path.join(home, cand)):
            return os.path.join(home, cand)
    return os.path.join(home, "lib64")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    files.append(os.path.join(INCLUDE, "kv_relayout.h"))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=(), lib: str = LIB) -> str:
    """Compile the translation units in parallel, then link; return the library path."""
    if not force and up_to_date(lib):
        return lib
    nvcc = nvcc_path()
    os.makedirs(BUILD, exist_ok=True)
    common = ["-O3", "-std=c++17", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC",
              "-I", INCLUDE, "-I", CSRC, *extra_flags]
    tag = os.path.splitext(os.path.basename(lib))[0]
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(BUILD, f"{tag}.{src}.o")
        cmd = [nvcc, *common, "-c", os.path.join(CSRC, src), "-o", obj]
        if src.endswith(".cu") and verbose:
            cmd += ["-Xptxas", "-v"]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                            stderr=subprocess.STDOUT, text=True)))
        objs.append(obj)
    for cmd, p in procs:
        out, _ = p.communicate()
        if verbose and out:
            print(out)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed ({' '.join(cmd)}):\n{out}")
    tmp = lib + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
            "-Xlinker", "-rpath," + _cuda_libdir(nvcc)]
    res = subprocess.run(link, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)
    return lib


def build_checked(force: bool = False) -> str:
    """The library with device-side address checks (kv_relayout_debug_status): every
    row a kernel computes is checked against the plan's pools before it is used."""
    return build(force=force, extra_flags=("-DKVR_DEVICE_CHECKS=1",), lib=LIB_CHECKED)


if __name__ == "__main__":
    print(build(force=True, verbose=True))
