"""Builds libcpattn.so in-tree with nvcc for sm_103a.

One object per translation unit, compiled in parallel, linked with the static
CUDA runtime (the library resolves the driver's tensor-map encoder at run
time, so it loads on machines without a GPU driver).

``build(check=True)`` builds the bounds-checking variant libcpattn_check.so
(-DCPATTN_CHECK, a debugging aid with the same ABI) next to it.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG, "libcpattn.so")
CHECK_LIB_PATH = os.path.join(PKG, "libcpattn_check.so")
SOURCES = ["attn_fwd.cu", "merge_permute.cu", "cpattn_api.cu", "ring_noalloc.cu"]
HEADERS = ["internal.h", "ptx.cuh", "tmem_ops.cuh", "check.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libcpattn.so")


def _stale(lib_path: str) -> bool:
    if not os.path.exists(lib_path):
        return True
    t = os.path.getmtime(lib_path)
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps += [os.path.join(ROOT, "include", "cpattn.h"), os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def build(force: bool = False, verbose: bool = False, extra_flags=None, check: bool = False) -> str:
    lib_path = CHECK_LIB_PATH if check else LIB_PATH
    if not force and not _stale(lib_path):
        return lib_path
    build_dir = os.path.join(BUILD_DIR, "check") if check else BUILD_DIR
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-I", os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]
    if check:
        flags.append("-DCPATTN_CHECK")
    flags += list(extra_flags or [])
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [cc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    errors = []
    for src, proc in procs:
        out, _ = proc.communicate()
        text = out.decode(errors="replace")
        if proc.returncode != 0:
            errors.append(f"{src}:\n{text}")
        elif verbose and text.strip():
            print(text, file=sys.stderr)
    if errors:
        raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
    tmp = lib_path + f".{os.getpid()}.tmp"
    link = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    res = subprocess.run(link, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("link failed:\n" + res.stdout + res.stderr)
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, check="--check" in sys.argv))
