"""In-tree build of libfi_gb300.so for sm_103a with nvcc (no cmake)."""
from __future__ import annotations

import glob
import os
import subprocess
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_DIR = os.path.join(HERE, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libfi_gb300.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fno-strict-aliasing"]
_lock = threading.Lock()


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _inputs():
    return _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def is_stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit in parallel, then link the shared library."""
    with _lock:
        if not force and not is_stale():
            return LIB_PATH
        os.makedirs(BUILD_DIR, exist_ok=True)
        os.makedirs(LIB_DIR, exist_ok=True)
        procs, objs = [], []
        for src in _sources():
            obj = os.path.join(BUILD_DIR, os.path.basename(src) + ".o")
            cmd = [NVCC, *ARCH, *FLAGS, "-I", INCLUDE, "-c", src, "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
            objs.append(obj)
        errors = []
        for src, pr in procs:
            out, _ = pr.communicate()
            if verbose and out:
                print(out)
            if pr.returncode != 0:
                errors.append(f"{src}:\n{out}")
        if errors:
            raise RuntimeError("nvcc failed:\n" + "\n".join(errors))
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call([NVCC, *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, LIB_PATH)
        return LIB_PATH
