"""Build libkvint4.so in-tree with nvcc for sm_103a (GB300).

The translation units are compiled in parallel and linked with the static
CUDA runtime, so loading the library needs only the NVIDIA driver.  A stamp
file records the host architecture and a hash of the sources, so a library
built on another machine (or from other sources) is rebuilt.
"""

from __future__ import annotations

import hashlib
import os
import platform
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libkvint4.so")
STAMP = os.path.join(BUILD_DIR, "stamp.txt")
HEADER = os.path.join(ROOT, "include", "kvint4.h")

SOURCES = ["api.cu", "write.cu", "write_int8.cu", "attention.cu", "rht.cu", "timing.cu", "noalloc.cu", "selftest.cu"]
GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden"]


def nvcc_path() -> str:
    cand = shutil.which("nvcc")
    if cand:
        return cand
    for p in ("/usr/local/cuda/bin/nvcc",):
        if os.path.exists(p):
            return p
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvint4.so")


def _inputs():
    files = [os.path.join(CSRC, f) for f in sorted(os.listdir(CSRC))
             if f.endswith((".cu", ".cuh", ".h"))]
    return files + [HEADER, os.path.abspath(__file__)]


def _fingerprint(extra=()) -> str:
    h = hashlib.sha256()
    h.update(platform.machine().encode())
    for f in _inputs():
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
    for e in extra:
        h.update(str(e).encode())
    return h.hexdigest()


def is_current(extra=()) -> bool:
    if not os.path.exists(LIB_PATH) or not os.path.exists(STAMP):
        return False
    with open(STAMP) as f:
        return f.read().strip() == _fingerprint(extra)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile (if needed) and return the path of libkvint4.so."""
    if not force and is_current():
        return LIB_PATH
    nvcc = nvcc_path()
    os.makedirs(BUILD_DIR, exist_ok=True)
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc, *GENCODE, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if ptxas_info:
            cmd.insert(1, "-Xptxas=-v")
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    logs = {}
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        logs[src] = out
        if p.returncode != 0:
            failed.append(src)
    if failed:
        msg = "\n".join(f"--- {s} ---\n{logs[s]}" for s in failed)
        raise RuntimeError(f"nvcc failed for {failed}:\n{msg}")
    tmp = LIB_PATH + ".tmp"
    link = [nvcc, *GENCODE, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}")
    os.replace(tmp, LIB_PATH)
    with open(STAMP, "w") as f:
        f.write(_fingerprint())
    if verbose or ptxas_info:
        for s in SOURCES:
            if logs[s].strip():
                print(f"--- {s} ---\n{logs[s]}", file=sys.stderr)
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB_PATH)
