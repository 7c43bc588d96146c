"""Builds libkvq.so in-tree with nvcc for sm_103a (GB300).

Each .cu file is compiled to an object in parallel, then linked into a
shared library next to this file.  Rebuilds only when a source, header or
flag changed.  ``python dynamically_quantized_paged_gb300/build.py [-f] [-v]``.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libkvq.so")

SOURCES = ["kvq_api.cu", "kvq_append.cu", "kvq_decode_int8.cu", "kvq_decode_fp8.cu",
           "kvq_decode_int4.cu", "kvq_decode_int4sym.cu", "kvq_decode_int8kc.cu", "kvq_merge.cu",
           "kvq_noalloc.cu"]
HEADERS = ["kvq_device.cuh", "kvq_internal.h", "kvq_decode.cuh", "kvq_tc.cuh", "kvq_alu.cuh", "kvq_quant.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                     "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvq.so")


def _fingerprint(extra: list[str]) -> str:
    h = hashlib.sha256()
    for name in SOURCES + HEADERS:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    with open(os.path.join(INCLUDE, "kvq.h"), "rb") as f:
        h.update(f.read())
    h.update(" ".join(NVCC_FLAGS + extra).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None) -> str:
    extra = list(extra_flags or [])
    if verbose:
        extra += ["-Xptxas", "-v"]
    fp = _fingerprint(extra)
    stamp = os.path.join(BUILD_DIR, "fingerprint")
    if not force and os.path.exists(LIB_PATH) and os.path.exists(stamp):
        if open(stamp).read() == fp:
            return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        cmd = [cc, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if verbose:
            sys.stderr.write(f"--- {src}\n{r.stderr}")
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    with open(stamp, "w") as f:
        f.write(fp)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="-f" in sys.argv, verbose="-v" in sys.argv))
