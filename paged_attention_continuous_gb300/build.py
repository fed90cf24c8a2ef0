"""Build the C-ABI shared library ``_lib/libcb.so`` in-tree with nvcc.

Every CUDA translation unit is compiled for sm_103a only
(``-gencode arch=compute_103a,code=sm_103a``); translation units compile in
parallel, then nvcc links them into one shared library with the CUDA runtime
linked statically, so the library loads on a machine without a GPU driver
(the host scheduler works there; GPU calls report CB_ERR_CUDA).

Usage: ``python paged_attention_continuous_gb300/build.py [-v] [-f]`` (a standalone
script: it does not import the package, which needs the library).
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libcb.so")
ROOT = os.path.dirname(HERE)

SOURCES = ["scheduler.cpp", "kv_append.cu", "attention.cu", "prefill_attention.cu",
           "decode_bf16.cu", "decode_f32.cu", "decode_noalloc.cu", "kv_swap.cu", "validate.cpp",
           "tensor_map.cpp", "launch_common.cpp", "executor.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-lineinfo",
          "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _inputs_digest() -> str:
    h = hashlib.sha256()
    for d in (CSRC, os.path.join(ROOT, "include")):
        for name in sorted(os.listdir(d)):
            with open(os.path.join(d, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    h.update(" ".join(ARCH + COMMON).encode())
    return h.hexdigest()


def build(verbose: bool = False, force: bool = False, extra_flags=None) -> str:
    """Compile and link; returns the library path.  Skips work when the
    sources, flags and library are unchanged."""
    os.makedirs(OUT_DIR, exist_ok=True)
    digest = _inputs_digest() + ":" + " ".join(extra_flags or [])
    stamp = os.path.join(OUT_DIR, "build.stamp")
    if not force and os.path.exists(LIB) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read() == digest:
                return LIB
    nvcc = _nvcc()
    obj_dir = os.path.join(OUT_DIR, "obj")
    os.makedirs(obj_dir, exist_ok=True)
    flags = ARCH + COMMON + list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(obj_dir, src + ".o")
        cmd = [nvcc, "-c", os.path.join(CSRC, src), "-o", obj] + flags
        if verbose:
            cmd.append("-Xptxas=-v")
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp"
    cmd = [nvcc, "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(digest)
    return LIB


if __name__ == "__main__":
    v = "-v" in sys.argv
    print(build(verbose=v, force="-f" in sys.argv))
