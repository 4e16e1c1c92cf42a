"""Builds the CUDA library libgqa_attn.so in-tree for sm_103a.

Each .cu file under csrc/ is compiled by its own nvcc process (in parallel),
then the objects are linked into one shared library next to this file. The
library links the shared CUDA runtime, so inside a process that already
loaded PyTorch it uses the same runtime instance (same current device, same
streams). Only one -gencode target is built: arch=compute_103a,code=sm_103a.

Usage:  python -m gqa_flash_attention_02_gb300.build [--force]
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(HERE, "libgqa_attn.so")

SOURCES = ["api.cu", "prefill_tc.cu", "decode_splitkv.cu", "attn_f32.cu", "decode_noalloc.cu",
           "attn_bwd.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgqa_attn.so")
    return cand


def _cuda_lib_dir(nvcc: str) -> str:
    home = os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))
    for sub in ("lib64", "lib", os.path.join("targets", "sbsa-linux", "lib"),
                os.path.join("targets", "x86_64-linux", "lib")):
        p = os.path.join(home, sub)
        if os.path.exists(os.path.join(p, "libcudart.so")):
            return p
    return os.path.join(home, "lib64")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of libgqa_attn.so."""
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= _deps_mtime():
        return LIB_PATH
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc, "-c", os.path.join(CSRC, src), "-o", obj] + common
        if verbose:
            cmd += ["-Xptxas", "-v"]
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                            text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append(f"--- {src}\n{out}")
        elif verbose and out:
            print(f"--- {src}\n{out}", file=sys.stderr)
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    libdir = _cuda_lib_dir(nvcc)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    link = [nvcc, "-shared", "--cudart", "shared", "-o", tmp] + objs + ARCH + [
        "-L", libdir, "-Xlinker", f"-rpath,{libdir}"]
    res = subprocess.run(link, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("link failed:\n" + res.stdout + res.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
