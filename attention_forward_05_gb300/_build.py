"""Builds libfa.so in-tree with nvcc for sm_103a (no CMake, no torch extension machinery).

The translation units compile in parallel; the shared library links the
CUDA runtime statically, so it depends only on the driver.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libfa.so")
SOURCES = ["fa_api.cu", "fa_fwd_bf16.cu", "fa_fwd_fp32.cu", "fa_fwd_merge.cu", "fa_decode.cu",
           "fa_decode_noalloc.cu", "fa_bwd.cu", "fa_bwd_fp32.cu",
           "fa_decode_gqa.cu", "fa_fwd_decode.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "fa.h"))
    files.append(os.path.abspath(__file__))
    return files


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale or forced) and return the path of libfa.so.

    FA_PTXAS_VERBOSE=1 in the environment adds ``-Xptxas -v`` and keeps its
    register / spill report in _build/ptxas.log.
    """
    if not force and not is_stale():
        return LIB
    os.makedirs(OUT, exist_ok=True)
    nvcc = _nvcc()
    ptxas_v = os.environ.get("FA_PTXAS_VERBOSE") == "1"
    flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                    "--expt-relaxed-constexpr"]
    if ptxas_v:
        flags += ["-Xptxas", "-v"]

    def compile_one(src: str):
        obj = os.path.join(OUT, src.replace(".cu", ".o"))
        cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    log = []
    for src, _, r in results:
        log.append(f"== {src}\n{r.stdout}{r.stderr}")
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError(f"nvcc failed on {src}")
    if ptxas_v or verbose:
        with open(os.path.join(OUT, "ptxas.log"), "w") as f:
            f.write("\n".join(log))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *[obj for _, obj, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc link failed")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
