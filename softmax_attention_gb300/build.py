"""Builds libfa.so (the CUDA library behind include/fa.h) in-tree with nvcc for sm_103a."""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libfa.so")
SOURCES = ["abi.cu", "prefill.cu", "decode.cu", "decode_noalloc.cu", "mla.cu", "merge.cu",
           "selftest.cu", "gated_delta.cu", "prefill_f32.cu"]
HEADERS = [os.path.join(CSRC, h) for h in ("internal.h", "sm103.cuh", "prefill_common.cuh")] + [
    os.path.join(ROOT, "include", "fa.h")]

NVCC = os.environ.get("NVCC", "nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(OUT_DIR, os.path.splitext(src)[0] + ".o")
    path = os.path.join(CSRC, src)
    if not _stale(obj, [path] + HEADERS):
        return obj, ""
    tmp = obj + f".{os.getpid()}.tmp.o"
    r = subprocess.run([NVCC] + FLAGS + ["-c", path, "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, obj)
    return obj, r.stderr


def build(verbose: bool = False) -> str:
    """Compile every translation unit (in parallel) and link libfa.so; return its path."""
    os.makedirs(OUT_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    objs = [o for o, _ in results]
    report = "".join(log for _, log in results)
    if report:
        with open(os.path.join(OUT_DIR, "ptxas.txt"), "w") as f:
            f.write(report)
        if verbose:
            sys.stderr.write(report)
    if _stale(LIB, objs):
        tmp = LIB + f".{os.getpid()}.tmp"
        r = subprocess.run([NVCC] + ARCH + ["-shared", "-o", tmp] + objs,
                           capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
