"""Build the CUDA library libpagedattn.so in-tree for sm_103a (nvcc only, no cmake).

Each translation unit is compiled in parallel, then linked into one shared library
next to this file. Used by ``__graft_entry__.build()``; also runnable directly:
``python -m paged_kv_attention_gb300.build [--verbose-ptxas]``.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpagedattn.so")
SOURCES = ["pa_api.cu", "cache_write.cu", "decode.cu", "decode_seg.cu", "varlen_tc.cu", "varlen_tc256.cu",
           "decode_static_scratch.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(ptxas_verbose: bool) -> list[str]:
    f = ["-O3", "-std=c++17", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC", "-I", INCLUDE,
         "--expt-relaxed-constexpr", "-Xcompiler", "-Wall"]
    if ptxas_verbose:
        f += ["-Xptxas", "-v"]
    return f


def _compile(src: str, ptxas_verbose: bool) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *_flags(ptxas_verbose), "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stdout + r.stderr


def is_stale() -> bool:
    """True when the library is missing or older than any source or header."""
    if not os.path.exists(LIB):
        return True
    built = os.path.getmtime(LIB)
    srcs = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + \
        [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return any(os.path.getmtime(f) > built for f in srcs)


def build(ptxas_verbose: bool = False, quiet: bool = True) -> str:
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, ptxas_verbose), SOURCES))
    objs = [o for o, _ in results]
    if not quiet or ptxas_verbose:
        for _, log in results:
            if log.strip():
                print(log)
    tmp = LIB + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lrt", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(ptxas_verbose="--verbose-ptxas" in sys.argv, quiet=False))
