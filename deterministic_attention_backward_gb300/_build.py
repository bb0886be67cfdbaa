"""Builds libdash_attn.so in-tree with nvcc for sm_103a (GB300).

Each .cu translation unit is compiled in parallel into ``_build/`` and linked into
``deterministic_attention_backward_gb300/libdash_attn.so`` with the CUDA runtime linked
statically, so the library loads without a GPU (symbol checks on CPU-only machines).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libdash_attn.so")
SOURCES = ["api.cu", "bwd.cu", "bwd_varlen.cu", "fwd.cu", "aux.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(cand, "bin", "nvcc") if cand else ""
        if p and os.path.exists(p):
            return p
    p = shutil.which("nvcc")
    if not p:
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdash_attn.so")
    return p


def _deps() -> list[str]:
    out = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    out += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return out + [__file__]


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False,
          trace: bool = False) -> str:
    """Build the library (``trace=True``: the development variant with per-event clocks of
    CTA 0, written to ``_build/trace/libdash_attn_trace.so``; never the product library)."""
    out_dir = os.path.join(BUILD, "trace") if trace else BUILD
    lib = os.path.join(out_dir, "libdash_attn_trace.so") if trace else LIB
    os.makedirs(out_dir, exist_ok=True)
    deps = _deps()
    if not force and not _stale(lib, deps):
        return lib
    cc = nvcc()
    common = [cc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-I", INCLUDE, "-I", CSRC]
    if trace:
        common += ["-DDASH_TRACE_BUILD"]
    if ptxas_verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(src: str) -> tuple[str, str]:
        obj = os.path.join(out_dir, src.replace(".cu", ".o"))
        cmd = common + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_verbose:
        for _, log in results:
            if log.strip():
                print(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "--cudart", "static", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_verbose="-v" in sys.argv))
