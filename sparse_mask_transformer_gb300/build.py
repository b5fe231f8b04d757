"""Builds libstof.so (the hot path) and libstof_synth.so (device input
generator) in-tree with nvcc for sm_103a.  Translation units compile in
parallel; objects go to ``_build/``.  No cmake, no torch extension
machinery: the libraries expose a plain C ABI."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libstof.so")
SYNTH_LIB = os.path.join(PKG, "libstof_synth.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]

STOF_SOURCES = ["stof_api.cu", "encode.cu", "rowwise.cu", "blockwise.cu", "blockwise_persist.cu", "tune.cu",
                "oproj.cu", "waitcheck.cu"]
SYNTH_SOURCES = ["synth_mask.cu"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _headers() -> list[str]:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def _compile(src: str, extra: list[str], verbose: bool) -> str:
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    if _stale(obj, [src] + _headers()):
        cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr.strip():
            print(r.stderr, file=sys.stderr)
    return obj


def _link(objs: list[str], out: str, verbose: bool) -> None:
    if _stale(out, objs):
        tmp = out + f".tmp{os.getpid()}"
        cmd = [_nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.check_call(cmd)
        os.replace(tmp, out)


def build(verbose: bool = False, extra_flags: list[str] | None = None) -> tuple[str, str]:
    """Compile both libraries (incrementally) and return their paths."""
    os.makedirs(BUILD, exist_ok=True)
    extra = list(extra_flags or [])
    srcs = [os.path.join(CSRC, s) for s in STOF_SOURCES + SYNTH_SOURCES]
    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, verbose), srcs))
    _link(objs[:len(STOF_SOURCES)], LIB, verbose)
    _link(objs[len(STOF_SOURCES):], SYNTH_LIB, verbose)
    return LIB, SYNTH_LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
