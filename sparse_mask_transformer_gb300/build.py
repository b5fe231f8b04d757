"""Builds libstof.so (the hot path) and libstof_synth.so (device input
generator) in-tree with nvcc for sm_103a.  Translation units compile in
parallel; objects go to ``_build/``.  No cmake, no torch extension
machinery: the libraries expose a plain C ABI.

Staleness is decided by content, not by file times: every object and
library has a ``.srchash`` file beside it holding the SHA-256 of what it was
built from (its sources, every header, the compiler flags, the nvcc version
line and the host machine type).  A copy of the tree whose binaries came
from another machine, or from other sources, is rebuilt.  ``source_hash()``
is the hash of the current sources and flags, which the library built from
them carries."""
from __future__ import annotations

import hashlib
import os
import platform
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


_NVCC_VERSION: str | None = None


def _nvcc_version() -> str:
    global _NVCC_VERSION
    if _NVCC_VERSION is None:
        out = subprocess.run([_nvcc(), "--version"], capture_output=True, text=True).stdout
        _NVCC_VERSION = [ln for ln in out.splitlines() if ln.strip()][-1] if out.strip() else "unknown"
    return _NVCC_VERSION


def _headers() -> list[str]:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return sorted(hs)


def _digest(files: list[str], flags: list[str]) -> str:
    h = hashlib.sha256()
    for f in files:
        h.update(os.path.basename(f).encode() + b"\0")
        with open(f, "rb") as fh:
            h.update(fh.read())
        h.update(b"\0")
    h.update(" ".join(flags).encode())
    h.update(_nvcc_version().encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def _read_hash(target: str) -> str | None:
    try:
        with open(target + ".srchash") as f:
            return f.read().strip()
    except OSError:
        return None


def _write_hash(target: str, digest: str) -> None:
    with open(target + ".srchash", "w") as f:
        f.write(digest + "\n")


def _fresh(target: str, digest: str) -> bool:
    return os.path.exists(target) and _read_hash(target) == digest


def source_hash(extra_flags: list[str] | None = None) -> str:
    """SHA-256 (first 16 hex digits) of libstof.so's sources, headers and
    build flags on this machine: the hash a library built from them carries."""
    srcs = [os.path.join(CSRC, s) for s in STOF_SOURCES]
    return _digest(srcs + _headers(), [*ARCH, *NVCC_FLAGS, *(extra_flags or [])])[:16]


def built_hash(lib: str = LIB) -> str | None:
    """The source hash recorded beside a built library (None if absent)."""
    h = _read_hash(lib)
    return h[:16] if h else None


def _compile(src: str, extra: list[str], verbose: bool) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.basename(src) + ".o")
    flags = [*ARCH, *NVCC_FLAGS, *extra]
    digest = _digest([src] + _headers(), flags)
    if not _fresh(obj, digest):
        cmd = [_nvcc(), *flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr.strip():
            print(r.stderr, file=sys.stderr)
        _write_hash(obj, digest)
    return obj, digest


def _link(objs: list[str], out: str, digest: str, verbose: bool) -> None:
    if not _fresh(out, digest):
        tmp = out + f".tmp{os.getpid()}"
        cmd = [_nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.check_call(cmd)
        os.replace(tmp, out)
        _write_hash(out, digest)


def build(verbose: bool = False, extra_flags: list[str] | None = None) -> tuple[str, str]:
    """Compile both libraries (incrementally, by content hash) and return
    their paths."""
    os.makedirs(BUILD, exist_ok=True)
    extra = list(extra_flags or [])
    srcs = [os.path.join(CSRC, s) for s in STOF_SOURCES + SYNTH_SOURCES]
    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, verbose), srcs))
    n = len(STOF_SOURCES)
    flags = [*ARCH, *NVCC_FLAGS, *extra]
    _link([o for o, _ in objs[:n]], LIB, _digest(srcs[:n] + _headers(), flags), verbose)
    _link([o for o, _ in objs[n:]], SYNTH_LIB, _digest(srcs[n:] + _headers(), flags), verbose)
    return LIB, SYNTH_LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
