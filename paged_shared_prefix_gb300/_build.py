"""Builds libpsp.so (the CUDA kernels and the C ABI) in-tree for sm_103a.

Every translation unit under csrc/ is compiled by nvcc in parallel into
_build/, then linked into paged_shared_prefix_gb300/libpsp.so against the
shared CUDA runtime.  Only changed sources are recompiled.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpsp.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
          "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpsp.so")


def _headers_digest() -> str:
    h = hashlib.sha256()
    for f in sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                    glob.glob(os.path.join(INCLUDE, "*.h"))):
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def _compile(src: str, digest: str, extra: list) -> str:
    base = os.path.splitext(os.path.basename(src))[0]
    obj = os.path.join(BUILD, f"{base}.{digest}.o")
    if os.path.exists(obj) and os.path.getmtime(obj) >= os.path.getmtime(src):
        return obj
    cmd = [nvcc()] + ARCH + COMMON + extra + ["-c", src, "-o", obj + ".tmp"]
    if src.endswith(".cpp"):
        cmd = [nvcc()] + COMMON + extra + ["-x", "c++", "-c", src, "-o", obj + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stderr}")
    os.replace(obj + ".tmp", obj)
    return obj


def build(verbose: bool = False, extra: list = None, ptxas_info: bool = False) -> str:
    """Compile every csrc/*.cu and csrc/*.cpp and link libpsp.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    extra = list(extra or [])
    if ptxas_info:
        extra += ["-Xptxas", "-v"]
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    digest = hashlib.sha256((_headers_digest() + " ".join(extra)).encode()).hexdigest()[:12]
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, digest, extra), srcs))
    newest = max(os.path.getmtime(o) for o in objs)
    if not os.path.exists(LIB) or os.path.getmtime(LIB) < newest or _stale_link(objs):
        cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", LIB + ".tmp"] + objs + [
            "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stderr}")
        os.replace(LIB + ".tmp", LIB)
        with open(LIB + ".objs", "w") as fh:
            fh.write("\n".join(objs))
    if verbose:
        print(f"built {LIB}")
    return LIB


def _stale_link(objs: list) -> bool:
    try:
        with open(LIB + ".objs") as fh:
            return fh.read().split("\n") != objs
    except OSError:
        return True


if __name__ == "__main__":
    build(verbose=True)
