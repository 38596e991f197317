"""Build libgqa_attn.so in-tree with nvcc for sm_103a (one -gencode, parallel
translation units, no cmake), and its debug twin libgqa_attn_checks.so (the
same sources with -DGQA_CHECKS: device-side checks of seg and of the kernels'
indices, reported through the workspace status word). Used by
``__graft_entry__.build()`` and by the binding when a library is missing or
older than its sources."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgqa_attn.so")
LIB_CHECKS = os.path.join(PKG, "libgqa_attn_checks.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-Xptxas", "-v", "--expt-relaxed-constexpr"]
# variant -> (library, object directory, extra flags)
VARIANTS = {"release": (LIB, BUILD, []),
            "checks": (LIB_CHECKS, os.path.join(BUILD, "checks"), ["-DGQA_CHECKS"])}


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libgqa_attn.so")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps() -> list[str]:
    out = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return out + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]


def up_to_date(variant: str = "release") -> bool:
    lib = VARIANTS[variant][0]
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _compile(nvcc: str, src: str, objdir: str, extra: list[str]) -> tuple[str, str]:
    obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc, *NVCC_FLAGS, *extra, "-I", INCLUDE, "-c", src, "-o", obj]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{p.stdout}\n{p.stderr}")
    with open(obj + ".ptxas.txt", "w") as f:   # register / spill / smem report
        f.write(p.stderr)
    return obj, p.stderr


def _link(nvcc: str, lib: str, objs: list[str]) -> None:
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stdout}\n{p.stderr}")
    os.replace(tmp, lib)


def build(force: bool = False, verbose: bool = False, variants=("release", "checks")) -> str:
    """Build the given variants (both by default; only those out of date unless
    force) in one pool of parallel nvcc jobs. Returns the release library's path."""
    todo = [v for v in variants if force or not up_to_date(v)]
    if not todo:
        return LIB
    nvcc = _nvcc()
    srcs = sources()
    jobs = []
    for v in todo:
        os.makedirs(VARIANTS[v][1], exist_ok=True)
        jobs += [(v, s) for s in srcs]
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        futs = [(v, ex.submit(_compile, nvcc, s, VARIANTS[v][1], VARIANTS[v][2])) for v, s in jobs]
        objs = {v: [] for v in todo}
        for v, f in futs:
            objs[v].append(f.result()[0])
    for v in todo:
        _link(nvcc, VARIANTS[v][0], objs[v])
        if verbose:
            print(f"built {VARIANTS[v][0]}", file=sys.stderr)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
