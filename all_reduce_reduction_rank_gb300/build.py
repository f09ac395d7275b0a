"""Build libar_gb300.so in-tree: nvcc for sm_103a only, one object per
source compiled in parallel, linked against the shared CUDA runtime (so a
process that already loaded libcudart.so.13, e.g. through torch, shares one
runtime with the library).  ``python -m all_reduce_reduction_rank_gb300.build``
or ``__graft_entry__.build()`` runs it."""

from __future__ import annotations

import os
import pathlib
import shutil
import subprocess
import sys

PKG = pathlib.Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
INCLUDE = ROOT / "include"
OUT_DIR = PKG / "_build"
LIB = PKG / "libar_gb300.so"
SOURCES = ["api.cu", "one_shot.cu", "two_shot.cu", "ring.cu", "ll.cu", "ring_noalloc.cu", "rmsnorm.cu",
           "one_shot_modes.cu", "tree.cu", "ring_persistent.cu", "ring_cluster.cu", "ring_fused.cu"]
HEADERS = ["common.cuh", "internal.h", "bulk.cuh", "lines.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    *ARCH, "-O3", "-lineinfo", "-std=c++17", "--fmad=false",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
    "-Xptxas", "-v", "-I", str(INCLUDE), "-I", str(CSRC),
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def _stale(target: pathlib.Path, deps: list[pathlib.Path]) -> bool:
    if not target.exists():
        return True
    t = target.stat().st_mtime
    return any(d.stat().st_mtime > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> pathlib.Path:
    """Compile every CUDA source for sm_103a and link libar_gb300.so."""
    OUT_DIR.mkdir(exist_ok=True)
    exe = nvcc()
    headers = [CSRC / h for h in HEADERS] + [INCLUDE / "ar.h"]
    jobs = []
    objs = []
    for src in SOURCES:
        s = CSRC / src
        o = OUT_DIR / (src + ".o")
        objs.append(o)
        if force or _stale(o, [s, *headers]):
            log = open(OUT_DIR / (src + ".ptxas.log"), "w")
            cmd = [exe, *NVCC_FLAGS, "-c", str(s), "-o", str(o)]
            jobs.append((src, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log))
    failed = []
    for src, p, log in jobs:
        p.wait()
        log.close()
        if p.returncode != 0:
            failed.append(src)
    if failed:
        for src in failed:
            sys.stderr.write((OUT_DIR / (src + ".ptxas.log")).read_text()[-4000:])
        raise RuntimeError(f"nvcc failed on {failed}")
    if force or _stale(LIB, objs):
        tmp = LIB.with_suffix(f".so.{os.getpid()}.tmp")
        cuda_lib = pathlib.Path(exe).resolve().parent.parent / "lib64"
        cmd = [exe, *ARCH, "-shared", "-cudart", "shared", "-o", str(tmp), *map(str, objs),
               "-Xlinker", f"-rpath,{cuda_lib}"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB}")
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
