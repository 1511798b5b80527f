"""Build libqv.so in-tree with nvcc for sm_103a.

    python -m quantized_verification_gb300.build      # or build() from Python

Each CUDA translation unit under ``csrc/`` is compiled in parallel into
``_build/``, then linked into ``quantized_verification_gb300/libqv.so``.
No fast-math and no flush-to-zero: the kernels rely on IEEE binary32
division and round-to-nearest-even conversions.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libqv.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
    "-Xcompiler", "-fvisibility=hidden",
    "--ftz=false", "--prec-div=true", "--prec-sqrt=true",
    "-I", INCLUDE, "-I", CSRC,
]
# Translation units whose floating point results are checked against a
# tolerance (attention, the logit-fidelity diagnostic) may contract a*b+c
# into one fused multiply-add; every other unit computes results that must
# equal the oracle's bit for bit, so no expression there may be contracted
# (explicit fused operations, where the definition has one, are written as
# such).
FMA_CONTRACTION_OK = {"k_attn.cu", "k_fidelity.cu"}


def flags_for(src: str) -> list[str]:
    return NVCC_FLAGS + ["--fmad=true" if os.path.basename(src) in FMA_CONTRACTION_OK else "--fmad=false"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers_mtime() -> float:
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs.append(os.path.join(INCLUDE, "qv.h"))
    return max(os.path.getmtime(h) for h in hs)


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          build_dir: str = BUILD, out: str = LIB) -> str:
    """Compile and link libqv.so (or `out`); returns its path. Skips up-to-date
    objects. `extra_flags` (e.g. -G for a debug build) go to every nvcc call."""
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    hdr = _headers_mtime()
    extra = list(extra_flags or [])
    jobs = []
    for src in sources():
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        stale = (force or not os.path.exists(obj)
                 or os.path.getmtime(obj) < max(os.path.getmtime(src), hdr))
        jobs.append((src, obj, stale))

    def compile_one(job):
        src, obj, stale = job
        if not stale:
            return None
        cmd = [nvcc, *flags_for(src), *extra, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return r.stderr

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for msg in ex.map(compile_one, jobs):
            if msg and verbose:
                print(msg, file=sys.stderr)

    objs = [j[1] for j in jobs]
    if force or not os.path.exists(out) or any(os.path.getmtime(o) > os.path.getmtime(out) for o in objs):
        tmp = out + f".tmp{os.getpid()}"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
