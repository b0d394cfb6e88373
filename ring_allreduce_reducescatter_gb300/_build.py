"""Build libringred.so in-tree with nvcc for sm_103a (GB300).

Each translation unit under csrc/ compiles in parallel to an object under
_build/ (rr_inst_one.cu once for every collective / storage / wire
combination, INSTANCES), then nvcc links the shared library next to this
file.  No fast-math
and no FMA contraction: the kernels' results are defined bit for bit.

A build is reused only when the digest recorded beside it (under _build/)
matches the digest of what it was built from: the contents of every file under
csrc/ and include/, the compiler command line, the nvcc binary and the host
machine type.  A library copied in from elsewhere, or one older or newer than
its sources by file time, is rebuilt rather than trusted.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import platform
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libringred.so")
# the same library with device-side bounds checks (RR_DEBUG_CHECKS)
DEBUG_LIB = os.path.join(PKG, "libringred_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-fmad=false",
         "-I", INCLUDE, "-I", CSRC]


# (collective, storage format, wire format) combinations, each compiled from
# rr_inst_one.cu into an object of its own (values of rr_params.h's kOp* / kF*)
OPS = {"allreduce": 0, "reduce_scatter": 1, "allgather": 2}
FMTS = {"f32": 0, "f16": 1, "bf16": 2}
FOLD_PAIRS = (("f32", "f32"), ("f16", "f16"), ("bf16", "bf16"), ("f32", "bf16"), ("f32", "f16"), ("f16", "f32"),
              ("bf16", "f32"))
INSTANCES = ([(op, dt, wt) for op in ("allreduce", "reduce_scatter") for dt, wt in FOLD_PAIRS] +
             [("allgather", dt, dt) for dt in ("f32", "f16", "bf16")])
INST_ONE = "rr_inst_one.cu"


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def source_digest(cc: str, flags) -> str:
    """Digest of everything the library is built from (see the module docstring)."""
    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h")))
    for f in files:
        h.update(os.path.relpath(f, ROOT).encode() + b"\0")
        with open(f, "rb") as fh:
            h.update(fh.read())
        h.update(b"\0")
    h.update(" ".join([os.path.realpath(cc), *ARCH, *flags]).encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def _digest_path(lib: str) -> str:
    return os.path.join(BUILD, os.path.basename(lib) + ".digest")


def _recorded_digest(lib: str):
    try:
        with open(_digest_path(lib)) as f:
            return f.read().strip()
    except OSError:
        return None


def build(force: bool = False, verbose_ptxas: bool = False, debug: bool = False) -> str:
    """Build libringred.so (or, debug=True, libringred_debug.so with every
    device access of a rank buffer checked against its extent) unless the
    recorded digest shows it is current.  Returns the library's path."""
    cc = nvcc()
    lib = DEBUG_LIB if debug else LIB
    flags = FLAGS + (["-DRR_DEBUG_CHECKS=1"] if debug else [])
    objdir = os.path.join(BUILD, "debug") if debug else BUILD
    digest = source_digest(cc, flags)
    if not force and os.path.exists(lib) and _recorded_digest(lib) == digest:
        return lib
    os.makedirs(objdir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []
    # (source, object name, defines): every .cu once, rr_inst_one.cu once per instance
    jobs = [(src, os.path.basename(src), []) for src in sorted(glob.glob(os.path.join(CSRC, "*.cu")))
            if os.path.basename(src) != INST_ONE]
    for op, dt, wt in INSTANCES:
        jobs.append((os.path.join(CSRC, INST_ONE), f"rr_inst_{op}_{dt}_{wt}.cu",
                     [f"-DRR_INST_OP={OPS[op]}", f"-DRR_INST_DT={FMTS[dt]}", f"-DRR_INST_WT={FMTS[wt]}"]))
    # the longest units first, so they start at once
    jobs.sort(key=lambda j: j[0].endswith(INST_ONE), reverse=True)

    def compile_one(job):
        src, name, defs = job
        obj = os.path.join(objdir, name + ".o")
        cmd = [cc, *ARCH, *flags, *defs, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {name}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    workers = max(1, min(len(jobs), (os.cpu_count() or 1) + 2))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        results = list(ex.map(compile_one, jobs))
    if verbose_ptxas:
        for _, log in results:
            print(log)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(_digest_path(lib) + f".tmp{os.getpid()}", "w") as f:
        f.write(digest + "\n")
    os.replace(_digest_path(lib) + f".tmp{os.getpid()}", _digest_path(lib))
    return lib


if __name__ == "__main__":
    import sys

    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv, debug="--debug" in sys.argv))
