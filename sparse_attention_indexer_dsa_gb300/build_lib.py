"""Build the in-tree C-ABI library libdsa_idx.so for sm_103a with nvcc.

Each .cu file under csrc/ is compiled in parallel to an object in _build/,
then linked into sparse_attention_indexer_dsa_gb300/libdsa_idx.so (CUDA
runtime linked statically, no libcuda link: the TMA encoder is fetched through
the runtime's driver entry-point query).  Objects are rebuilt when a source or
header is newer.

    python -m sparse_attention_indexer_dsa_gb300.build_lib [-v]
"""
from __future__ import annotations

import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdsa_idx.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdsa_idx.so")
    return exe


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    hs += [os.path.join(ROOT, "include", h) for h in ("dsa_idx.h", "dsa_idx_testing.h")]
    return hs


def build(verbose: bool = False, force: bool = False, defines=(), build_dir: str = BUILD,
          lib_path: str = LIB) -> str:
    """Compile and link; returns the library path.  `defines` (e.g.
    DSA_PHASE_TIMERS) go to every translation unit; use a separate build_dir
    and lib_path for such variants."""
    nvcc = _nvcc()
    BUILD_, LIB_ = build_dir, lib_path
    os.makedirs(BUILD_, exist_ok=True)
    stamp = os.path.join(BUILD_, "host_arch")
    arch = platform.machine()
    if not os.path.exists(stamp) or open(stamp).read().strip() != arch:
        force = True          # objects from another host architecture are never reused
    newest_header = max(os.path.getmtime(h) for h in _headers())
    jobs = []
    for src in _sources():
        obj = os.path.join(BUILD_, os.path.basename(src)[:-3] + ".o")
        stale = force or not os.path.exists(obj) or os.path.getmtime(obj) < max(
            os.path.getmtime(src), newest_header)
        if stale:
            jobs.append((src, obj))

    def compile_one(job):
        src, obj = job
        cmd = [nvcc, *ARCH, *FLAGS, *[f"-D{d}" for d in defines], "-c", src, "-o", obj + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        os.replace(obj + ".tmp", obj)
        if verbose:
            print(f"compiled {os.path.basename(src)}", flush=True)

    if jobs:
        with ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
            list(ex.map(compile_one, jobs))
    objs = [os.path.join(BUILD_, os.path.basename(s)[:-3] + ".o") for s in _sources()]
    if jobs or force or not os.path.exists(LIB_) or os.path.getmtime(LIB_) < max(map(os.path.getmtime, objs)):
        cmd = [nvcc, *ARCH, "-shared", "-o", LIB_ + ".tmp", *objs, "-Xcompiler", "-fPIC"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(LIB_ + ".tmp", LIB_)
        if verbose:
            print(f"linked {LIB_}", flush=True)
    with open(stamp, "w") as f:
        f.write(arch)
    return LIB_


LIB_CHECKED = os.path.join(PKG, "libdsa_idx_checked.so")


def build_checked(verbose: bool = False, force: bool = False) -> str:
    """The checked build (-DDSA_CHECKED): the same entry points, plus a NaN/Inf
    scan of every score + top-k call's inputs and device bounds checks on the
    fused kernel's candidate-buffer and output writes (status word).  A
    debugging aid and the tests' stand-in for a memory checker; not the
    product library."""
    return build(verbose=verbose, force=force, defines=("DSA_CHECKED",), build_dir=BUILD + "_checked",
                 lib_path=LIB_CHECKED)


if __name__ == "__main__":
    build(verbose="-v" in sys.argv, force="-f" in sys.argv)
