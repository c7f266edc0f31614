"""Builds libqsa.so in-tree for sm_103a with nvcc (one -gencode, translation
units compiled in parallel, no cmake), and its bounds-checked twin
libqsa_bounds.so (the same sources with QSA_DEBUG_BOUNDS defined), which the
binding loads instead when QSA_BOUNDS_CHECKED=1 is set in the environment."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libqsa.so")
BOUNDS_BUILD = os.path.join(HERE, "_build_bounds")
BOUNDS_LIB = os.path.join(HERE, "libqsa_bounds.so")
SOURCES = ["qsa_api.cu", "qsa_index_scores.cu", "qsa_select_topk.cu", "qsa_sparse_decode.cu",
           "qsa_attend.cu",
           "qsa_sparse_decode_noalloc.cu", "qsa_store_tokens.cu", "qsa_rollback.cu",
           "qsa_sparse_prefill.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++20", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the QSA library needs the CUDA 13 toolkit")
    return cand


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def _variants(bounds_checked):
    """(object dir, library, extra flags) of each library to build."""
    v = [(BUILD, LIB, [])]
    if bounds_checked:
        v.append((BOUNDS_BUILD, BOUNDS_LIB, ["-DQSA_DEBUG_BOUNDS"]))
    return v


def build(force: bool = False, verbose: bool = False, bounds_checked: bool = True) -> str:
    """Compiles every CUDA source and links libqsa.so (and, unless
    bounds_checked is False, libqsa_bounds.so, in the same parallel pass);
    returns the path of libqsa.so."""
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")]
    headers.append(os.path.join(os.path.dirname(HERE), "include", "qsa.h"))
    variants = _variants(bounds_checked)
    jobs = []
    for objdir, _, extra in variants:
        os.makedirs(objdir, exist_ok=True)
        for src in SOURCES:
            s = os.path.join(CSRC, src)
            o = os.path.join(objdir, src.replace(".cu", ".o"))
            if force or _stale(o, [s] + headers):
                jobs.append([nvcc, *ARCH, *FLAGS, *extra, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
        if verbose and r.stderr:
            print(r.stderr)

    # The largest translation units first, so the pass ends with small ones.
    jobs.sort(key=lambda cmd: -os.path.getsize(cmd[cmd.index("-c") + 1]))
    workers = max(1, min(len(jobs), os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(run, jobs))
    for objdir, lib, _ in variants:
        objs = [os.path.join(objdir, s.replace(".cu", ".o")) for s in SOURCES]
        if force or _stale(lib, objs):
            tmp = lib + ".tmp%d" % os.getpid()
            run([nvcc, *ARCH, "-shared", "-cudart=shared", "-o", tmp, *objs])
            os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
