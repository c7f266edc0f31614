"""CPU oracle for QSA block-sparse GQA decode / verify over an NVFP4 paged KV
cache: a thin ctypes wrapper around ``qsa_oracle.c`` (plain C, fp64).

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg import this package.  It imports nothing from the CUDA
library's package, and the library never imports it.

Every function takes host numpy arrays in the layouts of the workload
generator and returns host numpy arrays.  ``rows`` restricts the work to a
half-open range of query rows (for sampled checks on large workloads); rows
outside it are left at their initial fill.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qsa_oracle.c")
_LIB = os.path.join(_HERE, "libqsa_oracle.so")
_lib = None

INT32_MIN = np.iinfo(np.int32).min


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (OpenMP, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.run(["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.qsa_oracle_e2m1.restype = ctypes.c_double
        lib.qsa_oracle_e2m1.argtypes = [ctypes.c_int]
        lib.qsa_oracle_e4m3.restype = ctypes.c_double
        lib.qsa_oracle_e4m3.argtypes = [ctypes.c_int]
        lib.qsa_oracle_num_threads.restype = ctypes.c_int
        for name in ("qsa_oracle_index_scores", "qsa_oracle_select",
                     "qsa_oracle_attention"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(_load().qsa_oracle_num_threads())


def e2m1(code: int) -> float:
    return float(_load().qsa_oracle_e2m1(int(code)))


def e4m3(byte: int) -> float:
    return float(_load().qsa_oracle_e4m3(int(byte)))


def _geom(w):
    return (int(w["batch"]), int(w["rows_per_req"]), int(w["num_q_heads"]),
            int(w["num_kv_heads"]), int(w["head_dim"]), int(w["index_dim"]),
            int(w["page_size"]), int(w["max_blocks"]), int(w["num_pages"]))


def _rows(w, rows):
    T = int(w["batch"]) * int(w["rows_per_req"])
    if rows is None:
        return 0, T
    return int(rows[0]), int(rows[1])


def index_scores(w: dict, rows=None) -> np.ndarray:
    """int32 [T, MB] block scores (INT32_MIN for invalid / invisible blocks)."""
    B, R, Hq, Hkv, D, Di, P, MB, NP = _geom(w)
    r0, r1 = _rows(w, rows)
    iq = np.ascontiguousarray(w["iq"], dtype=np.int8)
    ik = np.ascontiguousarray(w["ik_pool"], dtype=np.int8)
    pt = np.ascontiguousarray(w["page_table"], dtype=np.int32)
    sl = np.ascontiguousarray(w["seqlens"], dtype=np.int32)
    out = np.zeros((B * R, MB), dtype=np.int32)
    rc = _load().qsa_oracle_index_scores(B, R, Hq, Di, P, MB, NP, _p(iq), _p(ik),
                                         _p(pt), _p(sl), r0, r1, _p(out))
    if rc != 0:
        raise RuntimeError("oracle index scores out of int32 range")
    return out


def select(w: dict, scores: np.ndarray, rows=None):
    """(sel int32 [T, k], nsel int32 [T]) canonical selection of ``scores``."""
    B, R, Hq, Hkv, D, Di, P, MB, NP = _geom(w)
    k, W = int(w["k"]), int(w["window"])
    r0, r1 = _rows(w, rows)
    sc = np.ascontiguousarray(scores, dtype=np.int32)
    assert sc.shape == (B * R, MB)
    sl = np.ascontiguousarray(w["seqlens"], dtype=np.int32)
    sel = np.full((B * R, k), -1, dtype=np.int32)
    nsel = np.zeros((B * R,), dtype=np.int32)
    rc = _load().qsa_oracle_select(B, R, P, MB, _p(sc), _p(sl), k, W, r0, r1,
                                   _p(sel), _p(nsel))
    if rc != 0:
        raise RuntimeError("oracle select failed (%d)" % rc)
    return sel, nsel


def attention(w: dict, sel: np.ndarray, rows=None):
    """(out float64 [T, Hq, D], lse float64 [T, Hq]) over the selected blocks."""
    B, R, Hq, Hkv, D, Di, P, MB, NP = _geom(w)
    r0, r1 = _rows(w, rows)
    k = int(sel.shape[1])
    q = np.ascontiguousarray(w["q"], dtype=np.uint16)
    kp = np.ascontiguousarray(w["k_pool"], dtype=np.uint8)
    ks = np.ascontiguousarray(w["k_sf"], dtype=np.uint8)
    vp = np.ascontiguousarray(w["v_pool"], dtype=np.uint8)
    vs = np.ascontiguousarray(w["v_sf"], dtype=np.uint8)
    pt = np.ascontiguousarray(w["page_table"], dtype=np.int32)
    sl = np.ascontiguousarray(w["seqlens"], dtype=np.int32)
    se = np.ascontiguousarray(sel, dtype=np.int32)
    out = np.zeros((B * R, Hq, D), dtype=np.float64)
    lse = np.zeros((B * R, Hq), dtype=np.float64)
    lib = _load()
    rc = lib.qsa_oracle_attention(
        B, R, Hq, Hkv, D, P, MB, NP, _p(q), _p(kp), _p(ks), _p(vp), _p(vs),
        ctypes.c_double(w["k_scale"]), ctypes.c_double(w["v_scale"]),
        ctypes.c_double(w["sm_scale"]), _p(pt), _p(sl), _p(se), k, r0, r1,
        _p(out), _p(lse))
    if rc != 0:
        raise RuntimeError("oracle attention failed (%d)" % rc)
    return out, lse


def step(w: dict, rows=None):
    """The whole path: scores -> selection -> attention."""
    sc = index_scores(w, rows)
    sel, nsel = select(w, sc, rows)
    out, lse = attention(w, sel, rows)
    return dict(scores=sc, sel=sel, nsel=nsel, out=out, lse=lse)
