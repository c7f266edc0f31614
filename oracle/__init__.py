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
        subprocess.run(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
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
        lib.qsa_oracle_set_threads.restype = None
        lib.qsa_oracle_set_threads.argtypes = [ctypes.c_int]
        lib.qsa_oracle_e4m3_encode.restype = ctypes.c_int
        lib.qsa_oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.qsa_oracle_e2m1_encode.restype = ctypes.c_int
        lib.qsa_oracle_e2m1_encode.argtypes = [ctypes.c_float]
        lib.qsa_oracle_quantize_block.restype = None
        lib.qsa_oracle_quantize_block.argtypes = [ctypes.c_void_p, ctypes.c_float,
                                                  ctypes.c_void_p, ctypes.c_void_p]
        lib.qsa_oracle_rollback.restype = ctypes.c_int
        lib.qsa_oracle_rollback.argtypes = [ctypes.c_int] * 9 + [ctypes.c_void_p] * 9
        lib.qsa_oracle_store_kv.restype = ctypes.c_int
        lib.qsa_oracle_store_kv.argtypes = ([ctypes.c_int] * 8 + [ctypes.c_void_p] * 3 +
                                            [ctypes.c_float] * 2 + [ctypes.c_void_p] * 7)
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


def set_threads(n: int) -> None:
    """Threads the following oracle calls use (OpenMP; n >= 1)."""
    _load().qsa_oracle_set_threads(int(n))


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


# ---------------------------------------------------------------------------
# decode prologue: NVFP4 quantiser and token store
# ---------------------------------------------------------------------------

def e4m3_encode(q: float) -> int:
    """e4m3 byte nearest to fp32 ``q`` >= 0 (ties to even, saturating)."""
    return _load().qsa_oracle_e4m3_encode(float(q))


def e2m1_encode(y: float) -> int:
    """e2m1 code nearest to fp32 ``y`` (ties to even, saturating, zero as +0)."""
    return _load().qsa_oracle_e2m1_encode(float(y))


def quantize_block(x: np.ndarray, scale: float):
    """16 fp32 values -> (16 e2m1 codes, e4m3 scale byte)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.shape == (16,)
    codes = np.zeros(16, dtype=np.uint8)
    sf = np.zeros(1, dtype=np.uint8)
    _load().qsa_oracle_quantize_block(_p(x), float(scale), _p(codes), _p(sf))
    return codes, int(sf[0])


def store_kv(w: dict, new: dict) -> dict:
    """The decode prologue on host copies of the pools: returns new k_pool,
    k_sf, v_pool, v_sf and ik_pool with the step's tokens stored.  ``new``
    holds k_new / v_new (bf16 bits as uint16 [T, Hkv, D]) and ik_new (int8
    [T, Di])."""
    out = {n: np.ascontiguousarray(w[n]).copy() for n in ("k_pool", "k_sf", "v_pool", "v_sf",
                                                           "ik_pool")}
    B, R, Hkv = w["batch"], w["rows_per_req"], w["num_kv_heads"]
    st = _load().qsa_oracle_store_kv(
        B, R, Hkv, w["head_dim"], w["index_dim"], w["page_size"], w["max_blocks"],
        w["num_pages"], _p(np.ascontiguousarray(new["k_new"], dtype=np.uint16)),
        _p(np.ascontiguousarray(new["v_new"], dtype=np.uint16)),
        _p(np.ascontiguousarray(new["ik_new"], dtype=np.int8)), float(w["k_scale"]),
        float(w["v_scale"]), _p(np.ascontiguousarray(w["page_table"], dtype=np.int32)),
        _p(np.ascontiguousarray(w["seqlens"], dtype=np.int32)), _p(out["k_pool"]),
        _p(out["k_sf"]), _p(out["v_pool"]), _p(out["v_sf"]), _p(out["ik_pool"]))
    if st != 0:
        raise RuntimeError("qsa_oracle_store_kv failed (%d)" % st)
    return out


def rollback_state_bytes(w: dict) -> int:
    return (w["batch"] * w["rows_per_req"] *
            (w["num_kv_heads"] * 2 * (w["head_dim"] // 2 + w["head_dim"] // 16) + w["index_dim"]))


def rollback_gather(w: dict, pools: dict, saved: np.ndarray = None) -> np.ndarray:
    """Saved state of the slots the step's rows own (bytes the rows own no
    slot for are left as given, zero by default)."""
    saved = (np.zeros(rollback_state_bytes(w), np.uint8) if saved is None
             else np.ascontiguousarray(saved, dtype=np.uint8).copy())
    p = {n: np.ascontiguousarray(pools[n]).copy() for n in ("k_pool", "k_sf", "v_pool", "v_sf",
                                                             "ik_pool")}
    _rollback(0, w, None, p, saved)
    return saved


def rollback_restore(w: dict, pools: dict, rejected: np.ndarray, saved: np.ndarray) -> dict:
    """Pools with the rejected rows' slots set back to ``saved``."""
    p = {n: np.ascontiguousarray(pools[n]).copy() for n in ("k_pool", "k_sf", "v_pool", "v_sf",
                                                             "ik_pool")}
    _rollback(1, w, np.ascontiguousarray(rejected, dtype=np.int32), p,
              np.ascontiguousarray(saved, dtype=np.uint8).copy())
    return p


def _rollback(restore, w, rejected, p, saved):
    rej = rejected if rejected is not None else np.zeros(1, np.int32)
    st = _load().qsa_oracle_rollback(
        restore, w["batch"], w["rows_per_req"], w["num_kv_heads"], w["head_dim"],
        w["index_dim"], w["page_size"], w["max_blocks"], w["num_pages"],
        _p(np.ascontiguousarray(w["page_table"], dtype=np.int32)),
        _p(np.ascontiguousarray(w["seqlens"], dtype=np.int32)), _p(rej), _p(p["k_pool"]),
        _p(p["k_sf"]), _p(p["v_pool"]), _p(p["v_sf"]), _p(p["ik_pool"]), _p(saved))
    if st != 0:
        raise RuntimeError("qsa_oracle_rollback failed (%d)" % st)
