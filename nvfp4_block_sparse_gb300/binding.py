"""ctypes binding of libqsa.so: the C entry points of include/qsa.h under the
same names, taking torch CUDA tensors.  Argument marshalling only -- every
step runs in the library's CUDA kernels; there is no CPU fallback, and a
missing library raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from . import build as _build

QSA_OK = 0
QSA_ERR_INVALID_ARG = 1
QSA_ERR_UNSUPPORTED = 2
QSA_ERR_CUDA = 3
QSA_ERR_WORKSPACE = 4
QSA_ERR_DEVICE_TIMEOUT = 5

# Every symbol include/qsa.h declares.
EXPORTS = (
    "qsa_status_string",
    "qsa_index_scores",
    "qsa_select_topk",
    "qsa_sparse_decode_workspace_bytes",
    "qsa_sparse_decode_workspace_bytes_ex",
    "qsa_workspace_init",
    "qsa_sparse_decode",
    "qsa_sparse_decode_ex",
    "qsa_sparse_decode_noalloc",
    "qsa_sparse_decode_noalloc_status",
    "qsa_debug_set_wait_ns",
    "qsa_debug_bounds_status",
    "qsa_workspace_status",
    "qsa_store_kv_tokens",
    "qsa_select_sparse_decode",
    "qsa_select_sparse_decode_fused",
    "qsa_rollback_state_bytes",
    "qsa_rollback_gather",
    "qsa_rollback_restore",
    "qsa_sparse_prefill_workspace_bytes",
    "qsa_sparse_prefill",
)


class QsaError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__("%s failed: %s (status %d)" % (fn, msg, status))
        self.status = status


class qsa_geom_t(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "batch", "rows_per_req", "num_q_heads", "num_kv_heads", "head_dim",
        "index_dim", "page_size", "max_blocks", "num_pages")]


_lib = None
_vp = ctypes.c_void_p


def bounds_checked() -> bool:
    """True when QSA_BOUNDS_CHECKED=1 selects the bounds-checked library."""
    return os.environ.get("QSA_BOUNDS_CHECKED", "") == "1"


def library_path() -> str:
    return _build.BOUNDS_LIB if bounds_checked() else _build.LIB


def load(build_if_missing: bool = False):
    """Loads libqsa.so, or libqsa_bounds.so under QSA_BOUNDS_CHECKED=1
    (building first only when asked)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise ImportError("%s is not built (run __graft_entry__.build() or "
                              "python -m nvfp4_block_sparse_gb300.build)" % os.path.basename(path))
        _build.build()
    lib = ctypes.CDLL(path)
    G = ctypes.POINTER(qsa_geom_t)
    st = ctypes.c_int
    lib.qsa_status_string.restype = ctypes.c_char_p
    lib.qsa_status_string.argtypes = [st]
    lib.qsa_index_scores.restype = st
    lib.qsa_index_scores.argtypes = [G, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.qsa_select_topk.restype = st
    lib.qsa_select_topk.argtypes = [G, _vp, _vp, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp]
    lib.qsa_sparse_decode_workspace_bytes.restype = ctypes.c_size_t
    lib.qsa_sparse_decode_workspace_bytes.argtypes = [G, ctypes.c_int]
    lib.qsa_sparse_decode_workspace_bytes_ex.restype = ctypes.c_size_t
    lib.qsa_sparse_decode_workspace_bytes_ex.argtypes = [G, ctypes.c_int, ctypes.c_int]
    lib.qsa_workspace_init.restype = st
    lib.qsa_workspace_init.argtypes = [_vp, ctypes.c_size_t, _vp]
    dec = [G, _vp, _vp, _vp, _vp, _vp, ctypes.c_float, ctypes.c_float, ctypes.c_float,
           _vp, _vp, _vp, ctypes.c_int, _vp, _vp, _vp, ctypes.c_size_t]
    lib.qsa_sparse_decode.restype = st
    lib.qsa_sparse_decode.argtypes = dec + [_vp]
    lib.qsa_sparse_decode_ex.restype = st
    lib.qsa_sparse_decode_ex.argtypes = dec + [ctypes.c_int, _vp]
    lib.qsa_select_sparse_decode_fused.restype = ctypes.c_int
    lib.qsa_select_sparse_decode_fused.argtypes = [G]
    lib.qsa_select_sparse_decode.restype = st
    lib.qsa_select_sparse_decode.argtypes = [G, _vp, ctypes.c_int, _vp, _vp, _vp, _vp, _vp,
                                             ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                             _vp, _vp, ctypes.c_int, _vp, _vp, _vp, _vp, _vp,
                                             ctypes.c_size_t, ctypes.c_int, _vp]
    lib.qsa_sparse_decode_noalloc.restype = st
    lib.qsa_sparse_decode_noalloc.argtypes = [G, _vp, _vp, _vp, _vp, _vp, ctypes.c_float,
                                              ctypes.c_float, ctypes.c_float, _vp, _vp, _vp,
                                              ctypes.c_int, _vp, _vp, _vp]
    lib.qsa_store_kv_tokens.restype = st
    lib.qsa_store_kv_tokens.argtypes = [G, _vp, _vp, _vp, ctypes.c_float, ctypes.c_float, _vp,
                                        _vp, _vp, _vp, _vp, _vp, _vp, _vp]
    lib.qsa_rollback_state_bytes.restype = ctypes.c_size_t
    lib.qsa_rollback_state_bytes.argtypes = [G]
    lib.qsa_rollback_gather.restype = st
    lib.qsa_rollback_gather.argtypes = [G] + [_vp] * 9
    lib.qsa_rollback_restore.restype = st
    lib.qsa_rollback_restore.argtypes = [G] + [_vp] * 10
    lib.qsa_sparse_prefill_workspace_bytes.restype = ctypes.c_size_t
    lib.qsa_sparse_prefill_workspace_bytes.argtypes = [G, ctypes.c_int]
    lib.qsa_sparse_prefill.restype = st
    lib.qsa_sparse_prefill.argtypes = dec + [_vp]
    lib.qsa_sparse_decode_noalloc_status.restype = st
    lib.qsa_sparse_decode_noalloc_status.argtypes = [ctypes.POINTER(ctypes.c_int), _vp]
    lib.qsa_debug_set_wait_ns.restype = None
    lib.qsa_debug_set_wait_ns.argtypes = [ctypes.c_ulonglong]
    lib.qsa_debug_bounds_status.restype = ctypes.c_int
    lib.qsa_debug_bounds_status.argtypes = []
    lib.qsa_workspace_status.restype = st
    lib.qsa_workspace_status.argtypes = [_vp, ctypes.POINTER(ctypes.c_int), _vp]
    _lib = lib
    return lib


def make_geom(**kw) -> qsa_geom_t:
    return qsa_geom_t(*[int(kw[n]) for n, _ in qsa_geom_t._fields_])


def _geom(geom) -> qsa_geom_t:
    return geom if isinstance(geom, qsa_geom_t) else make_geom(**geom)


def _check(fn: str, status: int):
    if status != QSA_OK:
        raise QsaError(fn, status, load().qsa_status_string(status).decode())


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: torch.Tensor, dtype, name: str) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t.data_ptr()


def qsa_status_string(status: int) -> str:
    return load().qsa_status_string(int(status)).decode()


def qsa_index_scores(geom, iq, ik_pool, page_table, seqlens, scores, stream=None):
    g = _geom(geom)
    _check("qsa_index_scores", load().qsa_index_scores(
        ctypes.byref(g), _ptr(iq, torch.int8, "iq"), _ptr(ik_pool, torch.int8, "ik_pool"),
        _ptr(page_table, torch.int32, "page_table"), _ptr(seqlens, torch.int32, "seqlens"),
        _ptr(scores, torch.int32, "scores"), _stream(stream)))


def qsa_store_kv_tokens(geom, k_new, v_new, ik_new, k_scale, v_scale, page_table, seqlens,
                        k_pool, k_sf, v_pool, v_sf, ik_pool, stream=None):
    g = _geom(geom)
    _check("qsa_store_kv_tokens", load().qsa_store_kv_tokens(
        ctypes.byref(g), _ptr(k_new, torch.bfloat16, "k_new"), _ptr(v_new, torch.bfloat16, "v_new"),
        _ptr(ik_new, torch.int8, "ik_new"), float(k_scale), float(v_scale),
        _ptr(page_table, torch.int32, "page_table"), _ptr(seqlens, torch.int32, "seqlens"),
        _ptr(k_pool, torch.uint8, "k_pool"), _ptr(k_sf, torch.uint8, "k_sf"),
        _ptr(v_pool, torch.uint8, "v_pool"), _ptr(v_sf, torch.uint8, "v_sf"),
        _ptr(ik_pool, torch.int8, "ik_pool"), _stream(stream)))


def qsa_rollback_state_bytes(geom) -> int:
    g = _geom(geom)
    return int(load().qsa_rollback_state_bytes(ctypes.byref(g)))


def qsa_rollback_gather(geom, page_table, seqlens, k_pool, k_sf, v_pool, v_sf, ik_pool, saved,
                        stream=None):
    g = _geom(geom)
    _check("qsa_rollback_gather", load().qsa_rollback_gather(
        ctypes.byref(g), _ptr(page_table, torch.int32, "page_table"),
        _ptr(seqlens, torch.int32, "seqlens"), _ptr(k_pool, torch.uint8, "k_pool"),
        _ptr(k_sf, torch.uint8, "k_sf"), _ptr(v_pool, torch.uint8, "v_pool"),
        _ptr(v_sf, torch.uint8, "v_sf"), _ptr(ik_pool, torch.int8, "ik_pool"),
        _ptr(saved, torch.uint8, "saved"), _stream(stream)))


def qsa_rollback_restore(geom, page_table, seqlens, rejected, saved, k_pool, k_sf, v_pool, v_sf,
                         ik_pool, stream=None):
    g = _geom(geom)
    _check("qsa_rollback_restore", load().qsa_rollback_restore(
        ctypes.byref(g), _ptr(page_table, torch.int32, "page_table"),
        _ptr(seqlens, torch.int32, "seqlens"), _ptr(rejected, torch.int32, "rejected"),
        _ptr(saved, torch.uint8, "saved"), _ptr(k_pool, torch.uint8, "k_pool"),
        _ptr(k_sf, torch.uint8, "k_sf"), _ptr(v_pool, torch.uint8, "v_pool"),
        _ptr(v_sf, torch.uint8, "v_sf"), _ptr(ik_pool, torch.int8, "ik_pool"), _stream(stream)))


def qsa_select_sparse_decode_fused(geom) -> bool:
    g = _geom(geom)
    return bool(load().qsa_select_sparse_decode_fused(ctypes.byref(g)))


def qsa_select_sparse_decode(geom, scores, window, q, k_pool, k_sf, v_pool, v_sf, k_scale,
                             v_scale, sm_scale, page_table, seqlens, k, sel, nsel, out, lse,
                             workspace, num_splits=0, stream=None):
    g = _geom(geom)
    _check("qsa_select_sparse_decode", load().qsa_select_sparse_decode(
        ctypes.byref(g), _ptr(scores, torch.int32, "scores"), int(window),
        _ptr(q, torch.bfloat16, "q"), _ptr(k_pool, torch.uint8, "k_pool"),
        _ptr(k_sf, torch.uint8, "k_sf"), _ptr(v_pool, torch.uint8, "v_pool"),
        _ptr(v_sf, torch.uint8, "v_sf"), float(k_scale), float(v_scale), float(sm_scale),
        _ptr(page_table, torch.int32, "page_table"), _ptr(seqlens, torch.int32, "seqlens"),
        int(k), _ptr(sel, torch.int32, "sel"), _ptr(nsel, torch.int32, "nsel"),
        _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), int(num_splits),
        _stream(stream)))


def qsa_select_topk(geom, scores, seqlens, k, window, sel, nsel, stream=None):
    g = _geom(geom)
    _check("qsa_select_topk", load().qsa_select_topk(
        ctypes.byref(g), _ptr(scores, torch.int32, "scores"),
        _ptr(seqlens, torch.int32, "seqlens"), int(k), int(window),
        _ptr(sel, torch.int32, "sel"), _ptr(nsel, torch.int32, "nsel"), _stream(stream)))


def qsa_sparse_decode_workspace_bytes(geom, k) -> int:
    return int(load().qsa_sparse_decode_workspace_bytes(ctypes.byref(_geom(geom)), int(k)))


def qsa_sparse_decode_workspace_bytes_ex(geom, k, num_splits) -> int:
    return int(load().qsa_sparse_decode_workspace_bytes_ex(ctypes.byref(_geom(geom)), int(k),
                                                            int(num_splits)))


def qsa_workspace_init(workspace, stream=None):
    _check("qsa_workspace_init", load().qsa_workspace_init(
        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)))


def _decode_args(geom, q, k_pool, k_sf, v_pool, v_sf, k_scale, v_scale, sm_scale, page_table,
                 seqlens, sel, k, out, lse, workspace):
    g = _geom(geom)
    return [ctypes.byref(g), _ptr(q, torch.bfloat16, "q"), _ptr(k_pool, torch.uint8, "k_pool"),
            _ptr(k_sf, torch.uint8, "k_sf"), _ptr(v_pool, torch.uint8, "v_pool"),
            _ptr(v_sf, torch.uint8, "v_sf"), float(k_scale), float(v_scale), float(sm_scale),
            _ptr(page_table, torch.int32, "page_table"), _ptr(seqlens, torch.int32, "seqlens"),
            _ptr(sel, torch.int32, "sel"), int(k), _ptr(out, torch.bfloat16, "out"),
            _ptr(lse, torch.float32, "lse"), _ptr(workspace, torch.uint8, "workspace"),
            workspace.numel()], g


def qsa_sparse_decode(geom, q, k_pool, k_sf, v_pool, v_sf, k_scale, v_scale, sm_scale,
                      page_table, seqlens, sel, k, out, lse, workspace, stream=None):
    args, _g = _decode_args(geom, q, k_pool, k_sf, v_pool, v_sf, k_scale, v_scale, sm_scale,
                            page_table, seqlens, sel, k, out, lse, workspace)
    _check("qsa_sparse_decode", load().qsa_sparse_decode(*args, _stream(stream)))


def qsa_sparse_decode_ex(geom, q, k_pool, k_sf, v_pool, v_sf, k_scale, v_scale, sm_scale,
                         page_table, seqlens, sel, k, out, lse, workspace, num_splits,
                         stream=None):
    args, _g = _decode_args(geom, q, k_pool, k_sf, v_pool, v_sf, k_scale, v_scale, sm_scale,
                            page_table, seqlens, sel, k, out, lse, workspace)
    _check("qsa_sparse_decode_ex",
           load().qsa_sparse_decode_ex(*args, int(num_splits), _stream(stream)))


def qsa_sparse_prefill_workspace_bytes(geom, k) -> int:
    g = _geom(geom)
    return int(load().qsa_sparse_prefill_workspace_bytes(ctypes.byref(g), int(k)))


def qsa_sparse_prefill(geom, q, k_pool, k_sf, v_pool, v_sf, k_scale, v_scale, sm_scale,
                       page_table, seqlens, sel, k, out, lse, workspace, stream=None):
    args, _g = _decode_args(geom, q, k_pool, k_sf, v_pool, v_sf, k_scale, v_scale, sm_scale,
                            page_table, seqlens, sel, k, out, lse, workspace)
    _check("qsa_sparse_prefill", load().qsa_sparse_prefill(*args, _stream(stream)))


def qsa_sparse_decode_noalloc(geom, q, k_pool, k_sf, v_pool, v_sf, k_scale, v_scale, sm_scale,
                              page_table, seqlens, sel, k, out, lse, stream=None):
    """qsa_sparse_decode without a workspace, for callers that cannot
    allocate device memory: the library's built-in scratch array is used
    instead (shared by every call on the device, so overlapping calls race)."""
    g = _geom(geom)
    _check("qsa_sparse_decode_noalloc", load().qsa_sparse_decode_noalloc(
        ctypes.byref(g), _ptr(q, torch.bfloat16, "q"), _ptr(k_pool, torch.uint8, "k_pool"),
        _ptr(k_sf, torch.uint8, "k_sf"), _ptr(v_pool, torch.uint8, "v_pool"),
        _ptr(v_sf, torch.uint8, "v_sf"), float(k_scale), float(v_scale), float(sm_scale),
        _ptr(page_table, torch.int32, "page_table"), _ptr(seqlens, torch.int32, "seqlens"),
        _ptr(sel, torch.int32, "sel"), int(k), _ptr(out, torch.bfloat16, "out"),
        _ptr(lse, torch.float32, "lse"), _stream(stream)))


def qsa_sparse_decode_noalloc_status(stream=None) -> int:
    """Reads and clears the built-in scratch array's status word on the
    current device: 0, or the code of a bounded device wait that gave up in a
    qsa_sparse_decode_noalloc call since the previous query."""
    code = ctypes.c_int(0)
    st = load().qsa_sparse_decode_noalloc_status(ctypes.byref(code), _stream(stream))
    if st not in (QSA_OK, QSA_ERR_DEVICE_TIMEOUT):
        _check("qsa_sparse_decode_noalloc_status", st)
    return int(code.value)


def qsa_debug_bounds_status() -> int:
    """First failed bounds-check code since the last call (clearing them), 0
    when every check held, -1 when the loaded library has no checks."""
    return int(load().qsa_debug_bounds_status())


def qsa_debug_set_wait_ns(ns: int) -> None:
    """Diagnostics: bound of the head_dim-128 decode kernel's copy waits in ns
    (0 restores the 2 s default)."""
    load().qsa_debug_set_wait_ns(int(ns))


def qsa_workspace_status(workspace, stream=None) -> int:
    code = ctypes.c_int(0)
    st = load().qsa_workspace_status(_ptr(workspace, torch.uint8, "workspace"),
                                     ctypes.byref(code), _stream(stream))
    if st not in (QSA_OK, QSA_ERR_DEVICE_TIMEOUT):
        _check("qsa_workspace_status", st)
    return int(code.value)
