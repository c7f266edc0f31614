"""C-ABI checks that need no GPU: the library loads, exports every function
include/qsa.h declares, and its host-side validation rejects bad arguments
before touching the device."""
import ctypes
import os
import re

import pytest

import nvfp4_block_sparse_gb300 as qsa
from nvfp4_block_sparse_gb300 import binding

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "qsa.h")


@pytest.fixture(scope="module")
def lib():
    return qsa.load(build_if_missing=True)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qsa_[a-z_0-9]+)\s*\(", text)))


def test_header_declarations_match_binding():
    assert declared_functions() == sorted(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_bounds_checked_library_exports_every_declared_symbol(lib):
    # libqsa_bounds.so (built beside libqsa.so) has the same C ABI; the normal
    # library answers the bounds query with -1 (no checks compiled in) without
    # touching a device.
    from nvfp4_block_sparse_gb300 import build
    if not os.path.exists(build.BOUNDS_LIB):
        build.build()
    blib = ctypes.CDLL(build.BOUNDS_LIB)
    for name in declared_functions():
        assert hasattr(blib, name), name
    if not qsa.bounds_checked():
        assert qsa.qsa_debug_bounds_status() == -1


def test_status_strings(lib):
    for s in range(6):
        assert qsa.qsa_status_string(s)
    assert "unknown" in qsa.qsa_status_string(99)


def geom(**kw):
    base = dict(batch=2, rows_per_req=1, num_q_heads=8, num_kv_heads=2, head_dim=128,
                index_dim=64, page_size=64, max_blocks=16, num_pages=32)
    base.update(kw)
    return qsa.make_geom(**base)


FAKE = ctypes.c_void_p(256)   # never dereferenced: validation fails first


@pytest.mark.parametrize("bad,status", [
    (dict(num_q_heads=7), 1), (dict(batch=0), 1), (dict(rows_per_req=0), 1),
    (dict(max_blocks=0), 1), (dict(num_pages=0), 1), (dict(head_dim=64), 2),
    (dict(index_dim=128), 2), (dict(page_size=32), 2), (dict(rows_per_req=4097), 2),
    (dict(head_dim=192), 2), (dict(head_dim=256, page_size=128), 2),
    (dict(head_dim=256, page_size=16), 2),
    (dict(num_q_heads=512, num_kv_heads=2), 2),
])
def test_geometry_validation(lib, bad, status):
    g = geom(**bad)
    st = lib.qsa_index_scores(ctypes.byref(g), FAKE, FAKE, FAKE, FAKE, FAKE, None)
    assert st == status


def test_null_pointers_rejected(lib):
    g = geom()
    assert lib.qsa_index_scores(ctypes.byref(g), None, FAKE, FAKE, FAKE, FAKE, None) == 1
    assert lib.qsa_select_topk(ctypes.byref(g), FAKE, FAKE, 4, 1, None, FAKE, None) == 1
    assert lib.qsa_index_scores(None, FAKE, FAKE, FAKE, FAKE, FAKE, None) == 1


@pytest.mark.parametrize("k,window,status", [(0, 0, 1), (4, -1, 1), (4, 5, 1), (2000, 2, 2)])
def test_select_argument_validation(lib, k, window, status):
    g = geom()
    assert lib.qsa_select_topk(ctypes.byref(g), FAKE, FAKE, k, window, FAKE, FAKE, None) == status


def test_unaligned_pool_rejected(lib):
    g = geom()
    odd = ctypes.c_void_p(257)
    assert lib.qsa_index_scores(ctypes.byref(g), FAKE, odd, FAKE, FAKE, FAKE, None) == 1


def test_workspace_sizes(lib):
    g = geom(rows_per_req=4)
    assert qsa.qsa_sparse_decode_workspace_bytes_ex(g, 8, 1) > 0
    one = qsa.qsa_sparse_decode_workspace_bytes_ex(g, 8, 1)
    four = qsa.qsa_sparse_decode_workspace_bytes_ex(g, 8, 4)
    assert four > one
    assert qsa.qsa_sparse_decode_workspace_bytes_ex(g, 0, 1) == 0          # k < 1
    assert qsa.qsa_sparse_decode_workspace_bytes_ex(geom(rows_per_req=8), 512, 1) == 0


def test_decode_rejects_small_workspace(lib):
    g = geom()
    need = qsa.qsa_sparse_decode_workspace_bytes_ex(g, 8, 4)
    args = [ctypes.byref(g)] + [FAKE] * 5 + [1.0, 1.0, 0.1] + [FAKE] * 3 + [8] + [FAKE] * 2
    st = lib.qsa_sparse_decode_ex(*args, FAKE, need - 1, 4, None)
    assert st == 4
    st = lib.qsa_sparse_decode_ex(*args, None, need, 4, None)
    assert st == 4


def test_no_cpu_fallback_without_library(monkeypatch, tmp_path):
    # The binding refuses to run when the library is absent instead of
    # computing anything on the host.
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding._build, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(ImportError):
        binding.load()


def test_context_row_groups_validation(lib):
    # Long row groups: index scores / selection / row-tile attention accept up
    # to 4096 rows per request; the decode attention keeps its 8.
    long = geom(rows_per_req=512, num_q_heads=32, num_kv_heads=4)
    assert qsa.qsa_sparse_prefill_workspace_bytes(long, 64) > 0
    assert qsa.qsa_sparse_decode_workspace_bytes_ex(long, 64, 0) == 0
    assert qsa.qsa_sparse_decode_workspace_bytes_ex(geom(rows_per_req=9), 8, 0) == 0
    assert qsa.qsa_sparse_prefill_workspace_bytes(long, 0) == 0                    # k < 1
    assert qsa.qsa_sparse_prefill_workspace_bytes(geom(head_dim=256, page_size=32), 8) > 0
    assert qsa.qsa_sparse_prefill_workspace_bytes(geom(head_dim=256, page_size=128), 8) == 0
    assert qsa.qsa_sparse_prefill_workspace_bytes(
        geom(num_q_heads=256, num_kv_heads=1), 8) == 0                            # G > 128
    assert qsa.qsa_sparse_prefill_workspace_bytes(geom(rows_per_req=4097), 8) == 0
    ws = qsa.qsa_sparse_prefill_workspace_bytes(long, 64)
    args = [ctypes.byref(long)] + [FAKE] * 5
    tail = [FAKE, FAKE, FAKE, 64, FAKE, FAKE, FAKE, ws, None]
    # non-positive or non-finite scales are rejected before any launch
    for ks, vs, sm in ((0.0, 1.0, 0.1), (1.0, 1.0, -0.1), (float("nan"), 1.0, 0.1),
                       (1.0, float("inf"), 0.1)):
        assert lib.qsa_sparse_prefill(*args, ks, vs, sm, *tail) == 1
    # a missing or short workspace
    good = [ctypes.byref(long)] + [FAKE] * 5 + [1.0, 1.0, 0.1, FAKE, FAKE, FAKE, 64, FAKE, FAKE]
    assert lib.qsa_sparse_prefill(*good, None, ws, None) == 4
    assert lib.qsa_sparse_prefill(*good, FAKE, ws - 1, None) == 4


def test_prologue_and_rollback_row_limits(lib):
    # The prologue stores context row groups (up to 4096 rows per request);
    # the rollback serves speculative rows (up to 8).
    ok_long = geom(rows_per_req=512, num_q_heads=32, num_kv_heads=4)
    too_long = geom(rows_per_req=4097)
    st = lib.qsa_store_kv_tokens(ctypes.byref(too_long), FAKE, FAKE, FAKE, 1.0, 1.0,
                                 FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None)
    assert st == 2
    # (every call here is rejected by host validation before any launch: the
    # pointers are placeholders)
    assert lib.qsa_rollback_state_bytes(ctypes.byref(ok_long)) == 0
    assert lib.qsa_rollback_state_bytes(ctypes.byref(geom(rows_per_req=9))) == 0
    assert lib.qsa_rollback_gather(ctypes.byref(geom(rows_per_req=9)), *([FAKE] * 8), None) == 2
    # non-positive scales are rejected by the prologue
    st = lib.qsa_store_kv_tokens(ctypes.byref(geom()), FAKE, FAKE, FAKE, 0.0, 1.0,
                                 FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None)
    assert st == 1
