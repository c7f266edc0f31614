"""qsa_sparse_decode_noalloc: the sparse decode call for callers that cannot
allocate device memory (allocator-free runtimes, fixed memory pools, plugins
handed only input and output pointers).  It uses the library's built-in
scratch array instead of a caller workspace, so it is checked here against the
regular entry point, through the C ABI, on two calls in a row (the second one
reuses whatever the first left in the shared array).

This file is collected last on purpose, and it also passes when run alone.
"""
import ctypes

import numpy as np
import pytest
import torch

import qsa_workloads as qw

pytestmark = pytest.mark.gpu

OUT_ABS, OUT_REL, LSE_ABS = 1e-2, 5e-3, 1e-3


@pytest.fixture(scope="module")
def qsa():
    import nvfp4_block_sparse_gb300 as m
    m.load(build_if_missing=True)
    return m


def _close(out, lse, ref_out, ref_lse):
    out = out.float().cpu().numpy().astype(np.float64)
    ref_out = ref_out.float().cpu().numpy().astype(np.float64)
    lse = lse.cpu().numpy().astype(np.float64)
    ref_lse = ref_lse.cpu().numpy().astype(np.float64)
    assert np.abs(out - ref_out).max() <= OUT_ABS
    den = np.linalg.norm(ref_out)
    assert (np.linalg.norm(out - ref_out) / den if den > 0 else np.linalg.norm(out)) <= OUT_REL
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    fin = np.isfinite(ref_lse)
    if fin.any():
        assert np.abs(lse[fin] - ref_lse[fin]).max() <= LSE_ABS


@pytest.mark.parametrize("cfg", [1, 2, 4])
def test_noalloc_matches_workspace_entry_point_twice(qsa, cfg):
    w = qw.make_workload(qw.small(qw.WORKLOADS[cfg]), "cuda")
    step = qsa.DecodeStep(qw.geometry(w), w["k"], w["window"])
    step.run(w)                     # scores, selection and the reference output
    torch.cuda.synchronize()
    ref_out, ref_lse = step.out.clone(), step.lse.clone()
    lib = qsa.load()
    g = qsa.make_geom(**qw.geometry(w))
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        out = torch.full_like(step.out, float("nan"))
        lse = torch.full_like(step.lse, float("nan"))
        st = lib.qsa_sparse_decode_noalloc(
            ctypes.byref(g), w["q"].data_ptr(), w["k_pool"].data_ptr(), w["k_sf"].data_ptr(),
            w["v_pool"].data_ptr(), w["v_sf"].data_ptr(), ctypes.c_float(w["k_scale"]),
            ctypes.c_float(w["v_scale"]), ctypes.c_float(w["sm_scale"]),
            w["page_table"].data_ptr(), w["seqlens"].data_ptr(), step.sel.data_ptr(),
            int(w["k"]), out.data_ptr(), lse.data_ptr(), ctypes.c_void_p(stream))
        assert st == 0, qsa.qsa_status_string(st)
        torch.cuda.synchronize()
        _close(out, lse, ref_out, ref_lse)


def test_noalloc_rejects_geometry_beyond_its_scratch(qsa):
    # 2^20 (request, KV head) units need more than the built-in array holds
    # even with one split: rejected with QSA_ERR_WORKSPACE, nothing launched.
    lib = qsa.load()
    g = qsa.make_geom(batch=65535, rows_per_req=1, num_q_heads=256, num_kv_heads=32,
                      head_dim=128, index_dim=64, page_size=64, max_blocks=1, num_pages=1)
    fake = ctypes.c_void_p(256)
    st = lib.qsa_sparse_decode_noalloc(ctypes.byref(g), fake, fake, fake, fake, fake,
                                       ctypes.c_float(1.0), ctypes.c_float(1.0),
                                       ctypes.c_float(0.1), fake, fake, fake, 1, fake, fake,
                                       ctypes.c_void_p(0))
    assert st == 4


NOALLOC_BYTES = 4 << 20


def _lowered_splits(qsa, geom, k):
    """The split count qsa_sparse_decode_noalloc runs: the automatic one,
    lowered until the workspace fits the 4 MiB array."""
    auto = qsa.qsa_sparse_decode_workspace_bytes(geom, k)
    splits = next(s for s in range(1, 65)
                  if qsa.qsa_sparse_decode_workspace_bytes_ex(geom, k, s) == auto)
    while splits > 1 and qsa.qsa_sparse_decode_workspace_bytes_ex(geom, k, splits) > NOALLOC_BYTES:
        splits -= 1
    return auto, splits


def test_noalloc_lowers_splits_to_fit_its_scratch(qsa):
    # Four rows per request, 8 query heads per KV head (32 query columns per
    # CTA) and 38 (request, KV head) units: the automatic plan spreads every
    # unit over 8 splits, whose partials need more than the 4 MiB array, so
    # the call runs fewer splits.  Checked against the workspace entry point
    # at that split count (the same bits) and against the oracle on sampled
    # requests.
    import oracle
    case = qw.Case("noalloc lowering", seed=31, batch=19, rows_per_req=4, num_q_heads=16,
                   num_kv_heads=2, page_size=64, ctx_lo=2600, ctx_hi=4100, k=12, window=2,
                   max_blocks=65, pool="perm")
    w = qw.make_workload(case, "cuda")
    geom = qw.geometry(w)
    auto, splits = _lowered_splits(qsa, geom, w["k"])
    assert auto > NOALLOC_BYTES and splits >= 1
    step = qsa.DecodeStep(geom, w["k"], w["window"], num_splits=splits)
    step.run(w)
    torch.cuda.synchronize()
    ref_out, ref_lse = step.out.clone(), step.lse.clone()
    for _ in range(2):
        out = torch.full_like(step.out, float("nan"))
        lse = torch.full_like(step.lse, float("nan"))
        qsa.qsa_sparse_decode_noalloc(step.cg, w["q"], w["k_pool"], w["k_sf"], w["v_pool"],
                                      w["v_sf"], w["k_scale"], w["v_scale"], w["sm_scale"],
                                      w["page_table"], w["seqlens"], step.sel, w["k"], out, lse)
        torch.cuda.synchronize()
        assert qsa.qsa_sparse_decode_noalloc_status() == 0
        # same kernel, same split count: the same bits
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)
    w_np = qw.to_numpy(w)
    R = case.rows_per_req
    for b in (0, case.batch // 2, case.batch - 1):
        ref = oracle.step(w_np, rows=(b * R, b * R + R))
        _close(out[b * R:b * R + R], lse[b * R:b * R + R],
               torch.from_numpy(ref["out"][b * R:b * R + R]),
               torch.from_numpy(ref["lse"][b * R:b * R + R]))


def test_noalloc_reports_a_wait_that_gave_up(qsa):
    # A wait bound of a few nanoseconds makes the kernel's copy waits give up
    # (the copies still land before it finishes): the built-in array's status
    # word then reports QSA_ERR_DEVICE_TIMEOUT until it is read, and the next
    # call under the default bound is correct again.
    w = qw.make_workload(qw.small(qw.WORKLOADS[1]), "cuda")
    step = qsa.DecodeStep(qw.geometry(w), w["k"], w["window"])
    step.run(w)
    torch.cuda.synchronize()
    assert qsa.qsa_sparse_decode_noalloc_status() == 0
    out = torch.empty_like(step.out)
    lse = torch.empty_like(step.lse)
    args = (step.cg, w["q"], w["k_pool"], w["k_sf"], w["v_pool"], w["v_sf"], w["k_scale"],
            w["v_scale"], w["sm_scale"], w["page_table"], w["seqlens"], step.sel, w["k"], out,
            lse)
    try:
        qsa.qsa_debug_set_wait_ns(4)
        qsa.qsa_sparse_decode_noalloc(*args)
        torch.cuda.synchronize()
    finally:
        qsa.qsa_debug_set_wait_ns(0)
    lib = qsa.load()
    code = ctypes.c_int(0)
    st = lib.qsa_sparse_decode_noalloc_status(ctypes.byref(code),
                                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 5 and code.value != 0                     # QSA_ERR_DEVICE_TIMEOUT
    assert qsa.qsa_sparse_decode_noalloc_status() == 0      # read and cleared
    qsa.qsa_sparse_decode_noalloc(*args)
    torch.cuda.synchronize()
    assert qsa.qsa_sparse_decode_noalloc_status() == 0
    _close(out, lse, step.out, step.lse)
