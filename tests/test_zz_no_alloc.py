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
    w = qw.make_workload(qw.small(qw.CONFIGS[cfg]), "cuda")
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
