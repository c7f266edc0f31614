"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bars: index scores, selections and selection counts bit-exact; out within max
abs 1e-2 and relative L2 5e-3; lse within 1e-3 absolute (the tolerances the
method's acceptance criteria state).
"""
import numpy as np
import pytest
import torch

import oracle
import qsa_workloads as qw

pytestmark = pytest.mark.gpu

OUT_ABS, OUT_REL, LSE_ABS = 1e-2, 5e-3, 1e-3


@pytest.fixture(scope="module")
def qsa():
    import nvfp4_block_sparse_gb300 as m
    m.load(build_if_missing=True)
    return m


def run_gpu(qsa, w, num_splits=0, window=None, k=None):
    step = qsa.DecodeStep(qw.geometry(w), k or w["k"], w["window"] if window is None else window,
                          device=w["q"].device, num_splits=num_splits)
    step.run(w)
    torch.cuda.synchronize()
    # A bounded wait that gave up leaves a status in the workspace.
    assert step.status() == 0
    return step


def host(step):
    return dict(scores=step.scores.cpu().numpy(), sel=step.sel.cpu().numpy(),
                nsel=step.nsel.cpu().numpy(),
                out=step.out.float().cpu().numpy().astype(np.float64),
                lse=step.lse.cpu().numpy().astype(np.float64))


def assert_out_close(out, lse, ref_out, ref_lse, rows=None):
    if rows is not None:
        out, lse, ref_out, ref_lse = out[rows], lse[rows], ref_out[rows], ref_lse[rows]
    err = np.abs(out - ref_out).max() if out.size else 0.0
    den = np.linalg.norm(ref_out)
    rel = np.linalg.norm(out - ref_out) / den if den > 0 else np.linalg.norm(out)
    assert err <= OUT_ABS, "max abs out error %.3e" % err
    assert rel <= OUT_REL, "relative L2 out error %.3e" % rel
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(lse), fin), "lse finiteness differs"
    assert np.array_equal(np.isneginf(lse), np.isneginf(ref_lse))
    if fin.any():
        le = np.abs(lse[fin] - ref_lse[fin]).max()
        assert le <= LSE_ABS, "max abs lse error %.3e" % le


def check_against_oracle(res, w_np, rows=None):
    ref = oracle.step(w_np, rows=rows)
    r = slice(None) if rows is None else slice(rows[0], rows[1])
    np.testing.assert_array_equal(res["scores"][r], ref["scores"][r])
    np.testing.assert_array_equal(res["sel"][r], ref["sel"][r])
    np.testing.assert_array_equal(res["nsel"][r], ref["nsel"][r])
    assert_out_close(res["out"][r], res["lse"][r], ref["out"][r], ref["lse"][r])
    return ref


# ---------------------------------------------------------------------------
# the workloads, reduced to oracle speed (several tiles + ragged tails)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("cfg", range(len(qw.WORKLOADS)))
def test_small_configs(qsa, cfg):
    case = qw.small(qw.WORKLOADS[cfg])
    w = qw.make_workload(case, "cuda")
    res = host(run_gpu(qsa, w))
    check_against_oracle(res, qw.to_numpy(w))


@pytest.mark.parametrize("cfg,splits", [(1, 1), (1, 2), (1, 7), (1, 64), (2, 1), (2, 3),
                                        (4, 1), (4, 5), (3, 1), (3, 16), (5, 1), (5, 2),
                                        (5, 8), (5, 24)])
def test_forced_splits(qsa, cfg, splits):
    case = qw.small(qw.WORKLOADS[cfg])
    w = qw.make_workload(case, "cuda")
    res = host(run_gpu(qsa, w, num_splits=splits))
    check_against_oracle(res, qw.to_numpy(w))


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------

def _case(**kw):
    base = dict(name="edge", seed=21, batch=3, rows_per_req=1, num_q_heads=8, num_kv_heads=2,
                page_size=64, ctx_lo=700, ctx_hi=1300, k=6, window=2, max_blocks=21,
                pool="perm")
    base.update(kw)
    return qw.Case(**base)


EDGE_CASES = {
    "ragged_tails_p64": _case(ctx_lo=65, ctx_hi=1283),
    "ragged_tails_p128": _case(page_size=128, ctx_lo=129, ctx_hi=2600, max_blocks=21),
    "k_covers_all": _case(k=40, window=3),
    "window_zero": _case(window=0),
    "window_is_k": _case(k=5, window=5),
    "k_one": _case(k=1, window=0),
    "invalid_pages": _case(invalid_frac=0.3, rows_per_req=2),
    "mostly_invalid": _case(invalid_frac=0.9, rows_per_req=3),
    "tiny_contexts_verify": _case(rows_per_req=4, ctx_lo=1, ctx_hi=6, max_blocks=2, k=2, window=1),
    "eight_draft_rows": _case(rows_per_req=8, num_q_heads=4, num_kv_heads=1, k=5),
    "gqa12_nt2": _case(num_q_heads=24, num_kv_heads=2),
    "wide_cols_two_groups": _case(num_q_heads=24, num_kv_heads=2, rows_per_req=4, k=5),
    "cols_24_team": _case(num_q_heads=24, num_kv_heads=4, rows_per_req=4),
    "mqa_64_heads": _case(num_q_heads=64, num_kv_heads=1, rows_per_req=1, batch=2),
    "ties": _case(tie_frac=0.5, rows_per_req=2),
    # page-table rows far wider than the requests' blocks
    "wide_table": _case(max_blocks=2100, rows_per_req=2, tie_frac=0.3),
    "wide_table_verify4": _case(max_blocks=2049, rows_per_req=4, k=9),
    # head_dim 256 (32-token stages): decode and verify rows, 32- and 64-token
    # pages, head groups wider than one 8-column slice, masks and tails
    "hd256_decode_p32": _case(head_dim=256, page_size=32, max_blocks=41, k=9, window=2,
                              num_q_heads=24, num_kv_heads=2),
    "hd256_decode_p64": _case(head_dim=256, num_q_heads=16, num_kv_heads=2),
    "hd256_verify2_p64": _case(head_dim=256, rows_per_req=2, num_q_heads=12, num_kv_heads=1),
    "hd256_verify3": _case(head_dim=256, page_size=32, max_blocks=41, rows_per_req=3, k=10),
    "hd256_verify4_g12": _case(head_dim=256, page_size=32, max_blocks=41, rows_per_req=4, k=12,
                               num_q_heads=24, num_kv_heads=2, invalid_frac=0.2),
    "hd256_eight_rows": _case(head_dim=256, page_size=32, max_blocks=41, rows_per_req=8,
                              num_q_heads=4, num_kv_heads=1, k=7),
    "hd256_ragged_tiny": _case(head_dim=256, page_size=32, rows_per_req=4, ctx_lo=1, ctx_hi=70,
                               max_blocks=3, k=2, window=1),
    "hd256_ties": _case(head_dim=256, page_size=32, max_blocks=41, tie_frac=0.5, rows_per_req=2,
                        k=8),
}


@pytest.mark.parametrize("name", sorted(EDGE_CASES))
def test_edge_cases(qsa, name):
    w = qw.make_workload(EDGE_CASES[name], "cuda")
    res = host(run_gpu(qsa, w))
    check_against_oracle(res, qw.to_numpy(w))


@pytest.mark.parametrize("rows", [2, 4, 8])
def test_index_large_head_sums(qsa, rows):
    # The first request's rows at +-127 with one sign per (row, dim) for every
    # head: head-summed weights of Hq * 127, beyond the single-product range of
    # the tensor-core index kernel, so its CTAs take the exact two-part
    # products while the other requests' CTAs take one product.
    w = qw.make_workload(_case(rows_per_req=rows, num_q_heads=32, num_kv_heads=4), "cuda")
    iq = w["iq"]
    Di = iq.shape[-1]
    gen = torch.Generator().manual_seed(11)
    sign = torch.randint(0, 2, (rows, 1, Di), generator=gen) * 254 - 127
    iq[:rows] = sign.to(torch.int8).to(iq.device).expand(-1, iq.shape[1], -1)
    res = host(run_gpu(qsa, w))
    check_against_oracle(res, qw.to_numpy(w))


def test_all_pages_invalid(qsa):
    w = qw.make_workload(_case(rows_per_req=2), "cuda")
    w["page_table"].fill_(-1)
    res = host(run_gpu(qsa, w))
    assert np.all(res["scores"] == np.iinfo(np.int32).min)
    assert np.all(res["nsel"] == 0) and np.all(res["sel"] == -1)
    assert np.all(res["out"] == 0) and np.all(np.isneginf(res["lse"]))


def test_all_equal_scores_select_highest_blocks(qsa):
    # Every index key zero -> every valid block scores 0 -> ties everywhere:
    # the canonical rule takes the highest-index blocks.
    w = qw.make_workload(_case(rows_per_req=1, batch=2, ctx_lo=1280, ctx_hi=1280), "cuda")
    w["ik_pool"].zero_()
    res = host(run_gpu(qsa, w))
    k = w["k"]
    for r in range(res["sel"].shape[0]):
        nb = 1280 // 64
        np.testing.assert_array_equal(res["sel"][r], np.arange(nb - k, nb))


def test_page_permutation_leaves_outputs_bitwise_unchanged(qsa):
    case = qw.small(qw.WORKLOADS[4])
    w = qw.make_workload(case, "cuda")
    res = host(run_gpu(qsa, w))
    NP = w["num_pages"]
    perm = torch.randperm(NP, generator=torch.Generator().manual_seed(3)).cuda()
    w2 = dict(w)
    for key in ("ik_pool", "k_pool", "k_sf", "v_pool", "v_sf"):
        arr = torch.empty_like(w[key])
        arr[perm] = w[key]
        w2[key] = arr
    pt = w["page_table"].long()
    w2["page_table"] = torch.where(pt >= 0, perm[pt.clamp(min=0)], pt).to(torch.int32)
    res2 = host(run_gpu(qsa, w2))
    for key in ("scores", "sel", "nsel", "out", "lse"):
        np.testing.assert_array_equal(res[key], res2[key])


def test_selection_deterministic_over_50_launches(qsa):
    case = qw.small(qw.WORKLOADS[4], batch=6)
    w = qw.make_workload(case, "cuda")
    step = run_gpu(qsa, w)
    sel0, out0 = step.sel.clone(), step.out.clone()
    for _ in range(50):
        step.run(w)
        assert torch.equal(step.sel, sel0)
        assert torch.equal(step.out, out0)


def test_cuda_graph_replay_matches_eager(qsa):
    case = qw.small(qw.WORKLOADS[2])
    w = qw.make_workload(case, "cuda")
    step = run_gpu(qsa, w)
    eager = host(step)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        step.run(w, stream=s)          # warm-up on the capture stream
        s.synchronize()
        with torch.cuda.graph(g, stream=s):
            step.run(w, stream=s)
    step.out.zero_()
    step.sel.zero_()
    g.replay()
    torch.cuda.synchronize()
    replay = host(step)
    for key in ("scores", "sel", "nsel", "out", "lse"):
        np.testing.assert_array_equal(eager[key], replay[key])


def test_workspace_status_clean(qsa):
    w = qw.make_workload(qw.small(qw.WORKLOADS[1]), "cuda")
    step = run_gpu(qsa, w)
    assert step.status() == 0


def test_workspace_too_small_is_rejected(qsa):
    w = qw.make_workload(qw.small(qw.WORKLOADS[1]), "cuda")
    step = run_gpu(qsa, w, num_splits=4)
    small_ws = step.workspace[:64]
    with pytest.raises(qsa.QsaError) as ei:
        qsa.qsa_sparse_decode_ex(step.cg, w["q"], w["k_pool"], w["k_sf"], w["v_pool"],
                                 w["v_sf"], w["k_scale"], w["v_scale"], w["sm_scale"],
                                 w["page_table"], w["seqlens"], step.sel, step.k, step.out,
                                 step.lse, small_ws, 4)
    assert ei.value.status == 4


# ---------------------------------------------------------------------------
# full-size workloads (the benchmark's launch configuration), sampled rows
# ---------------------------------------------------------------------------

def _selection_properties(res, w_np):
    R, P, k, W, MB = (w_np["rows_per_req"], w_np["page_size"], w_np["k"], w_np["window"],
                      w_np["max_blocks"])
    pt = w_np["page_table"]
    for r in range(res["sel"].shape[0]):
        b, j = divmod(r, R)
        n = max(0, min(int(w_np["seqlens"][b]) - R + 1 + j, MB * P))
        nb = -(-n // P)
        valid = pt[b, :nb] >= 0
        s = res["sel"][r, : res["nsel"][r]]
        assert res["nsel"][r] == min(k, int(valid.sum()))
        assert np.all(np.diff(s) > 0)
        assert np.all(valid[s])
        win = np.arange(max(0, nb - W), nb)
        assert np.all(np.isin(win[valid[win]], s))
        assert np.all(res["sel"][r, res["nsel"][r]:] == -1)


@pytest.mark.parametrize("cfg", range(len(qw.WORKLOADS)))
def test_full_size_sampled_rows(qsa, cfg):
    case = qw.WORKLOADS[cfg]
    w = qw.make_workload(case, "cuda")
    res = host(run_gpu(qsa, w))
    w_np = qw.to_numpy(w)
    _selection_properties(res, w_np)
    T = case.rows
    R = case.rows_per_req
    # first request, last request, and one in the middle (whole requests)
    picks = sorted({0, (case.batch // 2) * R, T - R})
    for r0 in picks:
        check_against_oracle(res, w_np, rows=(r0, r0 + R))


# ---------------------------------------------------------------------------
# fused selection + decode against the composed calls (bit for bit)
# ---------------------------------------------------------------------------

FUSED_CASES = [("cfg0", lambda: qw.small(qw.WORKLOADS[0]), 0),
               ("cfg1", lambda: qw.small(qw.WORKLOADS[1]), 0),
               ("cfg3", lambda: qw.small(qw.WORKLOADS[3]), 0),
               ("cfg1_full", lambda: qw.WORKLOADS[1], 0),
               ("cfg3_full", lambda: qw.WORKLOADS[3], 0),
               ("cfg1_split1", lambda: qw.small(qw.WORKLOADS[1]), 1),
               ("cfg1_split7", lambda: qw.small(qw.WORKLOADS[1]), 7),
               ("cfg1_split64", lambda: qw.small(qw.WORKLOADS[1]), 64),
               ("window0", lambda: EDGE_CASES["window_zero"], 0),
               ("k_one", lambda: EDGE_CASES["k_one"], 0),
               ("ties", lambda: _case(tie_frac=0.5), 0),
               ("invalid", lambda: _case(invalid_frac=0.3), 0),
               ("gqa12", lambda: EDGE_CASES["gqa12_nt2"], 0),
               ("hd256_p32", lambda: EDGE_CASES["hd256_decode_p32"], 0),
               ("hd256_p64_split3", lambda: EDGE_CASES["hd256_decode_p64"], 3),
               ("cfg2_composed_inside", lambda: qw.small(qw.WORKLOADS[2]), 0)]


@pytest.mark.parametrize("name,make,splits", FUSED_CASES, ids=[c[0] for c in FUSED_CASES])
def test_fused_selection_matches_composed(qsa, name, make, splits):
    w = qw.make_workload(make(), "cuda")
    c = run_gpu(qsa, w, num_splits=splits)
    step_f = qsa.DecodeStep(qw.geometry(w), w["k"], w["window"], device=w["q"].device,
                            num_splits=splits, fused=True)
    step_f.run(w)
    torch.cuda.synchronize()
    assert step_f.status() == 0
    ra, rc = host(step_f), host(c)
    for key in ("scores", "sel", "nsel", "out", "lse"):
        np.testing.assert_array_equal(ra[key], rc[key], err_msg=key)
    # One launch only where the per-row-warp kernel serves the geometry (head
    # dim 256, decode rows); head dim 128 selects, then attends.
    fused = qsa.qsa_select_sparse_decode_fused(qw.geometry(w))
    assert bool(fused) == (w["rows_per_req"] == 1 and w["head_dim"] == 256)
