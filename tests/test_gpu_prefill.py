"""GPU parity of the context row-tile path (qsa_sparse_prefill, tcgen05) against
the oracle: index scores and selections bit-exact for long row groups, out
within max abs 1e-2 / relative L2 5e-3 and lse within 1e-3.
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


def run_step(qsa, w):
    step = qsa.DecodeStep(qw.geometry(w), w["k"], w["window"], device=w["q"].device)
    assert step.prefill
    step.run(w)
    torch.cuda.synchronize()
    assert step.status() == 0
    return step


def check(step, w_np, rows=None):
    ref = oracle.step(w_np, rows=rows)
    r = slice(None) if rows is None else slice(rows[0], rows[1])
    np.testing.assert_array_equal(step.scores.cpu().numpy()[r], ref["scores"][r])
    np.testing.assert_array_equal(step.sel.cpu().numpy()[r], ref["sel"][r])
    np.testing.assert_array_equal(step.nsel.cpu().numpy()[r], ref["nsel"][r])
    out = step.out.float().cpu().numpy().astype(np.float64)[r]
    lse = step.lse.cpu().numpy().astype(np.float64)[r]
    ro, rl = ref["out"][r], ref["lse"][r]
    err = np.abs(out - ro).max()
    den = np.linalg.norm(ro)
    rel = np.linalg.norm(out - ro) / den if den > 0 else np.linalg.norm(out)
    assert err <= OUT_ABS, "max abs out error %.3e" % err
    assert rel <= OUT_REL, "relative L2 out error %.3e" % rel
    fin = np.isfinite(rl)
    assert np.array_equal(np.isneginf(lse), np.isneginf(rl))
    if fin.any():
        assert np.abs(lse[fin] - rl[fin]).max() <= LSE_ABS


def _case(**kw):
    base = dict(name="prefill", seed=61, batch=1, rows_per_req=48, num_q_heads=32,
                num_kv_heads=4, page_size=64, ctx_lo=3100, ctx_hi=3100, k=16, window=2,
                max_blocks=49, pool="perm", iq_row_noise=24)
    base.update(kw)
    return qw.Case(**base)


CASES = {
    # three 16-row tiles of 8 heads, partial block at the end of the context
    "g8_three_tiles": _case(),
    # ragged last tile, two requests of different lengths
    "g8_ragged_rows": _case(batch=2, rows_per_req=37, ctx_lo=2400, ctx_hi=3100),
    # 32-row tiles (4 heads per KV head) and 8-row tiles (16 heads)
    "g4_rows32": _case(num_q_heads=16, rows_per_req=70),
    "g16_rows8": _case(num_q_heads=32, num_kv_heads=2, rows_per_req=20),
    # 12 heads: 10-row tiles with 8 padding vectors
    "g12_padding": _case(num_q_heads=24, num_kv_heads=2, rows_per_req=23),
    # 128-token pages (two chunks per block), invalid pages, ties
    "p128_invalid_ties": _case(page_size=128, ctx_lo=4000, ctx_hi=6000, max_blocks=47,
                               invalid_frac=0.15, tie_frac=0.3, batch=2, rows_per_req=24),
    # independent rows: every tile's union covers most of the context
    "independent_rows": _case(iq_row_noise=0, rows_per_req=32),
    # the context is shorter than the row group: early rows see nothing
    "rows_longer_than_context": _case(rows_per_req=40, ctx_lo=30, ctx_hi=130, max_blocks=3,
                                      k=2, window=1),
    # k covers every block, window 0
    "dense_window0": _case(k=60, window=0, rows_per_req=17),
    # one KV head, 128 query heads per KV head: one row per tile
    "mqa_g128": _case(num_q_heads=128, num_kv_heads=1, rows_per_req=9, ctx_lo=1500,
                      ctx_hi=1500, max_blocks=24),
    # head_dim 256 (32-token chunks, 512 tensor-memory columns): the pages'
    # geometry (12 heads per KV head, 10-row tiles, 32-token pages), 64-token
    # pages with 8 heads, invalid pages and ties
    "hd256_g12_p32": _case(head_dim=256, page_size=32, num_q_heads=24, num_kv_heads=2,
                           rows_per_req=23, ctx_lo=1500, ctx_hi=1700, batch=2, max_blocks=54,
                           k=12),
    "hd256_g8_p64_ragged": _case(head_dim=256, num_q_heads=16, num_kv_heads=2, batch=2,
                                 rows_per_req=37, ctx_lo=2400, ctx_hi=3100),
    "hd256_invalid_ties": _case(head_dim=256, page_size=32, num_q_heads=8, num_kv_heads=1,
                                rows_per_req=24, ctx_lo=1200, ctx_hi=1400, max_blocks=44,
                                k=10, invalid_frac=0.15, tie_frac=0.3),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_prefill_matches_oracle(qsa, name):
    w = qw.make_workload(CASES[name], "cuda")
    step = run_step(qsa, w)
    check(step, qw.to_numpy(w))


def _saturate_iq(w, rows, seed):
    """Index queries of the given rows at +-127 with one sign per (row, dim)
    for every head: each head-summed weight is then Hq * 127 in magnitude,
    beyond the single-product range of the tensor-core index kernels."""
    iq = w["iq"]
    Di = iq.shape[-1]
    gen = torch.Generator().manual_seed(seed)
    sign = torch.randint(0, 2, (len(rows), 1, Di), generator=gen) * 254 - 127
    iq[rows] = sign.to(torch.int8).to(iq.device).expand(-1, iq.shape[1], -1)


def test_prefill_large_head_sums(qsa):
    # Rows 0-15 saturated (their 64-row group takes the exact two-part products),
    # the next 64-row group left as drawn: both index paths in one step.
    w = qw.make_workload(_case(rows_per_req=80, ctx_lo=4200, ctx_hi=4200, max_blocks=66), "cuda")
    _saturate_iq(w, list(range(16)), 5)
    step = run_step(qsa, w)
    check(step, qw.to_numpy(w))


def test_prefill_all_pages_invalid(qsa):
    w = qw.make_workload(_case(rows_per_req=20), "cuda")
    w["page_table"].fill_(-1)
    step = run_step(qsa, w)
    assert torch.all(step.out == 0)
    assert torch.all(torch.isneginf(step.lse))


def test_prefill_on_verify_rows_matches_decode(qsa):
    # The row-tile kernel called directly on a verify geometry (R <= 8) gives
    # the decode kernel's results within the tolerance, and the oracle's.
    w = qw.make_workload(qw.small(qw.WORKLOADS[2]), "cuda")
    step = qsa.DecodeStep(qw.geometry(w), w["k"], w["window"], device=w["q"].device)
    step.run(w)
    out = torch.empty_like(step.out)
    lse = torch.empty_like(step.lse)
    ws = torch.zeros(qsa.qsa_sparse_prefill_workspace_bytes(step.cg, step.k),
                     dtype=torch.uint8, device=w["q"].device)
    qsa.qsa_sparse_prefill(step.cg, w["q"], w["k_pool"], w["k_sf"], w["v_pool"], w["v_sf"],
                           w["k_scale"], w["v_scale"], w["sm_scale"], w["page_table"],
                           w["seqlens"], step.sel, step.k, out, lse, ws)
    torch.cuda.synchronize()
    assert qsa.qsa_workspace_status(ws) == 0
    d = (out.float() - step.out.float()).abs().max().item()
    assert d <= 2 * OUT_ABS
    fin = torch.isfinite(step.lse)
    assert torch.equal(torch.isfinite(lse), fin)
    assert (lse[fin] - step.lse[fin]).abs().max().item() <= 2 * LSE_ABS


@pytest.mark.parametrize("cfg", qw.PREFILL_WORKLOADS)
def test_prefill_full_size_sampled_rows(qsa, cfg):
    case = qw.WORKLOADS[cfg]
    w = qw.make_workload(case, "cuda")
    step = run_step(qsa, w)
    w_np = qw.to_numpy(w)
    R, T = case.rows_per_req, case.rows
    tr = 128 // (case.num_q_heads // case.num_kv_heads)
    # a tile at the start, one in the middle, the last rows of the last request
    mid = R + (R // 2 // tr) * tr
    for r0, r1 in ((0, tr), (mid, mid + tr), (T - tr, T)):
        check(step, w_np, rows=(r0, r1))


def test_prefill_deterministic(qsa):
    w = qw.make_workload(CASES["g8_three_tiles"], "cuda")
    step = run_step(qsa, w)
    out0, lse0 = step.out.clone(), step.lse.clone()
    for _ in range(5):
        step.run(w)
        torch.cuda.synchronize()
        assert torch.equal(step.out, out0)
        assert torch.equal(step.lse, lse0)
