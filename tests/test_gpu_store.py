"""GPU parity of the decode prologue (qsa_store_kv_tokens) against the oracle.

Every byte of every pool must match the oracle (stored codes, scales and index
keys, and the untouched remainder), so the quantiser's rounding decisions are
checked one by one.  A last test stores a step's tokens and then runs the
step on the updated cache, against the oracle on the oracle's updated cache.
"""
import numpy as np
import pytest
import torch

import oracle
import qsa_workloads as qw

pytestmark = pytest.mark.gpu

POOLS = ("k_pool", "k_sf", "v_pool", "v_sf", "ik_pool")


@pytest.fixture(scope="module")
def qsa():
    import nvfp4_block_sparse_gb300 as m
    m.load(build_if_missing=True)
    return m


def store_gpu(qsa, w, new):
    pools = {n: w[n].clone() for n in POOLS}
    qsa.qsa_store_kv_tokens(qw.geometry(w), new["k_new"], new["v_new"], new["ik_new"],
                            w["k_scale"], w["v_scale"], w["page_table"], w["seqlens"],
                            pools["k_pool"], pools["k_sf"], pools["v_pool"], pools["v_sf"],
                            pools["ik_pool"])
    torch.cuda.synchronize()
    return pools


def check_store(qsa, w, new):
    got = store_gpu(qsa, w, new)
    ref = oracle.store_kv(qw.to_numpy(w), qw.to_numpy(new))
    for n in POOLS:
        np.testing.assert_array_equal(got[n].cpu().numpy(), ref[n], err_msg=n)
    return got


@pytest.mark.parametrize("cfg", range(len(qw.WORKLOADS)))
def test_store_small_configs(qsa, cfg):
    w = qw.make_workload(qw.small(qw.WORKLOADS[cfg]), "cuda")
    check_store(qsa, w, qw.make_new_tokens(w))


@pytest.mark.parametrize("cfg", [1, 4, 5])
def test_store_full_size(qsa, cfg):
    w = qw.make_workload(qw.WORKLOADS[cfg], "cuda")
    check_store(qsa, w, qw.make_new_tokens(w))


def _case(**kw):
    base = dict(name="edge", seed=31, batch=3, rows_per_req=1, num_q_heads=8, num_kv_heads=2,
                page_size=64, ctx_lo=700, ctx_hi=1300, k=6, window=2, max_blocks=21,
                pool="perm")
    base.update(kw)
    return qw.Case(**base)


STORE_CASES = {
    "p128_verify": _case(page_size=128, rows_per_req=4, ctx_lo=129, ctx_hi=2600),
    "tiny_contexts_verify": _case(rows_per_req=4, ctx_lo=1, ctx_hi=6, max_blocks=2, k=2, window=1),
    "mostly_invalid": _case(invalid_frac=0.9, rows_per_req=3),
    "eight_rows_one_kv_head": _case(rows_per_req=8, num_q_heads=4, num_kv_heads=1, k=5),
    "hd256_p32_verify": _case(head_dim=256, page_size=32, max_blocks=41, rows_per_req=4,
                              num_q_heads=24, num_kv_heads=2),
    "hd256_p64_tiny": _case(head_dim=256, rows_per_req=4, ctx_lo=1, ctx_hi=6, max_blocks=2,
                            k=2, window=1),
}


@pytest.mark.parametrize("name", sorted(STORE_CASES))
def test_store_edge_cases(qsa, name):
    w = qw.make_workload(STORE_CASES[name], "cuda")
    check_store(qsa, w, qw.make_new_tokens(w))


@pytest.mark.parametrize("mult,cfg", [(1e4, 2), (1e-7, 2), (0.0, 2), (1e4, 5), (1e-7, 5)])
def test_store_saturation_underflow_and_zeros(qsa, mult, cfg):
    # Values far above the tensor scale saturate the block scale (448) and
    # the codes (6); values far below it flush the block to zero.
    w = qw.make_workload(qw.small(qw.WORKLOADS[cfg]), "cuda")
    new = qw.make_new_tokens(w)
    new["k_new"] = (new["k_new"].float() * mult).to(torch.bfloat16)
    new["v_new"] = (new["v_new"].float() * mult).to(torch.bfloat16)
    check_store(qsa, w, new)


@pytest.mark.parametrize("cfg", [2, 5])
def test_store_then_step_matches_the_oracle(qsa, cfg):
    w = qw.make_workload(qw.small(qw.WORKLOADS[cfg]), "cuda")
    new = qw.make_new_tokens(w)
    got = store_gpu(qsa, w, new)
    for n in POOLS:
        w[n] = got[n]
    step = qsa.DecodeStep(qw.geometry(w), w["k"], w["window"], device=w["q"].device)
    step.run(w)
    torch.cuda.synchronize()
    assert step.status() == 0
    ref = oracle.step(qw.to_numpy(w))
    np.testing.assert_array_equal(step.scores.cpu().numpy(), ref["scores"])
    np.testing.assert_array_equal(step.sel.cpu().numpy(), ref["sel"])
    out = step.out.float().cpu().numpy().astype(np.float64)
    assert np.abs(out - ref["out"]).max() <= 1e-2
    lse = step.lse.cpu().numpy().astype(np.float64)
    fin = np.isfinite(ref["lse"])
    assert np.abs(lse[fin] - ref["lse"][fin]).max() <= 1e-3


# ---------------------------------------------------------------------------
# speculative rollback: gather before the store, restore the rejected rows
# ---------------------------------------------------------------------------

def gather_gpu(qsa, w, pools):
    saved = torch.zeros(qsa.qsa_rollback_state_bytes(qw.geometry(w)), dtype=torch.uint8,
                        device=w["q"].device)
    qsa.qsa_rollback_gather(qw.geometry(w), w["page_table"], w["seqlens"], pools["k_pool"],
                            pools["k_sf"], pools["v_pool"], pools["v_sf"], pools["ik_pool"], saved)
    return saved


def restore_gpu(qsa, w, pools, rejected, saved):
    qsa.qsa_rollback_restore(qw.geometry(w), w["page_table"], w["seqlens"], rejected, saved,
                             pools["k_pool"], pools["k_sf"], pools["v_pool"], pools["v_sf"],
                             pools["ik_pool"])
    torch.cuda.synchronize()


ROLLBACK_CASES = [("cfg2", lambda: qw.small(qw.WORKLOADS[2])), ("cfg4", lambda: qw.small(qw.WORKLOADS[4])),
                  ("tiny", lambda: STORE_CASES["tiny_contexts_verify"]),
                  ("invalid", lambda: STORE_CASES["mostly_invalid"]),
                  ("full4", lambda: qw.WORKLOADS[4]),
                  ("cfg5", lambda: qw.small(qw.WORKLOADS[5])),
                  ("hd256_tiny", lambda: STORE_CASES["hd256_p64_tiny"])]


@pytest.mark.parametrize("name,make", ROLLBACK_CASES, ids=[c[0] for c in ROLLBACK_CASES])
def test_rollback_matches_oracle(qsa, name, make):
    w = qw.make_workload(make(), "cuda")
    new = qw.make_new_tokens(w)
    T = w["batch"] * w["rows_per_req"]
    w_np = qw.to_numpy(w)
    saved = gather_gpu(qsa, w, {n: w[n] for n in POOLS})
    torch.cuda.synchronize()
    ref_saved = oracle.rollback_gather(w_np, w_np)
    # bytes of rows without a slot stay as allocated (zero) on both sides
    np.testing.assert_array_equal(saved.cpu().numpy(), ref_saved)
    stored = store_gpu(qsa, w, new)
    ref_stored = oracle.store_kv(w_np, qw.to_numpy(new))
    for rej_np in (np.ones(T, np.int32), np.zeros(T, np.int32),
                   (np.arange(T) % 2 == 1).astype(np.int32)):
        pools = {n: stored[n].clone() for n in POOLS}
        restore_gpu(qsa, w, pools, torch.from_numpy(rej_np).to(w["q"].device), saved)
        ref = oracle.rollback_restore(w_np, ref_stored, rej_np, ref_saved)
        for n in POOLS:
            np.testing.assert_array_equal(pools[n].cpu().numpy(), ref[n], err_msg=n)
        if rej_np.all():
            for n in POOLS:      # everything rejected: the cache is back, byte for byte
                np.testing.assert_array_equal(pools[n].cpu().numpy(), w_np[n], err_msg=n)
