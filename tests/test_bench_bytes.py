"""The bench's roofline numerators on CPU: algorithmic bytes per kernel and the
row-tile kernel's useful FLOPs, recounted token by token from the workload and
the oracle's selection (independent loops, no shared helper)."""
import numpy as np

import bench
import oracle
import qsa_workloads as qw


def _recount(w, sel):
    B, R, P, MB = w["batch"], w["rows_per_req"], w["page_size"], w["max_blocks"]
    Hq, Hkv, D, Di = w["num_q_heads"], w["num_kv_heads"], w["head_dim"], w["index_dim"]
    pt, sl, NP = w["page_table"], w["seqlens"], w["num_pages"]
    keys = pages = union = att = 0
    for b in range(B):
        L = min(int(sl[b]), MB * P)
        # every visible token of a valid block of the request, once
        for t in range(L):
            if pt[b, t // P] >= 0:
                keys += 1
        blocks = set()
        for j in range(R):
            n = max(0, min(int(sl[b]) - R + 1 + j, MB * P))
            for beta in sel[b * R + j]:
                if beta < 0:
                    continue
                blocks.add(int(beta))
                if 0 <= pt[b, beta] < NP:
                    att += len([t for t in range(beta * P, beta * P + P) if t < n])
        union += len(blocks)
        for beta in blocks:
            pages += len([t for t in range(beta * P, beta * P + P) if t < L])
    T = B * R
    idx = keys * Di + T * Hq * Di + B * MB * 4 + B * 4
    dec = pages * Hkv * 2 * (D // 2 + D // 16) + T * Hq * (2 * D * 2 + 4) + union * 4
    return idx, dec, 4.0 * D * Hq * att


def _check(case):
    w = qw.to_numpy(qw.make_workload(case, "cpu"))
    sel = oracle.step(w)["sel"]
    wb = dict(w)
    wb["page_table_np"], wb["seqlens_np"] = w["page_table"], w["seqlens"]
    got = bench.algorithmic_bytes(wb, sel)
    idx, dec, flops = _recount(w, sel)
    assert got["index_scores"] == idx
    assert got["sparse_decode"] == dec and got["sparse_prefill"] == dec
    assert got["step"] == idx + dec
    assert got["flops"] == flops


def test_bytes_verify_workload_with_invalid_pages():
    _check(qw.small(qw.WORKLOADS[4], batch=2))


def test_bytes_head_dim_256():
    _check(qw.small(qw.WORKLOADS[5], batch=2))


def test_bytes_and_flops_context_rows():
    _check(qw.WORKLOADS[6].scaled(batch=1, rows_per_req=20, ctx_lo=1300, ctx_hi=1300,
                                max_blocks=21, k=8, window=2))
