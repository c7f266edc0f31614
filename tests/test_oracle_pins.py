"""Pins for the CPU oracle: each test ties the oracle to something other than
itself -- a published table, a library routine (torch's e4m3 decoder, numpy
einsum, float64 SDPA), a closed form, or brute force on tiny inputs.  No GPU.
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle
import qsa_workloads as qw

SENT = np.iinfo(np.int32).min


def _read_golden(golden_dir, name):
    rows = []
    with open(os.path.join(golden_dir, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


# ---------------------------------------------------------------------------
# element decoders
# ---------------------------------------------------------------------------

def test_e2m1_matches_spec_table(golden_dir):
    rows = _read_golden(golden_dir, "e2m1_values.txt")
    assert len(rows) == 16
    for line in rows:
        code, val = line.split()
        got = oracle.e2m1(int(code))
        assert got == float(val)
        assert math.copysign(1.0, got) == math.copysign(1.0, float(val))


def test_e4m3_matches_spec_points(golden_dir):
    for line in _read_golden(golden_dir, "e4m3_points.txt"):
        byte, val = line.split()
        got = oracle.e4m3(int(byte, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val)
            assert math.copysign(1.0, got) == math.copysign(1.0, float(val))


def test_e4m3_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).tolist()
    for b in range(256):
        got = oracle.e4m3(b)
        if math.isnan(ref[b]):
            assert math.isnan(got), b
        else:
            assert got == ref[b], (b, got, ref[b])


def test_e2m1_times_e4m3_exact_in_fp16_and_bf16():
    # Every product of an e2m1 value and a finite e4m3 value is exactly
    # representable in fp16 and in bf16 (the GPU path dequantises into them).
    e2 = [oracle.e2m1(c) for c in range(16)]
    e4 = [oracle.e4m3(b) for b in range(256) if not math.isnan(oracle.e4m3(b))]
    prods = torch.tensor([a * s for a in e2 for s in e4], dtype=torch.float64)
    assert torch.equal(prods.to(torch.float16).to(torch.float64), prods)
    assert torch.equal(prods.to(torch.bfloat16).to(torch.float64), prods)


# ---------------------------------------------------------------------------
# NVFP4 encoder of the workload generator, checked against the oracle decoders
# ---------------------------------------------------------------------------

def _decode_np(packed, sf, ts):
    e2 = np.array([oracle.e2m1(c) for c in range(16)])
    e4 = np.array([oracle.e4m3(b) for b in range(256)])
    lo = e2[packed & 15]
    hi = e2[packed >> 4]
    vals = np.stack([lo, hi], axis=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)
    scale = np.repeat(e4[sf], 16, axis=-1)
    return vals * scale * ts


def test_encoder_exact_on_grid():
    rng = np.random.default_rng(5)
    e2pos = np.array([0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    sfs = np.array([448.0, 1.0, 0.015625, 3.5, 96.0, 0.001953125])
    c = 2.0 ** -10
    blocks = []
    for i in range(24):
        s = sfs[i % len(sfs)]
        codes = rng.choice(e2pos, size=16) * rng.choice([-1.0, 1.0], size=16)
        codes[rng.integers(16)] = 6.0 * rng.choice([-1.0, 1.0])   # block amax = 6*s*c
        blocks.append(codes * s * c)
    x = torch.tensor(np.concatenate(blocks).reshape(3, 128), dtype=torch.float32)
    packed, sf, ts = qw.nvfp4_encode(x)
    assert ts == c
    got = _decode_np(packed.numpy(), sf.numpy(), ts)
    np.testing.assert_array_equal(got, x.numpy().astype(np.float64))


def test_encoder_recipe_and_error_bound():
    g = torch.Generator().manual_seed(3)
    x = torch.randn((4, 2, 64, 128), generator=g).to(torch.bfloat16)
    packed, sf, ts = qw.nvfp4_encode(x)
    xf = x.float()
    assert ts == pytest.approx(float(xf.abs().max()) / (6 * 448), rel=1e-7)
    bam = xf.reshape(4, 2, 64, 8, 16).abs().amax(-1)
    want_sf = (bam / 6.0 / torch.tensor(ts, dtype=torch.float32)).clamp(max=448).to(
        torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(sf, want_sf)
    deq = _decode_np(packed.numpy(), sf.numpy(), ts)
    sfv = np.repeat(np.array([oracle.e4m3(b) for b in range(256)])[sf.numpy()], 16, -1) * ts
    err = np.abs(deq - xf.numpy().astype(np.float64))
    # Largest e2m1 grid gap is 2 (between 4 and 6): RNE error <= 1 scale unit,
    # plus the fp32 rounding of x / scale inside the encoder.
    assert np.all(err <= sfv * (1.0 + 1e-6))


# ---------------------------------------------------------------------------
# A1 index scores
# ---------------------------------------------------------------------------

def _tiny_case(R=1, invalid=0.0, P=64, Hq=4, Hkv=2, B=2, lo=300, hi=333, k=4, W=1, D=128):
    mb = -(-hi // P)
    return qw.Case("pin", seed=11, batch=B, rows_per_req=R, num_q_heads=Hq,
                   num_kv_heads=Hkv, page_size=P, ctx_lo=lo, ctx_hi=hi, k=k,
                   window=W, max_blocks=mb, pool="perm", invalid_frac=invalid, head_dim=D)


def test_index_scores_closed_form():
    # iq[r, h, :] = c_rh (constant over d); ik[p, tau, :] = e_0 * key(p, tau).
    # Then the token score is (sum_h c_rh) * key, and the block score is the
    # max of that over the block's visible tokens.
    case = _tiny_case(R=3, B=2, lo=200, hi=230, P=64, Hq=4)
    w = qw.to_numpy(qw.make_workload(case, "cpu"))
    T, Hq, Di = w["iq"].shape
    rng = np.random.default_rng(0)
    c = rng.integers(-20, 21, size=(T, Hq)).astype(np.int8)
    c[0] = 3                                     # row 0: positive total
    c[1] = -2                                    # row 1: negative total
    w["iq"] = np.repeat(c[:, :, None], Di, axis=2).astype(np.int8)
    NP, P, _ = w["ik_pool"].shape
    key = ((np.arange(NP)[:, None] * 7 + np.arange(P)[None, :] * 3) % 200 - 100).astype(np.int8)
    ik = np.zeros((NP, P, Di), dtype=np.int8)
    ik[:, :, 0] = key
    w["ik_pool"] = ik
    got = oracle.index_scores(w)
    R, MB = w["rows_per_req"], w["max_blocks"]
    for r in range(T):
        b, j = divmod(r, R)
        n = max(0, min(int(w["seqlens"][b]) - R + 1 + j, MB * P))
        C = int(c[r].astype(np.int64).sum())
        for beta in range(MB):
            page = int(w["page_table"][b, beta])
            vis = [tau for tau in range(P) if beta * P + tau < n]
            if page < 0 or not vis:
                assert got[r, beta] == SENT
            else:
                assert got[r, beta] == max(C * int(key[page, tau]) for tau in vis)


def test_index_scores_match_einsum():
    case = _tiny_case(R=4, invalid=0.2, B=3, lo=250, hi=400, Hq=8, Hkv=2)
    w = qw.to_numpy(qw.make_workload(case, "cpu"))
    got = oracle.index_scores(w)
    R, P, MB = w["rows_per_req"], w["page_size"], w["max_blocks"]
    pt = w["page_table"]
    for r in range(w["iq"].shape[0]):
        b, j = divmod(r, R)
        n = max(0, min(int(w["seqlens"][b]) - R + 1 + j, MB * P))
        pages = np.where(pt[b] >= 0, pt[b], 0)
        keys = w["ik_pool"][pages].astype(np.int64)            # [MB, P, Di]
        tok = np.einsum("hd,btd->bt", w["iq"][r].astype(np.int64), keys)
        pos = np.arange(MB)[:, None] * P + np.arange(P)[None, :]
        tok = np.where(pos < n, tok, np.iinfo(np.int64).min)
        want = tok.max(axis=1)
        want = np.where((pt[b] < 0) | (np.arange(MB) * P >= n), SENT, want)
        np.testing.assert_array_equal(got[r], want.astype(np.int32))


def test_index_scores_zero_keys_and_bound():
    case = _tiny_case(R=1)
    w = qw.to_numpy(qw.make_workload(case, "cpu"))
    w["ik_pool"] = np.zeros_like(w["ik_pool"])
    got = oracle.index_scores(w)
    assert np.all((got == 0) | (got == SENT))
    # The largest magnitude the definition can reach fits int32.
    assert 64 * 64 * 127 * 127 < 2 ** 31 - 1


# ---------------------------------------------------------------------------
# A2 canonical selection
# ---------------------------------------------------------------------------

def _brute_select(scores_row, n, P, k, W):
    """Brute force: the unique candidate subset of the right size whose every
    member outranks every non-member under (score, block index)."""
    nb = -(-n // P)
    valid = [b for b in range(nb) if scores_row[b] != SENT]
    window = [b for b in valid if b >= nb - W]
    cand = [b for b in valid if b < nb - W]
    take = min(k - len(window), len(cand))
    key = lambda b: (int(scores_row[b]), b)
    found = []
    for sub in itertools.combinations(cand, take):
        rest = [b for b in cand if b not in sub]
        if all(key(x) > key(y) for x in sub for y in rest):
            found.append(sub)
    assert len(found) == 1
    return sorted(window + list(found[0]))


def _select_one(scores_row, seqlen, R, j, P, k, W):
    MB = len(scores_row)
    w = dict(batch=1, rows_per_req=R, num_q_heads=1, num_kv_heads=1, head_dim=128,
             index_dim=64, page_size=P, max_blocks=MB, num_pages=1, k=k, window=W,
             seqlens=np.array([seqlen], dtype=np.int32))
    sc = np.full((R, MB), SENT, dtype=np.int32)
    sc[j] = scores_row
    sel, nsel = oracle.select(w, sc)
    return sel[j], nsel[j]


def test_select_worked_examples(golden_dir):
    for line in _read_golden(golden_dir, "select_worked_examples.txt"):
        head, sc, want, nsel = [x.strip() for x in line.split("|")]
        P, L, R, j, k, W = map(int, head.split())
        scores = np.array([SENT if t == "x" else int(t) for t in sc.split()], dtype=np.int32)
        want = [int(t) for t in want.split()]
        want = want + [-1] * (k - len(want))
        got, gn = _select_one(scores, L, R, j, P, k, W)
        assert got.tolist() == want, line
        assert gn == int(nsel), line


def test_select_matches_brute_force():
    rng = np.random.default_rng(7)
    P = 4
    for trial in range(400):
        MB = int(rng.integers(1, 13))
        R = int(rng.integers(1, 4))
        j = int(rng.integers(0, R))
        L = int(rng.integers(0, MB * P + 1)) + R - 1 - j
        n = max(0, min(L - R + 1 + j, MB * P))
        scores = rng.integers(-3, 4, size=MB).astype(np.int32)    # many ties
        scores[rng.random(MB) < 0.25] = SENT
        nb = -(-n // P)
        scores[nb:] = SENT if rng.random() < 0.5 else scores[nb:]
        k = int(rng.integers(1, MB + 2))
        W = int(rng.integers(0, k + 1))
        got, gn = _select_one(scores, L, R, j, P, k, W)
        want = _brute_select(scores, n, P, k, W)
        assert got.tolist() == want + [-1] * (k - len(want)), (scores, L, R, j, k, W)
        assert gn == len(want)


def test_select_properties_on_generated_case():
    case = qw.small(qw.WORKLOADS[4], batch=4)
    w = qw.to_numpy(qw.make_workload(case, "cpu"))
    sc = oracle.index_scores(w)
    sel, nsel = oracle.select(w, sc)
    R, P, k, W, MB = w["rows_per_req"], w["page_size"], w["k"], w["window"], w["max_blocks"]
    for r in range(sel.shape[0]):
        b, j = divmod(r, R)
        n = max(0, min(int(w["seqlens"][b]) - R + 1 + j, MB * P))
        nb = -(-n // P)
        valid = [beta for beta in range(nb) if w["page_table"][b, beta] >= 0]
        s = sel[r][: nsel[r]].tolist()
        assert nsel[r] == min(k, len(valid))
        assert s == sorted(set(s))
        assert all(x in valid for x in s)                       # no invalid page
        assert all(x in s for x in valid if x >= nb - W)       # window kept
        assert np.all(sel[r][nsel[r]:] == -1)


# ---------------------------------------------------------------------------
# A3 attention
# ---------------------------------------------------------------------------

def _dense_kv(w, golden_dir):
    """Dense float64 K/V [NP, Hkv, P, D] from the page bytes, decoded without the
    oracle: e2m1 from the spec table, e4m3 through torch."""
    table = {}
    for line in _read_golden(golden_dir, "e2m1_values.txt"):
        c, v = line.split()
        table[int(c)] = float(v)
    e2 = torch.tensor([table[c] for c in range(16)], dtype=torch.float64)

    def dec(pool, sf, ts):
        p = torch.from_numpy(pool.astype(np.int64))
        codes = torch.stack([p & 15, p >> 4], dim=-1).reshape(*p.shape[:-1], p.shape[-1] * 2)
        s = torch.from_numpy(sf).view(torch.float8_e4m3fn).to(torch.float64)
        return e2[codes] * s.repeat_interleave(16, dim=-1) * ts

    return dec(w["k_pool"], w["k_sf"], w["k_scale"]), dec(w["v_pool"], w["v_sf"], w["v_scale"])


def _sdpa_reference(w, golden_dir):
    K, V = _dense_kv(w, golden_dir)
    q = torch.from_numpy(w["q"].astype(np.int32) << 16).view(torch.float32).to(torch.float64)
    B, R, Hq, Hkv = w["batch"], w["rows_per_req"], w["num_q_heads"], w["num_kv_heads"]
    P, MB, D = w["page_size"], w["max_blocks"], w["head_dim"]
    G = Hq // Hkv
    T = B * R
    out = torch.zeros((T, Hq, D), dtype=torch.float64)
    lse = torch.full((T, Hq), -math.inf, dtype=torch.float64)
    for r in range(T):
        b, j = divmod(r, R)
        n = max(0, min(int(w["seqlens"][b]) - R + 1 + j, MB * P))
        ks, vs = [], []
        for beta in range(-(-n // P)):
            page = int(w["page_table"][b, beta])
            if page < 0:
                continue
            m = min(P, n - beta * P)
            ks.append(K[page, :, :m])
            vs.append(V[page, :, :m])
        if not ks:
            continue
        Kr = torch.cat(ks, dim=1).repeat_interleave(G, dim=0)    # [Hq, N, D]
        Vr = torch.cat(vs, dim=1).repeat_interleave(G, dim=0)
        qr = q[r].unsqueeze(1)                                   # [Hq, 1, D]
        o = torch.nn.functional.scaled_dot_product_attention(
            qr.unsqueeze(0), Kr.unsqueeze(0), Vr.unsqueeze(0), scale=w["sm_scale"])
        out[r] = o[0, :, 0]
        lse[r] = torch.logsumexp((qr @ Kr.transpose(1, 2))[:, 0] * w["sm_scale"], dim=-1)
    return out.numpy(), lse.numpy()


@pytest.mark.parametrize("R,Hq,Hkv,P,invalid,D", [(1, 8, 2, 64, 0.0, 128), (4, 4, 2, 64, 0.15, 128),
                                                   (2, 6, 3, 128, 0.1, 128),
                                                   (4, 12, 1, 32, 0.1, 256), (1, 6, 2, 64, 0.0, 256)])
def test_attention_dense_when_k_covers_all(golden_dir, R, Hq, Hkv, P, invalid, D):
    hi = 2 * P + 70 if P >= 64 else 6 * P + 10      # several blocks, a ragged tail
    case = _tiny_case(R=R, invalid=invalid, P=P, Hq=Hq, Hkv=Hkv, B=2, lo=150, hi=hi,
                      k=16, W=2, D=D)
    w = qw.to_numpy(qw.make_workload(case, "cpu"))
    res = oracle.step(w)
    out_ref, lse_ref = _sdpa_reference(w, golden_dir)
    np.testing.assert_allclose(res["out"], out_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(res["lse"], lse_ref, rtol=1e-12, atol=1e-12)


def _small_attn_case(**kw):
    case = _tiny_case(**kw)
    return qw.to_numpy(qw.make_workload(case, "cpu"))


def test_attention_constant_v_and_single_token():
    w = _small_attn_case(R=1, B=1, lo=130, hi=130, k=3, W=1)
    # V codes all e2m1 1.0 (0x2) and scales 1.0 (0x38): out = v_scale exactly.
    w["v_pool"] = np.full_like(w["v_pool"], 0x22)
    w["v_sf"] = np.full_like(w["v_sf"], 0x38)
    res = oracle.step(w)
    np.testing.assert_allclose(res["out"], w["v_scale"], rtol=1e-14)
    # Single visible token in one selected block: out = V of that token, lse = z.
    w2 = _small_attn_case(R=1, B=1, lo=1, hi=1, k=1, W=1)
    res2 = oracle.step(w2)
    assert res2["nsel"][0] == 1
    K, V = _dense_kv(w2, os.path.join(os.path.dirname(__file__), "golden"))
    page = int(w2["page_table"][0, 0])
    G = w2["num_q_heads"] // w2["num_kv_heads"]
    q = (w2["q"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for h in range(w2["num_q_heads"]):
        g = h // G
        np.testing.assert_allclose(res2["out"][0, h], V[page, g, 0].numpy(), rtol=1e-14)
        z = w2["sm_scale"] * float(q[0, h] @ K[page, g, 0].numpy())
        assert res2["lse"][0, h] == pytest.approx(z, rel=1e-12, abs=1e-12)


def test_attention_empty_row():
    w = _small_attn_case(R=4, B=1, lo=2, hi=2, k=2, W=1)
    res = oracle.step(w)
    # Rows 0 and 1 of 4 see L - R + 1 + j = -1, 0 tokens.
    for r in (0, 1):
        assert res["nsel"][r] == 0
        assert np.all(res["out"][r] == 0.0)
        assert np.all(np.isneginf(res["lse"][r]))
    assert res["nsel"][2] == 1 and np.all(np.isfinite(res["lse"][2]))


def test_attention_lse_merge_of_two_halves():
    w = _small_attn_case(R=2, B=2, lo=600, hi=700, k=8, W=2)
    res = oracle.step(w)
    sel = res["sel"]
    a = np.where(np.arange(sel.shape[1]) % 2 == 0, sel, -1).astype(np.int32)
    b = np.where(np.arange(sel.shape[1]) % 2 == 1, sel, -1).astype(np.int32)
    oa, la = oracle.attention(w, a)
    ob, lb = oracle.attention(w, b)
    m = np.maximum(la, lb)
    L = m + np.log(np.exp(la - m) + np.exp(lb - m))
    o = (np.exp(la - L)[..., None] * oa + np.exp(lb - L)[..., None] * ob)
    np.testing.assert_allclose(L, res["lse"], rtol=1e-13)
    np.testing.assert_allclose(o, res["out"], rtol=1e-11, atol=1e-13)


def test_step_invariant_under_page_permutation():
    w = _small_attn_case(R=2, B=2, lo=400, hi=520, k=4, W=1, invalid=0.1)
    res = oracle.step(w)
    NP = w["num_pages"]
    perm = np.random.default_rng(1).permutation(NP)      # new id of old page p = perm[p]
    w2 = dict(w)
    for key in ("ik_pool", "k_pool", "k_sf", "v_pool", "v_sf"):
        arr = np.empty_like(w[key])
        arr[perm] = w[key]
        w2[key] = arr
    w2["page_table"] = np.where(w["page_table"] >= 0, perm[np.maximum(w["page_table"], 0)],
                                -1).astype(np.int32)
    res2 = oracle.step(w2)
    for key in ("scores", "sel", "nsel", "out", "lse"):
        np.testing.assert_array_equal(res[key], res2[key])


# ---------------------------------------------------------------------------
# decode prologue: the NVFP4 quantiser and the token store
# ---------------------------------------------------------------------------

def test_e4m3_encode_round_trips_every_finite_code():
    for c in range(0x7F):                       # 0x7F is NaN
        assert oracle.e4m3_encode(oracle.e4m3(c)) == c


def test_e4m3_encode_midpoints_go_to_the_even_code():
    for c in range(0x7E):
        lo, hi = oracle.e4m3(c), oracle.e4m3(c + 1)
        mid = (lo + hi) / 2                      # exact in fp32 (5 significant bits)
        assert oracle.e4m3_encode(mid) == (c if c % 2 == 0 else c + 1)
        assert oracle.e4m3_encode(np.nextafter(np.float32(mid), np.float32(0))) == c
        assert oracle.e4m3_encode(np.nextafter(np.float32(mid), np.float32(1e9))) == c + 1


def test_e4m3_encode_saturates_and_flushes():
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(1e30) == 0x7E
    assert oracle.e4m3_encode(0.0) == 0
    assert oracle.e4m3_encode(2.0 ** -10) == 0    # half the smallest subnormal: tie to 0
    assert oracle.e4m3_encode(2.0 ** -10 * 1.0001) == 1


def test_e4m3_encode_matches_torch_float8_cast():
    rng = np.random.default_rng(5)
    v = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(448.0), 4000)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_encode(float(x)) for x in v], dtype=np.uint8)
    np.testing.assert_array_equal(got, ref)


def test_e2m1_encode_from_the_definition():
    mags = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for c, m in enumerate(mags):
        assert oracle.e2m1_encode(m) == c
        if c:
            assert oracle.e2m1_encode(-m) == c | 8
    # midpoints between neighbours go to the even code
    for (a, b), want in zip(zip(mags, mags[1:]), [0, 2, 2, 4, 4, 6, 6]):
        assert oracle.e2m1_encode((a + b) / 2) == want
    assert oracle.e2m1_encode(7.5) == 7 and oracle.e2m1_encode(1e9) == 7
    assert oracle.e2m1_encode(-1e9) == 15
    assert oracle.e2m1_encode(-0.2) == 0        # rounds to zero: stored as +0
    assert oracle.e2m1_encode(-0.3) == 9


def test_quantize_block_round_trips_grid_values():
    rng = np.random.default_rng(6)
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    for _ in range(300):
        scale = 2.0 ** int(rng.integers(-8, 3))
        sf = int(rng.integers(0x08, 0x7E))      # a normal e4m3 scale
        codes = rng.integers(1, 16, 16)
        codes[codes == 8] = 1                   # no -0
        codes[int(rng.integers(0, 16))] = 7 | (8 if rng.random() < 0.5 else 0)  # |x|max = 6
        x = np.array([(-1 if c & 8 else 1) * mags[c & 7] for c in codes]) * oracle.e4m3(sf) * scale
        got_codes, got_sf = oracle.quantize_block(x.astype(np.float32), scale)
        assert got_sf == sf
        np.testing.assert_array_equal(got_codes, codes)


def test_quantize_block_zero_and_underflow():
    codes, sf = oracle.quantize_block(np.zeros(16, np.float32), 0.5)
    assert sf == 0 and not codes.any()
    x = np.full(16, 1e-6, np.float32)
    codes, sf = oracle.quantize_block(x, 1.0)    # (1e-6 / 6) / 1 is below half of 2^-9
    assert sf == 0 and not codes.any()


def test_quantize_matches_the_generators_encoder():
    # The input generator's torch encoder (midpoint thresholds + torch's
    # float8 cast) is an independent implementation of the same recipe.
    g = torch.Generator().manual_seed(7)
    x = torch.randn((64, 128), generator=g).to(torch.bfloat16).float()
    packed, sfs, ts = qw.nvfp4_encode(x)
    for r in range(64):
        for blk in range(8):
            codes, sf = oracle.quantize_block(x[r, 16 * blk:16 * blk + 16].numpy(), ts)
            assert sf == int(sfs[r, blk])
            np.testing.assert_array_equal(codes[0::2] | (codes[1::2] << 4),
                                          packed[r, 8 * blk:8 * blk + 8].numpy())


@pytest.mark.parametrize("cfg", [2, 4, 5])
def test_store_kv_writes_exactly_the_new_slots(cfg):
    w = qw.to_numpy(qw.make_workload(qw.small(qw.WORKLOADS[cfg]), "cpu"))
    new = qw.to_numpy(qw.make_new_tokens(qw.make_workload(qw.small(qw.WORKLOADS[cfg]), "cpu")))
    out = oracle.store_kv(w, new)
    B, R, P, MB, Hkv = w["batch"], w["rows_per_req"], w["page_size"], w["max_blocks"], w["num_kv_heads"]
    D = w["head_dim"]
    rows = np.zeros((w["num_pages"], Hkv, P), bool)
    keys = np.zeros((w["num_pages"], P), bool)
    for b in range(B):
        for j in range(R):
            pos = int(w["seqlens"][b]) - R + j
            if pos < 0 or pos >= MB * P:
                continue
            page = int(w["page_table"][b, pos // P])
            if page < 0 or page >= w["num_pages"]:
                continue
            rows[page, :, pos % P] = True
            keys[page, pos % P] = True
            # the stored row decodes to the quantised new values
            for g in range(Hkv):
                xk = new["k_new"][b * R + j, g].astype(np.uint32) << 16
                xk = xk.view(np.float32)
                for blk in range(D // 16):
                    codes, sf = oracle.quantize_block(xk[16 * blk:16 * blk + 16], w["k_scale"])
                    assert out["k_sf"].reshape(-1, Hkv, P, D // 16)[page, g, pos % P, blk] == sf
                    np.testing.assert_array_equal(
                        out["k_pool"].reshape(-1, Hkv, P, D // 2)[page, g, pos % P,
                                                                   8 * blk:8 * blk + 8],
                        codes[0::2] | (codes[1::2] << 4))
            np.testing.assert_array_equal(out["ik_pool"].reshape(-1, P, 64)[page, pos % P],
                                          new["ik_new"][b * R + j])
    for name, mask in (("k_pool", rows), ("v_pool", rows), ("k_sf", rows), ("v_sf", rows),
                       ("ik_pool", keys)):
        before = w[name].reshape(mask.shape + (-1,))
        after = out[name].reshape(mask.shape + (-1,))
        np.testing.assert_array_equal(after[~mask], before[~mask])
    assert rows.any()


# ---------------------------------------------------------------------------
# speculative rollback of the cache planes
# ---------------------------------------------------------------------------

def _half_rejected(T):
    # exactly half the rows rejected, interleaved (kept and rejected both occur)
    return (np.arange(T) % 2 == 1).astype(np.int32)


@pytest.mark.parametrize("cfg", [2, 4, 5])
def test_rollback_round_trip(cfg):
    w = qw.to_numpy(qw.make_workload(qw.small(qw.WORKLOADS[cfg]), "cpu"))
    new = qw.to_numpy(qw.make_new_tokens(qw.make_workload(qw.small(qw.WORKLOADS[cfg]), "cpu")))
    names = ("k_pool", "k_sf", "v_pool", "v_sf", "ik_pool")
    saved = oracle.rollback_gather(w, w)
    stored = oracle.store_kv(w, new)
    T = w["batch"] * w["rows_per_req"]
    # every row rejected: the cache is back to what it was, byte for byte
    back = oracle.rollback_restore(w, stored, np.ones(T, np.int32), saved)
    for n in names:
        np.testing.assert_array_equal(back[n], w[n])
    # no row rejected: the step's stores stay
    keep = oracle.rollback_restore(w, stored, np.zeros(T, np.int32), saved)
    for n in names:
        np.testing.assert_array_equal(keep[n], stored[n])
    # half rejected: exactly the rejected rows' slots go back
    rej = _half_rejected(T)
    mixed = oracle.rollback_restore(w, stored, rej, saved)
    # slots of rejected rows equal the original, those of kept rows the store
    rows_rej = np.zeros(T, bool)
    rows_rej[rej == 1] = True
    P, R, Hkv, D = w["page_size"], w["rows_per_req"], w["num_kv_heads"], w["head_dim"]
    for r in range(T):
        b, j = divmod(r, R)
        pos = int(w["seqlens"][b]) - R + j
        if pos < 0 or pos >= w["max_blocks"] * P:
            continue
        page = int(w["page_table"][b, pos // P])
        if page < 0 or page >= w["num_pages"]:
            continue
        want = w if rows_rej[r] else stored
        kp = mixed["k_pool"].reshape(-1, Hkv, P, D // 2)[page, :, pos % P]
        np.testing.assert_array_equal(kp, want["k_pool"].reshape(-1, Hkv, P, D // 2)[page, :, pos % P])
        ik = mixed["ik_pool"].reshape(-1, P, 64)[page, pos % P]
        np.testing.assert_array_equal(ik, want["ik_pool"].reshape(-1, P, 64)[page, pos % P])
    assert rows_rej.any() and (~rows_rej).any()


@pytest.mark.parametrize("cfg", [2, 5])
def test_rollback_saved_layout(cfg):
    # the saved bytes of a row are its slots' bytes in the documented order
    w = qw.to_numpy(qw.make_workload(qw.small(qw.WORKLOADS[cfg]), "cpu"))
    saved = oracle.rollback_gather(w, w)
    Hkv, P, R, D = w["num_kv_heads"], w["page_size"], w["rows_per_req"], w["head_dim"]
    c, f = D // 2, D // 16            # code and scale bytes per token row
    per = 2 * (c + f)
    row_bytes = Hkv * per + 64
    b, j = 1, 2
    r = b * R + j
    pos = int(w["seqlens"][b]) - R + j
    page = int(w["page_table"][b, pos // P])
    s = saved[r * row_bytes:(r + 1) * row_bytes]
    for g in range(Hkv):
        part = s[g * per:(g + 1) * per]
        np.testing.assert_array_equal(part[:c], w["k_pool"].reshape(-1, Hkv, P, c)[page, g, pos % P])
        np.testing.assert_array_equal(part[c:c + f], w["k_sf"].reshape(-1, Hkv, P, f)[page, g, pos % P])
        np.testing.assert_array_equal(part[c + f:2 * c + f],
                                      w["v_pool"].reshape(-1, Hkv, P, c)[page, g, pos % P])
        np.testing.assert_array_equal(part[2 * c + f:per],
                                      w["v_sf"].reshape(-1, Hkv, P, f)[page, g, pos % P])
    np.testing.assert_array_equal(s[Hkv * per:].view(np.int8),
                                  w["ik_pool"].reshape(-1, P, 64)[page, pos % P])


# ---------------------------------------------------------------------------
# context row groups reduce to single rows
# ---------------------------------------------------------------------------

def test_row_group_rows_equal_single_rows():
    # Row j of a request with R rows and L cached tokens sees L - R + 1 + j
    # tokens; scored, selected and attended alone (one row, that length) it
    # must give exactly the same scores, selection and outputs.
    case = _tiny_case(R=24, B=1, lo=1500, hi=1500, P=64, Hq=4, Hkv=2, k=6, W=2)
    w = qw.to_numpy(qw.make_workload(case, "cpu"))
    ref = oracle.step(w)
    R, L = w["rows_per_req"], int(w["seqlens"][0])
    for j in (0, 1, 11, R - 2, R - 1):
        w1 = dict(w)
        w1["rows_per_req"] = 1
        w1["seqlens"] = np.array([L - R + 1 + j], dtype=np.int32)
        w1["q"] = w["q"][j:j + 1]
        w1["iq"] = w["iq"][j:j + 1]
        one = oracle.step(w1)
        np.testing.assert_array_equal(one["scores"][0], ref["scores"][j])
        np.testing.assert_array_equal(one["sel"][0], ref["sel"][j])
        np.testing.assert_array_equal(one["nsel"][0], ref["nsel"][j])
        np.testing.assert_array_equal(one["out"][0], ref["out"][j])
        np.testing.assert_array_equal(one["lse"][0], ref["lse"][j])
