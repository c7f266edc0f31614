"""Seeded synthetic inputs for QSA block-sparse GQA decode / verify over an
NVFP4 paged KV cache.

This module is the one piece shared by the CUDA path's tests and benchmark and
by the CPU oracle's tests: it draws inputs and nothing else.  It computes none
of the path's arithmetic (no index scores, no selection, no attention, no
NVFP4 *decoding*).  It does hold the NVFP4 *encoder* that turns the drawn bf16
K/V into pages, because the workloads are specified as "bf16 N(0,1) quantised
to NVFP4" and the path itself never quantises.

Workloads (TensorRT-LLM PR #20276, "Qwen3.8-Flash-Next NVFP4 target", Features
table: NVFP4 KV cache = uint8 e2m1 pages + e4m3 block scales, QSA side planes
addressed by the same page index):

* ``q``          bf16  [T, Hq, D]         T = B * R query rows, row r = b*R + j
* ``iq``         int8  [T, Hq, Di]        index query, uniform [-127, 127]
* ``ik_pool``    int8  [NP, P, Di]        index keys, uniform [-127, 127]
* ``k_pool``     uint8 [NP, Hkv, P, D/2]  two e2m1 codes per byte, low nibble =
                                          even element
* ``k_sf``       uint8 [NP, Hkv, P, D/16] one e4m3 scale per 16 elements
* ``v_pool``, ``v_sf``                    same as K
* ``k_scale``, ``v_scale``  python float  fp32 per-tensor dequant multiplier
* ``page_table`` int32 [B, MB]            -1 marks an invalid entry
* ``seqlens``    int32 [B]                tokens in each request's cache,
                                          including its R newest rows

Draw order is fixed: context lengths, q, K, V, iq, ik, page table, invalid
mask, tie duplication.  Every draw comes from one ``torch.Generator`` seeded
with the case's seed on the device the tensors are made on (CPU draws and CUDA
draws of the same seed differ; each test uses one device consistently).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

E2M1_MAX = 6.0
E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class Case:
    """Shape and structure of one synthetic workload."""

    name: str
    seed: int
    batch: int
    rows_per_req: int
    num_q_heads: int
    num_kv_heads: int
    page_size: int
    ctx_lo: int               # context lengths uniform in [ctx_lo, ctx_hi]
    ctx_hi: int
    k: int                    # selection size in blocks, window included
    window: int               # always-kept recent window, in blocks
    max_blocks: int           # MB: page-table row stride
    pool: str = "perm"        # "identity" | "perm"
    pool_pages: Optional[int] = None   # None: exactly the blocks in use
    invalid_frac: float = 0.0
    tie_frac: float = 0.0
    head_dim: int = 128
    index_dim: int = 64
    # 0: every row's index query is drawn independently.  n > 0: one base
    # query per request plus per-row integer noise in [-n, n] (clipped to
    # int8), so that the rows of a context chunk select overlapping blocks.
    iq_row_noise: int = 0

    @property
    def rows(self) -> int:
        return self.batch * self.rows_per_req

    def scaled(self, **kw) -> "Case":
        return dataclasses.replace(self, **kw)


# The workloads the method is measured on: five at head_dim 128, then one in
# the geometry the pages tune their kernels on (24 q / 2 KV heads, head_dim
# 256, 32-token pages, four rows per request as in an MTP-3 verify step).
WORKLOADS = [
    Case("tiny decode", seed=0, batch=1, rows_per_req=1, num_q_heads=8,
         num_kv_heads=1, page_size=64, ctx_lo=4096, ctx_hi=4096, k=16,
         window=2, max_blocks=64, pool="identity"),
    Case("batched decode", seed=1, batch=8, rows_per_req=1, num_q_heads=32,
         num_kv_heads=4, page_size=64, ctx_lo=32768, ctx_hi=32768, k=64,
         window=4, max_blocks=512, pool="perm", pool_pages=4096),
    Case("speculative verify", seed=2, batch=16, rows_per_req=4,
         num_q_heads=64, num_kv_heads=8, page_size=128, ctx_lo=8192,
         ctx_hi=16384, k=32, window=2, max_blocks=128, pool="perm"),
    Case("long-context decode", seed=3, batch=4, rows_per_req=1,
         num_q_heads=32, num_kv_heads=4, page_size=64, ctx_lo=131072,
         ctx_hi=131072, k=64, window=4, max_blocks=2048, pool="perm",
         pool_pages=8192),
    Case("wide aggregated verify", seed=4, batch=48, rows_per_req=4,
         num_q_heads=32, num_kv_heads=4, page_size=64, ctx_lo=4096,
         ctx_hi=32768, k=48, window=4, max_blocks=512, pool="perm",
         invalid_frac=0.05, tie_frac=0.10),
    Case("head_dim-256 verify", seed=5, batch=32, rows_per_req=4,
         num_q_heads=24, num_kv_heads=2, page_size=32, ctx_lo=8192,
         ctx_hi=16384, k=64, window=4, max_blocks=512, pool="perm",
         head_dim=256),
    Case("context prefill", seed=6, batch=2, rows_per_req=512, num_q_heads=32,
         num_kv_heads=4, page_size=64, ctx_lo=32768, ctx_hi=32768, k=64,
         window=4, max_blocks=512, pool="perm", iq_row_noise=24),
    Case("head_dim-256 context prefill", seed=7, batch=4, rows_per_req=256,
         num_q_heads=24, num_kv_heads=2, page_size=32, ctx_lo=16384, ctx_hi=16384,
         k=64, window=4, max_blocks=512, pool="perm", iq_row_noise=24,
         head_dim=256),
]

# Workloads whose rows are context row groups (served by the row-tile path).
PREFILL_WORKLOADS = (6, 7)


def small(case: Case, batch: Optional[int] = None, ctx_lo: Optional[int] = None,
          ctx_hi: Optional[int] = None) -> Case:
    """A reduced copy of ``case`` for oracle-speed tests: same heads, page size,
    k, window and structure; fewer requests and shorter contexts."""
    b = batch if batch is not None else min(case.batch, 3)
    lo = ctx_lo if ctx_lo is not None else min(case.ctx_lo, 40 * case.page_size + 37)
    hi = ctx_hi if ctx_hi is not None else max(lo, min(case.ctx_hi, 48 * case.page_size + 5))
    mb = -(-hi // case.page_size)
    pool_pages = None
    if case.pool == "identity":
        pool_pages = b * mb
    return dataclasses.replace(case, name=case.name + " (small)", batch=b,
                               ctx_lo=lo, ctx_hi=hi, max_blocks=mb,
                               pool_pages=pool_pages)


# ---------------------------------------------------------------------------
# NVFP4 encoder (input preparation only)
# ---------------------------------------------------------------------------

# e2m1 magnitudes in code order 0..7 and the rounding midpoints between them.
_E2M1_MAGS = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
_E2M1_MIDS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def _e2m1_encode(x: torch.Tensor) -> torch.Tensor:
    """Round-to-nearest-even, saturating fp32 -> e2m1 code (uint8 0..15)."""
    a = x.abs().clamp(max=E2M1_MAX)
    code = torch.zeros_like(a, dtype=torch.int32)
    for i, m in enumerate(_E2M1_MIDS):
        above = a > m
        # A tie goes to the even code: code i+1 is even when i is odd.
        if i % 2 == 1:
            above = above | (a == m)
        code += above.to(torch.int32)
    sign = (x < 0) & (code > 0)
    return (code | (sign.to(torch.int32) << 3)).to(torch.uint8)


def _e4m3_encode(x: torch.Tensor) -> torch.Tensor:
    """Round-to-nearest-even, saturating non-negative fp32 -> e4m3 byte."""
    y = x.clamp(min=0.0, max=E4M3_MAX).to(torch.float8_e4m3fn)
    return y.view(torch.uint8)


def _e4m3_value(b: torch.Tensor) -> torch.Tensor:
    return b.view(torch.float8_e4m3fn).to(torch.float32)


def nvfp4_encode(x: torch.Tensor):
    """Quantise ``x`` (last dim a multiple of 16) to NVFP4.

    Returns ``(packed uint8 [..., D/2], scales uint8 [..., D/16], tensor_scale)``
    where the dequantised element is e2m1(code) * e4m3(scale) * tensor_scale.
    Recipe: tensor_scale = amax(|x|) / (6 * 448); block scale =
    e4m3(amax_16 / 6 / tensor_scale); code = e2m1(x / (e4m3(scale) *
    tensor_scale)); a block whose scale is zero encodes as zeros.
    """
    xf = x.to(torch.float32)
    d = xf.shape[-1]
    assert d % 16 == 0
    amax = xf.abs().amax()
    ts = (amax / (E2M1_MAX * E4M3_MAX)).item()
    if ts == 0.0:
        ts = 1.0
    ts_t = torch.tensor(ts, dtype=torch.float32, device=xf.device)
    blocks = xf.reshape(*xf.shape[:-1], d // 16, 16)
    bamax = blocks.abs().amax(dim=-1)
    sf = _e4m3_encode(bamax / E2M1_MAX / ts_t)
    sfv = _e4m3_value(sf) * ts_t
    safe = torch.where(sfv > 0, sfv, torch.ones_like(sfv))
    codes = _e2m1_encode(blocks / safe.unsqueeze(-1))
    codes = torch.where((sfv > 0).unsqueeze(-1), codes, torch.zeros_like(codes))
    codes = codes.reshape(*xf.shape[:-1], d)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).to(torch.uint8)
    return packed.contiguous(), sf.contiguous(), float(ts)


# ---------------------------------------------------------------------------
# Workload generation
# ---------------------------------------------------------------------------

def _uniform_int(gen, lo, hi, shape, device):
    return torch.randint(lo, hi + 1, shape, generator=gen, device=device,
                         dtype=torch.int64)


def make_workload(case: Case, device="cpu", seed: Optional[int] = None) -> dict:
    """Draw every input of ``case`` on ``device``.  ``seed`` overrides the
    case's own seed (benchmark replicas)."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(case.seed if seed is None else seed)
    B, R, P = case.batch, case.rows_per_req, case.page_size
    Hq, Hkv, D, Di = case.num_q_heads, case.num_kv_heads, case.head_dim, case.index_dim
    MB = case.max_blocks
    T = B * R

    # 1. context lengths
    if case.ctx_lo == case.ctx_hi:
        lens = torch.full((B,), case.ctx_lo, dtype=torch.int64, device=device)
    else:
        lens = _uniform_int(gen, case.ctx_lo, case.ctx_hi, (B,), device)
    lens_cpu = lens.cpu().tolist()
    nblocks = [-(-L // P) for L in lens_cpu]
    assert max(nblocks) <= MB, "context exceeds the page-table width"
    used = sum(nblocks)
    if case.pool == "identity":
        NP = case.pool_pages if case.pool_pages is not None else B * MB
    else:
        NP = case.pool_pages if case.pool_pages is not None else used
    assert NP >= used

    # 2. q
    q = torch.randn((T, Hq, D), generator=gen, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    # 3./4. K, V: bf16 N(0,1), then NVFP4
    kb = torch.randn((NP, Hkv, P, D), generator=gen, device=device,
                     dtype=torch.float32).to(torch.bfloat16)
    k_pool, k_sf, k_scale = nvfp4_encode(kb)
    del kb
    vb = torch.randn((NP, Hkv, P, D), generator=gen, device=device,
                     dtype=torch.float32).to(torch.bfloat16)
    v_pool, v_sf, v_scale = nvfp4_encode(vb)
    del vb
    # 5./6. index query and keys
    if case.iq_row_noise > 0:
        base = _uniform_int(gen, -127, 127, (B, 1, Hq, Di), device)
        noise = _uniform_int(gen, -case.iq_row_noise, case.iq_row_noise, (B, R, Hq, Di), device)
        iq = (base + noise).clamp(-127, 127).reshape(T, Hq, Di).to(torch.int8)
    else:
        iq = _uniform_int(gen, -127, 127, (T, Hq, Di), device).to(torch.int8)
    ik_pool = _uniform_int(gen, -127, 127, (NP, P, Di), device).to(torch.int8)

    # 7. page table
    pt = torch.full((B, MB), -1, dtype=torch.int64, device=device)
    if case.pool == "identity":
        order = torch.arange(NP, device=device)
    else:
        order = torch.randperm(NP, generator=gen, device=device)
    off = 0
    for b in range(B):
        nb = nblocks[b]
        pt[b, :nb] = order[off:off + nb]
        off += nb

    # 8. invalid entries (below each request's block count, window included)
    if case.invalid_frac > 0:
        u = torch.rand((B, MB), generator=gen, device=device)
        col = torch.arange(MB, device=device).unsqueeze(0)
        inside = col < torch.tensor(nblocks, device=device).unsqueeze(1)
        pt = torch.where((u < case.invalid_frac) & inside, torch.full_like(pt, -1), pt)

    # 9. ties: copy whole index-key blocks between full valid blocks of a request
    if case.tie_frac > 0:
        pt_cpu = pt.cpu()
        for b in range(B):
            full = (lens_cpu[b] - R + 1) // P       # blocks fully visible to every row
            valid = [beta for beta in range(full) if int(pt_cpu[b, beta]) >= 0]
            ndst = int(round(case.tie_frac * len(valid)))
            if ndst == 0 or len(valid) < 2:
                continue
            perm = torch.randperm(len(valid), generator=gen, device=device).cpu().tolist()
            dst = [valid[i] for i in perm[:ndst]]
            src_pool = [valid[i] for i in perm[ndst:]]
            if not src_pool:
                continue
            pick = torch.randint(0, len(src_pool), (ndst,), generator=gen,
                                 device=device).cpu().tolist()
            for d_beta, si in zip(dst, pick):
                s_page = int(pt_cpu[b, src_pool[si]])
                d_page = int(pt_cpu[b, d_beta])
                ik_pool[d_page].copy_(ik_pool[s_page])

    return dict(
        case=case, batch=B, rows_per_req=R, num_q_heads=Hq, num_kv_heads=Hkv,
        head_dim=D, index_dim=Di, page_size=P, max_blocks=MB, num_pages=NP,
        k=case.k, window=case.window, sm_scale=1.0 / math.sqrt(D),
        q=q.contiguous(), iq=iq.contiguous(), ik_pool=ik_pool.contiguous(),
        k_pool=k_pool, k_sf=k_sf, v_pool=v_pool, v_sf=v_sf,
        k_scale=k_scale, v_scale=v_scale,
        page_table=pt.to(torch.int32).contiguous(),
        seqlens=lens.to(torch.int32).contiguous(),
    )


def geometry(w: dict) -> dict:
    """The geometry fields of a workload, as plain ints."""
    return {k: int(w[k]) for k in ("batch", "rows_per_req", "num_q_heads",
                                   "num_kv_heads", "head_dim", "index_dim",
                                   "page_size", "max_blocks", "num_pages")}


def make_new_tokens(w: dict, seed: Optional[int] = None) -> dict:
    """The step's new rows for the decode prologue: k_new, v_new ~ N(0, 1) as
    bf16 [T, Hkv, D] and ik_new uniform int8 [T, Di] in [-127, 127], drawn in
    that order from their own seeded generator (inputs only; the quantiser
    lives in the library and in the oracle)."""
    T = w["batch"] * w["rows_per_req"]
    Hkv, D, Di = w["num_kv_heads"], w["head_dim"], w["index_dim"]
    device = w["q"].device
    gen = torch.Generator(device=device)
    gen.manual_seed((w["case"].seed if seed is None else seed) + 1000003)
    k_new = torch.randn((T, Hkv, D), generator=gen, device=device).to(torch.bfloat16)
    v_new = torch.randn((T, Hkv, D), generator=gen, device=device).to(torch.bfloat16)
    ik_new = _uniform_int(gen, -127, 127, (T, Di), device).to(torch.int8)
    return {"k_new": k_new, "v_new": v_new, "ik_new": ik_new}


def to_numpy(w: dict) -> dict:
    """Host copies of a workload's tensors (bf16 as raw uint16 bits)."""
    out = {}
    for key, val in w.items():
        if isinstance(val, torch.Tensor):
            t = val.detach().cpu().contiguous()
            if t.dtype == torch.bfloat16:
                t = t.view(torch.int16)
                out[key] = t.numpy().view("uint16")
            else:
                out[key] = t.numpy()
        else:
            out[key] = val
    return out
