"""QSA block-sparse GQA decode / speculative verify over an NVFP4 paged KV
cache, for one GB300 (sm_103a).

The compute lives in libqsa.so (hand-written CUDA kernels behind the C ABI of
include/qsa.h); this package is its ctypes binding plus a small helper that
owns the per-step output buffers.  Importing the package does not load the
library; the first call does, and raises if it is not built.
"""
from __future__ import annotations

import math

import torch

from .binding import (EXPORTS, QsaError, load, make_geom, qsa_geom_t, qsa_index_scores,
                      qsa_select_sparse_decode, qsa_select_sparse_decode_fused,
                      qsa_select_topk, qsa_sparse_decode, qsa_sparse_decode_ex, qsa_sparse_decode_noalloc,
                      qsa_sparse_decode_noalloc_status, qsa_debug_set_wait_ns,
                      qsa_debug_bounds_status, bounds_checked, library_path,
                      qsa_sparse_decode_workspace_bytes, qsa_sparse_decode_workspace_bytes_ex,
                      qsa_rollback_gather, qsa_rollback_restore, qsa_rollback_state_bytes,
                      qsa_sparse_prefill, qsa_sparse_prefill_workspace_bytes,
                      qsa_status_string, qsa_store_kv_tokens, qsa_workspace_init,
                      qsa_workspace_status)

__all__ = [
    "EXPORTS", "QsaError", "load", "make_geom", "qsa_geom_t", "qsa_index_scores",
    "qsa_select_sparse_decode", "qsa_select_sparse_decode_fused",
    "qsa_select_topk", "qsa_sparse_decode", "qsa_sparse_decode_ex", "qsa_sparse_decode_noalloc",
    "qsa_sparse_decode_noalloc_status", "qsa_debug_set_wait_ns", "qsa_debug_bounds_status",
    "bounds_checked", "library_path",
    "qsa_sparse_decode_workspace_bytes", "qsa_sparse_decode_workspace_bytes_ex",
    "qsa_rollback_gather", "qsa_rollback_restore", "qsa_rollback_state_bytes",
    "qsa_sparse_prefill", "qsa_sparse_prefill_workspace_bytes",
    "qsa_status_string", "qsa_store_kv_tokens", "qsa_workspace_init", "qsa_workspace_status",
    "DecodeStep", "MAX_DECODE_ROWS",
]

# Rows per request the decode / verify attention takes; longer row groups
# (context chunks) go to the row-tile path, qsa_sparse_prefill.
MAX_DECODE_ROWS = 8

GEOM_FIELDS = [n for n, _ in qsa_geom_t._fields_]


class DecodeStep:
    """Device buffers for one QSA step of a fixed geometry, and the library
    calls that fill them: index scores -> top-k selection -> sparse decode,
    chained by programmatic dependent launch.  ``fused`` runs selection and
    decode through qsa_select_sparse_decode instead.  ``num_splits`` = 0 lets
    the library choose the KV split count.  A geometry with more than
    MAX_DECODE_ROWS rows per request (a context row group) runs
    qsa_sparse_prefill as its attention."""

    def __init__(self, geom: dict, k: int, window: int, device="cuda", num_splits: int = 0,
                 fused: bool = False):
        self.fused = bool(fused)
        self.geom = {n: int(geom[n]) for n in GEOM_FIELDS}
        self.cg = make_geom(**self.geom)
        self.k, self.window, self.num_splits = int(k), int(window), int(num_splits)
        T = self.geom["batch"] * self.geom["rows_per_req"]
        Hq, D, MB = self.geom["num_q_heads"], self.geom["head_dim"], self.geom["max_blocks"]
        dev = torch.device(device)
        self.scores = torch.empty((T, MB), dtype=torch.int32, device=dev)
        self.sel = torch.empty((T, self.k), dtype=torch.int32, device=dev)
        self.nsel = torch.empty((T,), dtype=torch.int32, device=dev)
        # out and lse share one allocation (lse right after out, 256-byte
        # aligned) so that a host can read a step's results in one copy.
        out_bytes = T * Hq * D * 2
        lse_off = (out_bytes + 255) // 256 * 256
        self.results = torch.empty((lse_off + T * Hq * 4,), dtype=torch.uint8, device=dev)
        self.out = self.results[:out_bytes].view(torch.bfloat16).view(T, Hq, D)
        self.lse = self.results[lse_off:].view(torch.float32).view(T, Hq)
        self.prefill = self.geom["rows_per_req"] > MAX_DECODE_ROWS
        if self.prefill:
            nbytes = qsa_sparse_prefill_workspace_bytes(self.cg, self.k)
        else:
            nbytes = qsa_sparse_decode_workspace_bytes_ex(self.cg, self.k, self.num_splits)
        if nbytes == 0:
            raise QsaError("qsa_sparse_decode_workspace_bytes", 1, "invalid geometry")
        self.workspace = torch.empty((nbytes,), dtype=torch.uint8, device=dev)
        qsa_workspace_init(self.workspace)

    def buffers(self) -> dict:
        """A fresh set of the step's intermediate and output buffers (scores,
        sel, nsel, out, lse and a zero-filled workspace) on the step's device,
        e.g. one per input replica of a benchmark."""
        dev = self.scores.device
        ws = torch.empty_like(self.workspace)
        qsa_workspace_init(ws)
        b = dict(scores=torch.empty_like(self.scores), sel=torch.empty_like(self.sel),
                 nsel=torch.empty_like(self.nsel), out=torch.empty_like(self.out),
                 lse=torch.empty_like(self.lse), workspace=ws)
        return b

    def own_buffers(self) -> dict:
        return dict(scores=self.scores, sel=self.sel, nsel=self.nsel, out=self.out,
                    lse=self.lse, workspace=self.workspace)

    def status(self) -> int:
        """Device status word of this step's workspace: 0 when every bounded
        wait completed."""
        return qsa_workspace_status(self.workspace)

    def launches(self):
        """The step's library calls in order, as (name, fn) pairs; fn(w, bufs,
        stream, sm_scale=None) issues that call for workload tensors ``w``
        with the buffers ``bufs`` (the keys of buffers())."""
        def sm_of(w, sm_scale):
            return float(w["sm_scale"]) if sm_scale is None else float(sm_scale)

        def index(w, bufs, stream, sm_scale=None):
            qsa_index_scores(self.cg, w["iq"], w["ik_pool"], w["page_table"], w["seqlens"],
                             bufs["scores"], stream)

        def select(w, bufs, stream, sm_scale=None):
            qsa_select_topk(self.cg, bufs["scores"], w["seqlens"], self.k, self.window,
                            bufs["sel"], bufs["nsel"], stream)

        def prefill(w, bufs, stream, sm_scale=None):
            qsa_sparse_prefill(self.cg, w["q"], w["k_pool"], w["k_sf"], w["v_pool"], w["v_sf"],
                               w["k_scale"], w["v_scale"], sm_of(w, sm_scale), w["page_table"],
                               w["seqlens"], bufs["sel"], self.k, bufs["out"], bufs["lse"],
                               bufs["workspace"], stream)

        def decode(w, bufs, stream, sm_scale=None):
            qsa_sparse_decode_ex(self.cg, w["q"], w["k_pool"], w["k_sf"], w["v_pool"],
                                 w["v_sf"], w["k_scale"], w["v_scale"], sm_of(w, sm_scale),
                                 w["page_table"], w["seqlens"], bufs["sel"], self.k, bufs["out"],
                                 bufs["lse"], bufs["workspace"], self.num_splits, stream)

        def select_decode(w, bufs, stream, sm_scale=None):
            qsa_select_sparse_decode(self.cg, bufs["scores"], self.window, w["q"], w["k_pool"],
                                     w["k_sf"], w["v_pool"], w["v_sf"], w["k_scale"],
                                     w["v_scale"], sm_of(w, sm_scale), w["page_table"],
                                     w["seqlens"], self.k, bufs["sel"], bufs["nsel"],
                                     bufs["out"], bufs["lse"], bufs["workspace"],
                                     self.num_splits, stream)

        if self.prefill:
            return [("index_scores", index), ("select_topk", select), ("sparse_prefill", prefill)]
        if self.fused:
            return [("index_scores", index), ("select_sparse_decode", select_decode)]
        return [("index_scores", index), ("select_topk", select), ("sparse_decode", decode)]

    def run(self, w: dict, stream=None, sm_scale=None, out=None, lse=None, bufs=None):
        """One step over workload tensors ``w`` (the generator's layout).
        ``out`` / ``lse`` (optional) receive the results instead of the step's
        own buffers, e.g. one span per step of a pipelined serving loop;
        ``bufs`` (optional, from buffers()) replaces every buffer."""
        b = dict(self.own_buffers() if bufs is None else bufs)
        if out is not None:
            b["out"] = out
        if lse is not None:
            b["lse"] = lse
        for _, fn in self.launches():
            fn(w, b, stream, sm_scale)
        return self

    @staticmethod
    def default_sm_scale(head_dim: int = 128) -> float:
        return 1.0 / math.sqrt(head_dim)
