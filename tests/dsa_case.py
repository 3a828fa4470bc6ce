"""Helpers for the GPU parity tests: stage a seeded batch on the device, run
the C-ABI calls, and compare with the oracle under the stated tolerances.

Tolerances (fixed by the method's precision and the bf16 output):
  scores     |gpu - oracle| <= 1e-3 * (1 + |oracle|)      fp32 vs fp64
  top-k      bit-exact against the oracle's top-k of the GPU's fp32 scores
  attention  |gpu - oracle| <= 1e-2 + 1e-2 * |oracle|     given the same indices
  lse        |gpu - oracle| <= 1e-3 * (1 + |oracle|)
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
import sparse_attention_gb300 as dsa
import workloads as W

SCORE_RTOL = 1e-3
ATT_ATOL, ATT_RTOL = 1e-2, 1e-2
LSE_RTOL = 1e-3


def bf16_dev(a: np.ndarray, dev="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)


class Staged:
    """A numpy Batch copied to the device, with output buffers."""

    def __init__(self, bt: W.Batch, dev="cuda", ld=None):
        self.bt = bt
        self.b = dsa.make_batch(bt.q_off, bt.ctx_len, bt.max_q, bt.max_ctx, bt.stride, device=dev)
        self.q_idx, self.k_idx = bf16_dev(bt.q_idx, dev), bf16_dev(bt.k_idx, dev)
        self.q, self.kv = bf16_dev(bt.q, dev), bf16_dev(bt.kv, dev)
        self.w = torch.from_numpy(bt.w).to(dev)
        self.ld = ld or max(4, (bt.max_ctx + 3) // 4 * 4)
        self.ws = dsa.workspace(self.b, bt.k, device=dev)
        self.dev = dev

    def new_scores(self):
        return torch.full((self.bt.total_q, self.ld), float("nan"), dtype=torch.float32, device=self.dev)

    def new_idx(self):
        return torch.full((self.bt.total_q, self.bt.k), -7, dtype=torch.int32, device=self.dev)

    def new_out(self):
        return (torch.full((self.bt.total_q, 64, 512), float("nan"), dtype=torch.bfloat16, device=self.dev),
                torch.full((self.bt.total_q, 64), float("nan"), dtype=torch.float32, device=self.dev))

    def scores(self):
        s = self.new_scores()
        dsa.indexer_scores(self.b, self.q_idx, self.w, self.k_idx, s, ws=self.ws)
        return s

    def topk(self, scores):
        ix = self.new_idx()
        dsa.topk(self.b, scores, self.bt.k, ix, ws=self.ws)
        return ix

    def attention(self, idx):
        out, lse = self.new_out()
        dsa.sparse_mla_fwd(self.b, self.q, self.kv, idx, self.bt.k, self.bt.sm_scale, out, lse, ws=self.ws)
        return out, lse

    def forward(self, with_intermediates=True):
        out, lse = self.new_out()
        idx = self.new_idx() if with_intermediates else None
        sc = self.new_scores() if with_intermediates else None
        dsa.forward(self.b, self.q_idx, self.w, self.k_idx, self.q, self.kv, self.bt.k, self.bt.sm_scale, out, lse,
                    idx_out=idx, scores_out=sc, ld=self.ld, ws=self.ws)
        return out, lse, idx, sc

    def status(self):
        return dsa.read_device_status(self.ws)


def check_scores(st: Staged, scores: torch.Tensor, rows=None):
    rows = list(range(st.bt.total_q)) if rows is None else list(rows)
    ref = oracle.indexer_scores(st.bt, rows, ld=st.ld)
    got = scores[rows].cpu().numpy().astype(np.float64)
    pos = st.bt.positions()
    for j, r in enumerate(rows):
        t = pos[r][1]
        d = np.abs(got[j, :t + 1] - ref[j, :t + 1])
        bad = d > SCORE_RTOL * (1 + np.abs(ref[j, :t + 1]))
        assert not bad.any(), f"row {r} (t={t}): {int(bad.sum())} scores off, max err {d.max():.3g}"
        assert np.all(np.isnan(got[j, t + 1:])), f"row {r}: entries s > t were written"


def check_topk(st: Staged, scores: torch.Tensor, idx: torch.Tensor, rows=None):
    rows = list(range(st.bt.total_q)) if rows is None else list(rows)
    sc = np.nan_to_num(scores[rows].cpu().numpy(), nan=0.0)
    ref = oracle.topk(st.bt, sc, rows=rows, k=st.bt.k)
    got = idx[rows].cpu().numpy()
    if not np.array_equal(got, ref):
        bad = np.nonzero((got != ref).any(axis=1))[0]
        raise AssertionError(f"top-k differs on {len(bad)} rows, first {rows[bad[0]]}: "
                             f"gpu {got[bad[0]][:8]} oracle {ref[bad[0]][:8]}")


def check_attention(st: Staged, idx: torch.Tensor, out: torch.Tensor, lse: torch.Tensor, rows=None):
    rows = list(range(st.bt.total_q)) if rows is None else list(rows)
    o_ref, l_ref = oracle.sparse_mla(st.bt, idx[rows].cpu().numpy(), rows=rows)
    o = out[rows].float().cpu().numpy()
    d = np.abs(o - o_ref)
    bad = d > ATT_ATOL + ATT_RTOL * np.abs(o_ref)
    assert not bad.any(), f"attention: {int(bad.sum())} outputs off, max err {d.max():.3g}"
    lg = lse[rows].cpu().numpy()
    finite = np.isfinite(l_ref)
    assert np.array_equal(np.isfinite(lg), finite)
    dl = np.abs(lg[finite] - l_ref[finite])
    assert np.all(dl <= LSE_RTOL * (1 + np.abs(l_ref[finite]))), f"lse max err {dl.max():.3g}"
