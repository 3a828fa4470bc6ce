"""Parity at the full benchmark sizes, in the benchmark's launch
configuration (dsa_forward without exported intermediates), against the
fp64 oracle run on many rows at once:

  * the benchmark call equals the same call with scores / indices exported,
    bit for bit (so the exported intermediates are the benchmark's own);
  * indexer scores within 1e-3 (1 + |ref|), attention within
    1e-2 + 1e-2 |ref| given the GPU's indices, lse within 1e-3 (1 + |ref|):
    every row of the decode workloads; a stratified sample of the
    16384-token prefill (t = 0, k-1, k, the last row, random rows) plus
    every row with t < k, where the selection must be all of [0, t] and the
    result is dense causal attention; in the chunked prefill, every row with
    t < k of the first chunk and sampled rows of later chunks;
  * top-k bit-exact against the oracle on the GPU's fp32 scores on every
    row of every workload (all 65,536 rows of the chunked prefill);
  * the chunked prefill equals the same rows computed in one call, bit for
    bit (each row's arithmetic does not depend on how the rows are batched).
"""

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_gb300 as dsa
import workloads as W
from dsa_case import ATT_ATOL, ATT_RTOL, LSE_RTOL, SCORE_RTOL

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_attention_gb300 import build as B
    B.build()
    dsa.load_library()


def _bits(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _host_batch(bt, q_off, ctx_len, rows):
    """The numpy batch the oracle reads: query-side arrays of the packed rows
    `rows` (a slice of bt's query arrays), every sequence's caches."""
    q_off = np.asarray(q_off, np.int32)
    return W.Batch(B=len(ctx_len), stride=bt.stride, q_off=q_off, ctx_len=np.asarray(ctx_len, np.int32),
                   q_idx=_bits(bt.q_idx[rows]), w=bt.w[rows].cpu().numpy(), k_idx=_bits(bt.k_idx),
                   q=_bits(bt.q[rows]), kv=_bits(bt.kv), k=bt.k, sm_scale=bt.sm_scale)


def _check_rows(hb, rows, scores, idx, out, lse):
    """Scores, top-k and attention of the packed rows `rows` of hb (GPU
    results indexed by the same packed rows) against the oracle."""
    rows = list(rows)
    pos = hb.positions()
    ld = scores.shape[1]
    assert min(rows) >= 0 and max(rows) < scores.shape[0]   # checked on the host before device indexing
    ri = torch.tensor(rows, dtype=torch.long, device=scores.device)
    sc = scores[ri].cpu().numpy()
    ref = oracle.indexer_scores(hb, rows, ld=ld)
    for j, r in enumerate(rows):
        t = pos[r][1]
        a, e = sc[j, :t + 1], ref[j, :t + 1]
        bad = np.nonzero(np.abs(a - e) > SCORE_RTOL * (1 + np.abs(e)))[0]
        assert len(bad) == 0, f"scores row {r} (t={t}) position {bad[0]}: {a[bad[0]]} vs {e[bad[0]]}"
    gi = idx[ri].cpu().numpy()
    ref_i = oracle.topk(hb, np.nan_to_num(sc, nan=0.0), rows=rows, k=hb.k)
    bad = np.nonzero((gi != ref_i).any(axis=1))[0]
    assert len(bad) == 0, f"top-k differs on {len(bad)} rows, first row {rows[bad[0]]}"
    o_ref, l_ref = oracle.sparse_mla(hb, gi, rows=rows)
    o = out[ri].float().cpu().numpy()
    err = np.abs(o - o_ref) - (ATT_ATOL + ATT_RTOL * np.abs(o_ref))
    assert err.max() <= 0, f"attention row {rows[int(np.argmax(err.max(axis=(1, 2))))]} off by {err.max()}"
    lg = lse[ri].cpu().numpy()
    assert np.all(np.abs(lg - l_ref) <= LSE_RTOL * (1 + np.abs(l_ref))), "lse"
    return gi


def _run(b, bt, q_idx, w, q, ld, export):
    n = b.total_q
    out = torch.empty((n, 64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((n, 64), dtype=torch.float32, device="cuda")
    ws = dsa.workspace(b, bt.k)
    idx = torch.empty((n, bt.k), dtype=torch.int32, device="cuda") if export else None
    sc = torch.full((n, ld), float("nan"), dtype=torch.float32, device="cuda") if export else None
    dsa.forward(b, q_idx, w, bt.k_idx, q, bt.kv, bt.k, bt.sm_scale, out, lse, idx_out=idx, scores_out=sc, ld=ld,
                ws=ws)
    torch.cuda.synchronize()
    assert dsa.read_device_status(ws) == 0
    return out, lse, idx, sc


def _same(o1, l1, o2, l2):
    return torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)


def _topk_one_sequence(first_pos, scores, idx, k):
    """Bit-exact top-k of consecutive query rows of one sequence starting at
    position first_pos (GPU scores and indices of those rows)."""
    n, L = scores.shape
    lay = W.Batch(B=1, stride=L, q_off=np.array([0, n], np.int32), ctx_len=np.array([first_pos + n], np.int32),
                  q_idx=None, w=None, k_idx=None, q=None, kv=None, k=k, sm_scale=W.SM_SCALE)
    ref = oracle.topk(lay, np.nan_to_num(scores.cpu().numpy(), nan=0.0), k=k)
    got = idx.cpu().numpy()
    bad = np.nonzero((got != ref).any(axis=1))[0]
    assert len(bad) == 0, f"top-k differs on {len(bad)} rows, first at position {first_pos + bad[0]}"


@pytest.mark.parametrize("name", ["decode_B64_ctx32768", "long_decode_B8_ctx202752"])
def test_decode_full_size(name):
    wl = W.WORKLOADS[name]
    bt = W.make_batch_torch([wl.ctx] * wl.B, [1] * wl.B, wl.k, wl.seed, key_kind=wl.key_kind)
    ld = (wl.ctx + 3) // 4 * 4
    for step in sorted({0, wl.steps - 1}):
        ctx = wl.ctx - wl.steps + 1 + step
        cl = torch.full((wl.B,), ctx, dtype=torch.int32, device="cuda")
        b = dsa.Batch(bt.q_off, cl, 1, wl.ctx, bt.stride, total_q=wl.B)
        o1, l1, _, _ = _run(b, bt, bt.q_idx, bt.w, bt.q, ld, export=False)
        o2, l2, ix, sc = _run(b, bt, bt.q_idx, bt.w, bt.q, ld, export=True)
        assert _same(o1, l1, o2, l2)
        hb = _host_batch(bt, np.arange(wl.B + 1), [ctx] * wl.B, slice(0, wl.B))
        _check_rows(hb, range(wl.B), sc, ix, o2, l2)          # every row


def test_prefill_full_size():
    wl = W.WORKLOADS["prefill_T16384"]
    T, k = wl.ctx, wl.k
    bt = W.make_batch_torch([T], [T], k, wl.seed, key_kind=wl.key_kind)
    b = dsa.Batch(bt.q_off, bt.ctx_len, T, T, bt.stride, total_q=T)
    o1, l1, _, _ = _run(b, bt, bt.q_idx, bt.w, bt.q, T, export=False)
    o2, l2, ix, sc = _run(b, bt, bt.q_idx, bt.w, bt.q, T, export=True)
    assert _same(o1, l1, o2, l2)
    for r0 in range(0, T, 2048):                               # top-k on every row
        _topk_one_sequence(r0, sc[r0:r0 + 2048], ix[r0:r0 + 2048], k)
    # rows t < k select all of [0, t]: the result is dense causal attention
    head = ix[:k].cpu().numpy()
    for t in range(k):
        assert np.array_equal(head[t, :t + 1], np.arange(t + 1)) and np.all(head[t, t + 1:] == -1)
    rng = np.random.default_rng(wl.seed)
    fixed = [0, 1, 2, 127, 128, k - 2, k - 1, k, k + 1, 8191, 8192, T - 2, T - 1]
    rows = sorted(set(fixed) | set(rng.choice(np.arange(k, T), 243, replace=False).tolist()) | set(range(k)))
    hb = _host_batch(bt, [0, T], [T], slice(0, T))
    _check_rows(hb, rows, sc, ix, o2, l2)


def test_chunked_prefill_full_size():
    wl = W.WORKLOADS["chunked_prefill_T65536_c8192"]
    T, C = wl.ctx, wl.n_new
    bt = W.make_batch_torch([T], [T], wl.k, wl.seed, key_kind=wl.key_kind)
    # the same 65,536 rows in one call
    b1 = dsa.Batch(bt.q_off, bt.ctx_len, T, T, bt.stride, total_q=T)
    o_all, l_all, _, _ = _run(b1, bt, bt.q_idx, bt.w, bt.q, T, export=False)
    rng = np.random.default_rng(wl.seed)
    for c in range(T // C):
        qo = torch.tensor([0, C], dtype=torch.int32, device="cuda")
        cl = torch.tensor([C * (c + 1)], dtype=torch.int32, device="cuda")
        b = dsa.Batch(qo, cl, C, C * (c + 1), bt.stride, total_q=C)
        s = slice(C * c, C * (c + 1))
        ld = C * (c + 1)
        o2, l2, ix, sc = _run(b, bt, bt.q_idx[s], bt.w[s], bt.q[s], ld, export=True)
        assert _same(o2, l2, o_all[s], l_all[s]), f"chunk {c} differs from the one-call prefill"
        if c in (0, T // C - 1):
            o1, l1, _, _ = _run(b, bt, bt.q_idx[s], bt.w[s], bt.q[s], ld, export=False)
            assert _same(o1, l1, o2, l2)
        _topk_one_sequence(C * c, sc, ix, wl.k)                 # every row of the chunk
        if c in (0, 3, 7):
            rows = sorted({0, 1, C // 2, C - 1} | set(rng.choice(C, 12, replace=False).tolist()))
            if c == 0:
                rows = sorted(set(rows) | set(range(wl.k)))        # every row with t < k
            hb = _host_batch(bt, [0, C], [C * (c + 1)], s)
            _check_rows(hb, rows, sc, ix, o2, l2)
        del o2, l2, ix, sc
