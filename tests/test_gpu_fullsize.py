"""Parity at the full benchmark sizes, in the benchmark's launch
configuration (dsa_forward without exported intermediates), checked on
outputs the oracle computes one row at a time:

  * the benchmark call equals the same call with scores / indices exported,
    bit for bit (so the exported intermediates are the benchmark's own);
  * indexer scores of sampled rows within 1e-3 (1 + |ref|);
  * top-k bit-exact against the oracle on the GPU's fp32 scores, on every
    row of the decode workloads and the 16384-token prefill, on sampled
    rows of the chunked prefill;
  * attention of sampled rows within 1e-2 + 1e-2 |ref| given the GPU's
    indices, lse within 1e-3 (1 + |ref|).
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


def _host_seq(bt, b, rows_global, pos, ctx):
    """A one-sequence numpy batch holding sequence b's caches and the given
    query rows (positions pos), for the oracle."""
    n = len(rows_global)
    cache = slice(b * bt.stride, b * bt.stride + ctx)
    ri = torch.tensor(rows_global, dtype=torch.long, device=bt.q.device)
    return W.Batch(B=1, stride=ctx, q_off=np.array([0, n], np.int32), ctx_len=np.array([ctx], np.int32),
                   q_idx=_bits(bt.q_idx[ri]), w=bt.w[ri].cpu().numpy(), k_idx=_bits(bt.k_idx[cache]),
                   q=_bits(bt.q[ri]), kv=_bits(bt.kv[cache]), k=bt.k, sm_scale=bt.sm_scale), \
        [int(p) for p in pos]


def _check_rows(bt, b, rows_global, pos, ctx, scores, idx, out, lse):
    """Oracle checks of packed rows of sequence b, each in a one-row batch of
    its own whose context ends at the row's position."""
    for r, t in zip(rows_global, pos):
        hb, _ = _host_seq(bt, b, [r], [t], t + 1)   # ctx = t + 1: the row is the last query
        sc = scores[r, :t + 1].cpu().numpy()
        ref = oracle.indexer_scores(hb, [0], ld=t + 1)[0]
        assert np.all(np.abs(sc - ref) <= SCORE_RTOL * (1 + np.abs(ref))), f"scores row {r} (t={t})"
        got_idx = idx[r].cpu().numpy()
        assert np.array_equal(got_idx, oracle.topk(hb, sc[None, :], rows=[0], k=bt.k)[0]), f"top-k row {r}"
        o_ref, l_ref = oracle.sparse_mla(hb, got_idx[None, :], rows=[0])
        o = out[r].float().cpu().numpy()
        assert np.all(np.abs(o - o_ref[0]) <= ATT_ATOL + ATT_RTOL * np.abs(o_ref[0])), f"attention row {r}"
        lg = lse[r].cpu().numpy()
        assert np.all(np.abs(lg - l_ref[0]) <= LSE_RTOL * (1 + np.abs(l_ref[0]))), f"lse row {r}"


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


def _topk_all_rows(bt_rows_pos_ctx, scores, idx, k):
    """Bit-exact top-k on every listed row (one sequence per group)."""
    for pos, rows in bt_rows_pos_ctx:
        sc = np.nan_to_num(scores[rows].cpu().numpy(), nan=0.0)
        L = sc.shape[1]
        lay = W.Batch(B=1, stride=L, q_off=np.array([0, len(rows)], np.int32),
                      ctx_len=np.array([pos[-1] + 1], np.int32), q_idx=None, w=None, k_idx=None, q=None, kv=None,
                      k=k, sm_scale=W.SM_SCALE)
        assert np.all(np.diff(pos) == 1) and pos[-1] + 1 - len(rows) == pos[0]
        ref = oracle.topk(lay, sc, k=k)
        got = idx[rows].cpu().numpy()
        bad = np.nonzero((got != ref).any(axis=1))[0]
        assert len(bad) == 0, f"top-k differs on {len(bad)} rows, first row {rows[bad[0]]}"


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
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
        # top-k on every row (each row is its sequence's last position)
        for r in range(wl.B):
            _topk_all_rows([([ctx - 1], [r])], sc, ix, wl.k)
        for r in sorted({0, wl.B // 2, wl.B - 1}):
            _check_rows(bt, r, [r], [ctx - 1], ctx, sc, ix, o2, l2)


def test_prefill_full_size():
    wl = W.WORKLOADS["prefill_T16384"]
    T = wl.ctx
    bt = W.make_batch_torch([T], [T], wl.k, wl.seed, key_kind=wl.key_kind)
    b = dsa.Batch(bt.q_off, bt.ctx_len, T, T, bt.stride, total_q=T)
    o1, l1, _, _ = _run(b, bt, bt.q_idx, bt.w, bt.q, T, export=False)
    o2, l2, ix, sc = _run(b, bt, bt.q_idx, bt.w, bt.q, T, export=True)
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
    # top-k on every row, in slabs of 2048 rows
    for r0 in range(0, T, 2048):
        rows = list(range(r0, r0 + 2048))
        _topk_all_rows([(rows, rows)], sc[:, :], ix, wl.k)
    rows = [0, 1, 127, 2046, 2047, 2048, 2049, 5000, 8191, 12000, T - 2, T - 1]
    for r in rows:
        _check_rows(bt, 0, [r], [r], r + 1, sc, ix, o2, l2)


def test_chunked_prefill_full_size():
    wl = W.WORKLOADS["chunked_prefill_T65536_c8192"]
    T, C = wl.ctx, wl.n_new
    bt = W.make_batch_torch([T], [T], wl.k, wl.seed, key_kind=wl.key_kind)
    for c in (0, 3, 7):
        qo = torch.tensor([0, C], dtype=torch.int32, device="cuda")
        cl = torch.tensor([C * (c + 1)], dtype=torch.int32, device="cuda")
        b = dsa.Batch(qo, cl, C, C * (c + 1), bt.stride, total_q=C)
        s = slice(C * c, C * (c + 1))
        ld = C * (c + 1)
        o1, l1, _, _ = _run(b, bt, bt.q_idx[s], bt.w[s], bt.q[s], ld, export=False)
        o2, l2, ix, sc = _run(b, bt, bt.q_idx[s], bt.w[s], bt.q[s], ld, export=True)
        assert torch.equal(o1.view(torch.int16), o2.view(torch.int16)) and torch.equal(l1, l2)
        rows = [0, 1, C // 2, C - 1]
        _topk_all_rows([([C * c + i for i in range(C - 256, C)], list(range(C - 256, C)))], sc, ix, wl.k)
        # oracle rows: the chunk's row i is position C*c + i; the helper takes
        # the packed rows of this chunk and the full cache
        for i in rows:
            t = C * c + i
            hb, _ = _host_seq(bt, 0, [C * c + i], [t], t + 1)
            scv = sc[i, :t + 1].cpu().numpy()
            ref = oracle.indexer_scores(hb, [0], ld=t + 1)[0]
            assert np.all(np.abs(scv - ref) <= SCORE_RTOL * (1 + np.abs(ref))), f"chunk {c} row {i}"
            gi = ix[i].cpu().numpy()
            assert np.array_equal(gi, oracle.topk(hb, scv[None, :], rows=[0], k=wl.k)[0])
            o_ref, l_ref = oracle.sparse_mla(hb, gi[None, :], rows=[0])
            o = o2[i].float().cpu().numpy()
            assert np.all(np.abs(o - o_ref[0]) <= ATT_ATOL + ATT_RTOL * np.abs(o_ref[0])), f"chunk {c} row {i}"
