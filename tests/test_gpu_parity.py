"""GPU parity: every C-ABI call against the fp64 oracle on seeded inputs
sized so the oracle finishes in seconds, spanning several tiles and ragged
tails, plus the edge cases of the method."""

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_gb300 as dsa
import workloads as W
from dsa_case import Staged, check_attention, check_scores, check_topk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_attention_gb300 import build as B
    B.build()
    dsa.load_library()


CASES = {
    # the tiny prefill workload: T=512, k=128
    "tiny_prefill": dict(ctx=[512], new=[512], k=128, kind="iid"),
    # ragged multi-sequence prefill: tails that are not multiples of the
    # 8-query group or the 128-key tile, a single-token sequence at t = 0
    "ragged_prefill": dict(ctx=[300, 190, 1, 129, 257], new=[300, 2, 1, 64, 19], k=64, kind="lowrank16"),
    # decode: one query per sequence, some contexts shorter than k
    "decode": dict(ctx=[1000, 2500, 128, 129, 4097, 2048, 2049], new=[1] * 7, k=2048, kind="zipf"),
    # chunked-prefill shape: the second half of the queries of one sequence
    "chunk": dict(ctx=[1200], new=[600], k=256, kind="lowrank16"),
}


@pytest.fixture(scope="module", params=list(CASES))
def staged(request):
    c = CASES[request.param]
    bt = W.make_batch_np(c["ctx"], c["new"], k=c["k"], seed=101 + list(CASES).index(request.param),
                         key_kind=c["kind"], name=request.param)
    st = Staged(bt)
    return st


def test_indexer_scores(staged):
    s = staged.scores()
    check_scores(staged, s)
    assert staged.status() == 0


def test_topk_bit_exact(staged):
    s = staged.scores()
    ix = staged.topk(s)
    check_topk(staged, s, ix)
    assert staged.status() == 0


def test_attention(staged):
    s = staged.scores()
    ix = staged.topk(s)
    out, lse = staged.attention(ix)
    check_attention(staged, ix, out, lse)
    assert staged.status() == 0


def test_forward_equals_steps_and_is_deterministic(staged):
    s = staged.scores()
    ix = staged.topk(s)
    out, lse = staged.attention(ix)
    o1, l1, i1, s1 = staged.forward()
    o2, l2, i2, s2 = staged.forward()
    torch.cuda.synchronize()
    pos = staged.bt.positions()
    for r, (_, t) in enumerate(pos):
        assert torch.equal(s1[r, :t + 1], s[r, :t + 1])
    assert torch.equal(i1, ix) and torch.equal(i2, ix)
    assert torch.equal(o1.view(torch.int16), out.view(torch.int16))
    assert torch.equal(o2.view(torch.int16), out.view(torch.int16))
    assert torch.equal(l1, lse) and torch.equal(l2, lse)
    # without exported intermediates (the benchmark's call) the result is the same
    o3, l3, _, _ = staged.forward(with_intermediates=False)
    assert torch.equal(o3.view(torch.int16), out.view(torch.int16)) and torch.equal(l3, lse)
    assert staged.status() == 0


# ----------------------------------------------------------- top-k edges --

def _topk_rows(scores_np, k, ld=None):
    """Run dsa_topk on explicit score rows: row r sits at position r."""
    T = scores_np.shape[0]
    bt = W.Batch(B=1, stride=T, q_off=np.array([0, T], np.int32), ctx_len=np.array([T], np.int32),
                 q_idx=None, w=None, k_idx=None, q=None, kv=None, k=k, sm_scale=W.SM_SCALE)
    b = dsa.make_batch(bt.q_off, bt.ctx_len, T, T, T)
    ld = ld or scores_np.shape[1]
    sc = torch.from_numpy(np.ascontiguousarray(scores_np, dtype=np.float32)).cuda()
    ix = torch.empty((T, k), dtype=torch.int32, device="cuda")
    ws = dsa.workspace(b, k)
    dsa.topk(b, sc, k, ix, ld=ld, ws=ws)
    assert dsa.read_device_status(ws) == 0
    return ix.cpu().numpy(), oracle.topk(bt, scores_np.astype(np.float32), k=k)


@pytest.mark.parametrize("k", [1, 7, 64])
def test_topk_ties_and_signed_zeros(k):
    rng = np.random.default_rng(5)
    T = 300
    vals = np.array([-3.0, -0.0, 0.0, 0.5, 0.5, 1.0, 2.0, np.inf, -np.inf], dtype=np.float32)
    s = rng.choice(vals, size=(T, T)).astype(np.float32)
    s[10] = 0.0                       # a constant row
    s[11] = -0.0
    s[12, ::2] = -0.0                 # alternating signed zeros
    got, ref = _topk_rows(s, k)
    assert np.array_equal(got, ref)


def test_topk_long_rows_global_path():
    # rows longer than the shared-memory key buffer take the global-memory path
    rng = np.random.default_rng(6)
    T = 45000
    k = 2048
    bt = W.Batch(B=1, stride=T, q_off=np.array([0, 4], np.int32), ctx_len=np.array([T], np.int32),
                 q_idx=None, w=None, k_idx=None, q=None, kv=None, k=k, sm_scale=W.SM_SCALE)
    s = rng.standard_normal((4, T)).astype(np.float32)
    s[1] = np.round(s[1] * 4) / 4      # heavy ties
    s[2, :] = 1.0
    b = dsa.make_batch(bt.q_off, bt.ctx_len, 4, T, T)
    sc = torch.from_numpy(s).cuda()
    ix = torch.empty((4, k), dtype=torch.int32, device="cuda")
    ws = dsa.workspace(b, k)
    dsa.topk(b, sc, k, ix, ws=ws)
    assert dsa.read_device_status(ws) == 0
    assert np.array_equal(ix.cpu().numpy(), oracle.topk(bt, s, k=k))


def test_topk_boundary_positions():
    # positions t = k-2 .. k+1: all-selected rows and the first rows that select
    rng = np.random.default_rng(8)
    k = 128
    s = rng.standard_normal((k + 2, k + 4)).astype(np.float32)
    got, ref = _topk_rows(s[:, :k + 4][:k + 2], k, ld=k + 4)
    assert np.array_equal(got, ref)
    assert np.all(got[k - 2][:k - 1] == np.arange(k - 1)) and got[k - 2][-1] == -1
    assert np.all(got[k - 1] == np.arange(k))


# ------------------------------------------------------- attention edges --

def test_attention_holes_and_single_index():
    bt = W.make_batch_np([700], [3], k=96, seed=77)
    st = Staged(bt)
    rng = np.random.default_rng(2)
    idx = np.full((3, 96), -1, dtype=np.int32)
    idx[0, :1] = [5]                                    # a single selected row
    idx[1, ::3] = np.sort(rng.choice(699, size=32, replace=False))   # -1 holes in between
    idx[2, :] = np.sort(rng.choice(700, size=96, replace=False))
    ix = torch.from_numpy(idx).cuda()
    out, lse = st.attention(ix)
    check_attention(st, ix, out, lse)
    assert st.status() == 0
    v = W.f32_from_bf16_bits(bt.kv).reshape(-1, 576)[5, :512]
    assert np.allclose(out[0].float().cpu().numpy(), np.tile(v, (64, 1)), atol=1e-2, rtol=1e-2)


def test_attention_items_of_mixed_block_counts():
    # 400 query rows over 152 persistent CTAs: each CTA walks two or three
    # rows whose block counts differ (no valid index, one index, an empty
    # first block, full and holed selections), so the per-item handshakes
    # and the read-out of one row overlapping the next row's gathers are
    # exercised with every shape
    k = 256
    bt = W.make_batch_np([600], [400], k=k, seed=80)
    st = Staged(bt)
    rng = np.random.default_rng(3)
    idx = np.full((400, k), -1, dtype=np.int32)
    for i in range(400):
        t = 600 - 400 + i                                  # the row's position
        kind = i % 5
        if kind == 1:
            idx[i, 0] = int(rng.integers(0, t + 1))
        elif kind == 2:                                     # only the second block
            idx[i, 128:128 + 40] = np.sort(rng.choice(t + 1, size=40, replace=False))
        elif kind == 3:                                     # every position it may see, up to k
            n = min(k, t + 1)
            idx[i, :n] = np.sort(rng.choice(t + 1, size=n, replace=False))
        elif kind == 4:
            idx[i, ::2] = np.sort(rng.choice(t + 1, size=k // 2, replace=False))
    ix = torch.from_numpy(idx).cuda()
    out, lse = st.attention(ix)
    torch.cuda.synchronize()
    assert st.status() == 0
    empty = torch.from_numpy(np.arange(400) % 5 == 0).cuda()
    assert torch.all(out[empty].float() == 0) and torch.all(torch.isneginf(lse[empty]))
    check_attention(st, ix, out, lse)


def test_attention_empty_selection_and_bad_index():
    bt = W.make_batch_np([50], [2], k=8, seed=78)
    st = Staged(bt)
    idx = np.full((2, 8), -1, dtype=np.int32)
    idx[1, :3] = [1, 60, 2]                  # 60 > t = 49: out of [-1, t]
    out, lse = st.attention(torch.from_numpy(idx).cuda())
    torch.cuda.synchronize()
    assert torch.all(out[0].float() == 0) and torch.all(torch.isneginf(lse[0]))
    assert st.status() == 7                  # DSA_ERR_BAD_INDEX latched
    # the bad entry was skipped: row 1 attends over positions 1 and 2 only
    o_ref, _ = oracle.sparse_mla(bt, np.array([[1, 2, -1, -1, -1, -1, -1, -1]], np.int32), rows=[1])
    assert np.allclose(out[1].float().cpu().numpy(), o_ref[0], atol=1e-2, rtol=1e-2)
    dsa.reset_device_status(st.ws)
    assert st.status() == 0


def test_bad_batch_is_latched_not_faulted():
    bt = W.make_batch_np([40], [4], k=8, seed=79)
    st = Staged(bt)
    # ctx_len beyond the host bound max_ctx: the kernels must skip and latch
    st.b.ctx_len.fill_(10_000)
    s = st.new_scores()
    dsa.indexer_scores(st.b, st.q_idx, st.w, st.k_idx, s, ws=st.ws)
    assert st.status() == 6
    assert torch.all(torch.isnan(s))


def test_empty_batch_is_noop():
    b = dsa.make_batch([0, 0], [5], 0, 5, 8, total_q=0)
    ws = dsa.workspace(b, 4)
    z = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    f = torch.empty(16, dtype=torch.float32, device="cuda")
    dsa.forward(b, z, f, z, z, z, 4, 0.0625, z, ws=ws)
    assert dsa.read_device_status(ws) == 0


@pytest.mark.parametrize("T,rows", [(33000, 3), (100000, 3), (340000, 2)])
def test_topk_cluster_slices_and_global_fallback(T, rows):
    # Rows 0 and 1 are tied so heavily that the sampled bound keeps too many
    # candidates (the whole-row select runs); row 2 is random (the candidate
    # select runs).  T = 100000 and 340000 split each row over a cluster of
    # 4 and 8 CTAs, so tied runs straddle the slices of different CTAs.
    rng = np.random.default_rng(T)
    k = 2048
    bt = W.Batch(B=1, stride=T, q_off=np.array([0, rows], np.int32), ctx_len=np.array([T], np.int32),
                 q_idx=None, w=None, k_idx=None, q=None, kv=None, k=k, sm_scale=W.SM_SCALE)
    s = rng.standard_normal((rows, T)).astype(np.float32)
    s[0, :] = 0.5                                   # all tied: the first k positions win
    s[1, ::3] = 7.0                                 # ties far above the rest, across every slice
    b = dsa.make_batch(bt.q_off, bt.ctx_len, rows, T, T)
    sc = torch.from_numpy(s).cuda()
    ix = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    ws = dsa.workspace(b, k)
    dsa.topk(b, sc, k, ix, ws=ws)
    assert dsa.read_device_status(ws) == 0
    got = ix.cpu().numpy()
    assert np.array_equal(got, oracle.topk(bt, s, k=k))
    assert np.array_equal(got[0], np.arange(k))


def test_indexshare_window_reuses_the_full_layers_indices():
    # IndexShare: layer 0 runs the whole path; layers 1 and 2 ("shared") run
    # attention only, on their own q and latent cache, with layer 0's indices
    full = W.make_batch_np([3000, 2500, 700], [1, 1, 1], k=512, seed=81, key_kind="zipf")
    st = Staged(full)
    out0, lse0, idx, _ = st.forward()
    check_attention(st, idx, out0, lse0)
    for layer in (1, 2):
        lb = W.make_batch_np([3000, 2500, 700], [1, 1, 1], k=512, seed=81 + 10 * layer)
        sl = Staged(lb)
        out, lse = sl.attention(idx)
        check_attention(sl, idx, out, lse)          # the shared layer against the oracle on the reused indices
        assert sl.status() == 0


def test_chunked_equals_one_call():
    # chunked prefill: the queries of one sequence in chunks of 1000 rows
    # (not a multiple of the 8-query group, so the groups fall differently
    # than in one call), each chunk against the cache written so far
    T, C, k = 2600, 1000, 256
    full = W.make_batch_np([T], [T], k=k, seed=83, key_kind="lowrank16")
    st = Staged(full)
    out_all, lse_all, idx_all, _ = st.forward()
    check_attention(st, idx_all, out_all, lse_all, rows=[0, 999, 1000, 1001, 2599])
    for c0 in range(0, T, C):
        n = min(C, T - c0)
        b = dsa.make_batch([0, n], [c0 + n], n, c0 + n, T)
        ws = dsa.workspace(b, k)
        out = torch.empty((n, 64, 512), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((n, 64), dtype=torch.float32, device="cuda")
        idx = torch.empty((n, k), dtype=torch.int32, device="cuda")
        s = slice(c0, c0 + n)
        dsa.forward(b, st.q_idx[s], st.w[s], st.k_idx, st.q[s], st.kv, k, full.sm_scale, out, lse, idx_out=idx,
                    ws=ws)
        assert dsa.read_device_status(ws) == 0
        assert torch.equal(idx, idx_all[s])
        assert torch.equal(out.view(torch.int16), out_all[s].view(torch.int16)) and torch.equal(lse, lse_all[s])


def test_maximum_batch_of_sequences():
    # 65,535 sequences (the most one launch's grid takes), contexts 1..4;
    # queries in every 997th sequence and the last two, none elsewhere, so
    # every kernel's sequence index runs to its maximum over empty sequences;
    # k = 2: rows with t + 1 <= k keep all positions, the others select
    B = 65535
    rng = np.random.default_rng(84)
    ctx = rng.integers(1, 5, B).tolist()
    new = [1 if (b % 997 == 0 or b >= B - 2) else 0 for b in range(B)]
    bt = W.make_batch_np(ctx, new, k=2, seed=85)
    st = Staged(bt)
    out, lse, idx, sc = st.forward()
    torch.cuda.synchronize()
    assert st.status() == 0
    check_scores(st, sc)
    check_topk(st, sc, idx)
    check_attention(st, idx, out, lse)


@pytest.mark.parametrize("B,k", [(64, 256), (38, 512), (19, 1024), (40, 2048), (100, 2048)])
def test_split_partials_merge(B, k):
    # decode rows whose selected lists are split over 2, 4 and 8 CTAs
    # (merged inside a cluster) and over 3 CTAs (fp32 partials merged by a
    # second kernel; at 100 rows a persistent CTA walks two of the 300
    # items); short contexts leave the later splits of a row without any
    # valid index
    rng = np.random.default_rng(B)
    ctx = [int(c) for c in rng.integers(2, 3 * k, B)]
    ctx[0], ctx[1] = 1, k // 3
    bt = W.make_batch_np(ctx, [1] * B, k=k, seed=90 + B, key_kind="zipf")
    st = Staged(bt)
    out, lse, idx, sc = st.forward()
    torch.cuda.synchronize()
    assert st.status() == 0
    check_topk(st, sc, idx)
    check_attention(st, idx, out, lse)
