"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these checks re-types the oracle's own formula: each one compares it
with a brute force written differently (pure Python), a hand-computed value,
a library routine (torch SDPA in fp64), a closed form printed on the pages,
or an invariant of the definition.  They run on the CPU.
"""

import json
import math
import os
import random

import numpy as np
import pytest

import oracle
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _blank_batch(ctx_len, n_new, k=8, stride=None, sm_scale=W.SM_SCALE):
    return W.make_batch_np(ctx_len, n_new, k=k, seed=1, stride=stride, sm_scale=sm_scale)


# ---------------------------------------------------------------- indexer --

def _bruteforce_scores(batch, rows):
    """Pure-Python loops over (t, s, h, d), no numpy arithmetic."""
    qf = W.f32_from_bf16_bits(batch.q_idx).reshape(batch.total_q, 32, 128).tolist()
    kf = W.f32_from_bf16_bits(batch.k_idx).reshape(-1, 128).tolist()
    wf = batch.w.tolist()
    pos = batch.positions()
    out = {}
    for r in rows:
        b, t = pos[r]
        row = []
        for s in range(t + 1):
            key = kf[b * batch.stride + s]
            tot = 0.0
            for h in range(32):
                qh = qf[r][h]
                dot = math.fsum(qh[d] * key[d] for d in range(128))
                tot += wf[r][h] * max(dot, 0.0)
            row.append(tot)
        out[r] = row
    return out


def test_scores_match_python_bruteforce():
    batch = W.make_batch_np([7, 11], [3, 4], k=4, seed=11)
    rows = list(range(batch.total_q))
    got = oracle.indexer_scores(batch, rows)
    ref = _bruteforce_scores(batch, rows)
    for j, r in enumerate(rows):
        n = len(ref[r])
        np.testing.assert_allclose(got[j, :n], ref[r], rtol=1e-12, atol=1e-14)
        assert np.all(np.isnan(got[j, n:])), "entries s > t must not be written"


def test_scores_hand_example_orientation():
    # q_idx[h, d] = a_h if d == h else 0, so q_idx[h] . k[s] = a_h * k[s, h] and
    # I[t, s] = sum_h w_h * max(0, a_h * k[s, h]).  A transposed operand or a
    # head/dim mix-up changes the result.
    batch = _blank_batch([5], [1])
    a = np.array([1.0 + (h % 3) for h in range(32)], dtype=np.float32)
    q = np.zeros((1, 32, 128), dtype=np.float32)
    for h in range(32):
        q[0, h, h] = a[h]
    kk = np.zeros((5, 128), dtype=np.float32)
    rng = np.random.default_rng(3)
    kk[:, :40] = rng.choice([-2.0, -0.5, 0.25, 1.0, 3.0], size=(5, 40))
    w = rng.choice([-1.0, 0.5, 2.0], size=(1, 32)).astype(np.float32)
    batch.q_idx = W.bf16_bits_from_f32(q)
    batch.k_idx = W.bf16_bits_from_f32(kk)
    batch.w = w
    got = oracle.indexer_scores(batch)[0]
    for s in range(5):
        expect = sum(float(w[0, h]) * max(0.0, float(a[h]) * float(kk[s, h])) for h in range(32))
        assert got[s] == pytest.approx(expect, abs=1e-12)


def test_scores_all_negative_dots_give_zero():
    batch = _blank_batch([6], [2])
    v = np.random.default_rng(5).standard_normal(128).astype(np.float32)
    q = np.tile(v, (2, 32, 1))
    kk = np.stack([-(0.5 + s) * v for s in range(6)]).astype(np.float32)
    batch.q_idx = W.bf16_bits_from_f32(q)
    batch.k_idx = W.bf16_bits_from_f32(kk)
    got = oracle.indexer_scores(batch)
    assert np.all(got[0, :5] == 0.0) and np.all(got[1, :6] == 0.0)


def test_scores_identical_heads_unit_weights():
    # w = 1 and 32 identical heads: I = 32 * ReLU(q . k)
    batch = _blank_batch([9], [9])
    rng = np.random.default_rng(7)
    v = rng.standard_normal((9, 128)).astype(np.float32)
    batch.q_idx = W.bf16_bits_from_f32(np.repeat(v[:, None, :], 32, axis=1))
    batch.w = np.ones((9, 32), dtype=np.float32)
    got = oracle.indexer_scores(batch)
    qv = W.f32_from_bf16_bits(batch.q_idx)[:, 0, :].astype(np.float64)
    kv = W.f32_from_bf16_bits(batch.k_idx).astype(np.float64)
    for t in range(9):
        for s in range(t + 1):
            assert got[t, s] == pytest.approx(32.0 * max(0.0, float(qv[t] @ kv[s])), rel=1e-12, abs=1e-14)


def test_scores_homogeneity_and_sign():
    batch = W.make_batch_np([10], [4], k=4, seed=21)
    base = oracle.indexer_scores(batch)
    b2 = W.make_batch_np([10], [4], k=4, seed=21)
    b2.w = (2.0 * b2.w).astype(np.float32)                       # exact in fp32
    np.testing.assert_allclose(oracle.indexer_scores(b2), 2.0 * base, rtol=1e-14, equal_nan=True)
    b3 = W.make_batch_np([10], [4], k=4, seed=21)
    b3.q_idx = W.bf16_bits_from_f32(2.0 * W.f32_from_bf16_bits(b3.q_idx))  # exact in bf16
    np.testing.assert_allclose(oracle.indexer_scores(b3), 2.0 * base, rtol=1e-14, equal_nan=True)
    b4 = W.make_batch_np([10], [4], k=4, seed=21)
    b4.w = (-b4.w).astype(np.float32)
    np.testing.assert_allclose(oracle.indexer_scores(b4), -base, rtol=1e-14, equal_nan=True)


def test_scores_multi_sequence_uses_own_cache():
    # two sequences whose caches differ; each query must read its own keys
    batch = W.make_batch_np([4, 4], [1, 1], k=4, seed=31, stride=6)
    got = oracle.indexer_scores(batch)
    ref = _bruteforce_scores(batch, [0, 1])
    np.testing.assert_allclose(got[0, :4], ref[0], rtol=1e-12)
    np.testing.assert_allclose(got[1, :4], ref[1], rtol=1e-12)


# ------------------------------------------------------------------- top-k --

def _layout_only(L):
    """A one-sequence batch of L queries at positions 0..L-1 with no tensors
    (the top-k oracle reads only the row layout)."""
    return W.Batch(B=1, stride=L, q_off=np.array([0, L], dtype=np.int32),
                   ctx_len=np.array([L], dtype=np.int32), q_idx=None, w=None, k_idx=None,
                   q=None, kv=None, k=W.TOPK, sm_scale=W.SM_SCALE)


def _bruteforce_topk(row, t, k):
    cand = sorted(range(t + 1), key=lambda s: (-float(row[s]), s))
    m = min(k, t + 1)
    chosen = sorted(cand[:m])
    return chosen + [-1] * (k - m)


def test_topk_hand_example_ties_and_signed_zero():
    batch = _blank_batch([6], [1], k=3)
    scores = np.array([[1.0, 3.0, 3.0, 2.0, -0.0, 0.0]], dtype=np.float32)
    assert oracle.topk(batch, scores, k=3).tolist() == [[1, 2, 3]]
    # five picks: the tied -0.0 (s=4) and +0.0 (s=5) compare equal, lower wins
    assert oracle.topk(batch, scores, k=5).tolist() == [[0, 1, 2, 3, 4]]
    # more picks than positions: all of them, then -1 padding
    assert oracle.topk(batch, scores, k=8).tolist() == [[0, 1, 2, 3, 4, 5, -1, -1]]


def test_topk_matches_python_sort_with_ties():
    rng = np.random.default_rng(17)
    T = 40
    batch = _layout_only(T)
    scores = rng.choice([-1.5, -0.0, 0.0, 0.5, 0.5, 2.0, 7.25], size=(T, T)).astype(np.float32)
    scores += np.float32(0.0) * rng.standard_normal((T, T)).astype(np.float32)
    got = oracle.topk(batch, scores, k=9)
    for t in range(T):
        assert got[t].tolist() == _bruteforce_topk(scores[t], t, 9)


def test_topk_invariants_random_rows():
    rng = np.random.default_rng(19)
    k = 2048
    ts = [0, 1, 2046, 2047, 2048, 2049, 3000, 5000]
    L = max(ts) + 1
    batch = _layout_only(L)
    scores = rng.standard_normal((len(ts), L)).astype(np.float32)
    scores[:, ::7] = np.round(scores[:, ::7], 1)                   # plenty of ties
    got = oracle.topk(batch, scores, rows=ts, k=k)
    for j, t in enumerate(ts):
        m = min(k, t + 1)
        sel = got[j, :m]
        assert np.all(got[j, m:] == -1)
        assert np.all(np.diff(sel) > 0) and sel[0] >= 0 and sel[-1] <= t
        if m < t + 1:
            row = scores[j, :t + 1]
            mask = np.zeros(t + 1, dtype=bool)
            mask[sel] = True
            lo, hi = row[mask].min(), row[~mask].max()
            assert lo >= hi
            if lo == hi:    # at the boundary value, every tied loser is after every tied winner
                assert sel[row[sel] == lo].max() < np.nonzero((~mask) & (row == hi))[0].min()


def test_topk_valid_count_and_pages_pair_counts():
    g = json.load(open(os.path.join(GOLDEN, "pair_counts.json")))
    L, k = g["L"], g["k"]
    # the pages' closed forms (t counted from 1 on the page, from 0 here)
    assert L * (L + 1) // 2 == g["dense_causal_pairs"]
    assert sum(min(k, t + 1) for t in range(L)) == g["topk_causal_pairs"]
    assert round(100.0 * k / L, 4) == g["last_query_selected_percent"]
    # the oracle selects exactly min(k, t+1) positions, across the whole range
    rng = np.random.default_rng(23)
    ts = [0, 5, 2046, 2047, 2048, 100000, L - 1]
    batch = _layout_only(L)
    scores = rng.standard_normal((len(ts), L)).astype(np.float32)
    got = oracle.topk(batch, scores, rows=ts, k=k)
    for j, t in enumerate(ts):
        assert int((got[j] >= 0).sum()) == min(k, t + 1)


# --------------------------------------------------------------- attention --

def test_attention_dense_equivalence_sdpa():
    # t + 1 <= k: the selection is every causal position, so sparse MLA is
    # dense causal attention; checked against torch SDPA in fp64.
    torch = pytest.importorskip("torch")
    T, k = 24, 32
    batch = W.make_batch_np([T], [T], k=k, seed=41)
    idx = np.full((T, k), -1, dtype=np.int32)
    for t in range(T):
        idx[t, :t + 1] = np.arange(t + 1)
    out, lse = oracle.sparse_mla(batch, idx)
    q = torch.from_numpy(W.f32_from_bf16_bits(batch.q).astype(np.float64)).reshape(T, 64, 576)
    kv = torch.from_numpy(W.f32_from_bf16_bits(batch.kv).astype(np.float64)).reshape(-1, 576)[:T]
    qh = q.permute(1, 0, 2)                       # [64, T, 576]
    K = kv.unsqueeze(0).expand(64, T, 576)
    V = kv[:, :512].unsqueeze(0).expand(64, T, 512)
    ref = torch.nn.functional.scaled_dot_product_attention(qh, K, V, is_causal=True, scale=W.SM_SCALE)
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)
    logits = torch.einsum("htd,sd->hts", qh, kv) * W.SM_SCALE
    logits = logits.masked_fill(torch.triu(torch.ones(T, T, dtype=torch.bool), 1), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(logits, -1).T.numpy(), rtol=1e-12)


def test_attention_hand_two_rows():
    # logits 0 and ln 3 -> probabilities 1/4, 3/4; lse = ln 4
    batch = _blank_batch([2], [1], k=2, sm_scale=math.log(3.0))
    q = np.zeros((1, 64, 576), dtype=np.float32)
    q[0, :, 575] = 1.0
    kv = np.zeros((2, 576), dtype=np.float32)
    kv[1, 575] = 1.0
    kv[0, :512] = np.linspace(-1, 1, 512)
    kv[1, :512] = np.linspace(2, -2, 512)
    batch.q, batch.kv = W.bf16_bits_from_f32(q), W.bf16_bits_from_f32(kv)
    out, lse = oracle.sparse_mla(batch, np.array([[0, 1]], dtype=np.int32))
    v = W.f32_from_bf16_bits(batch.kv).astype(np.float64)
    np.testing.assert_allclose(out[0], np.tile(0.25 * v[0, :512] + 0.75 * v[1, :512], (64, 1)), rtol=1e-13)
    np.testing.assert_allclose(lse[0], math.log(4.0), rtol=1e-14)


def test_attention_single_index_and_identical_rows():
    batch = W.make_batch_np([10], [1], k=4, seed=43)
    v = W.f32_from_bf16_bits(batch.kv).astype(np.float64).reshape(-1, 576)
    out, lse = oracle.sparse_mla(batch, np.array([[6, -1, -1, -1]], dtype=np.int32))
    assert np.array_equal(out[0], np.tile(v[6, :512], (64, 1)))
    qv = W.f32_from_bf16_bits(batch.q).astype(np.float64).reshape(64, 576)
    np.testing.assert_allclose(lse[0], W.SM_SCALE * (qv @ v[6]), rtol=1e-13)
    kvb = batch.kv.reshape(-1, 576).copy()
    kvb[:] = kvb[3]
    batch.kv = kvb
    out2, _ = oracle.sparse_mla(batch, np.array([[0, 2, 5, 9]], dtype=np.int32))
    np.testing.assert_allclose(out2[0], np.tile(v[3, :512], (64, 1)), rtol=1e-13)


def test_attention_logit_shift_invariance():
    # every cached row has 1.0 in the last RoPE column; moving q along that
    # column adds the same constant to every logit of the head.
    batch = W.make_batch_np([30], [1], k=16, seed=47)
    kv = W.f32_from_bf16_bits(batch.kv).reshape(-1, 576).copy()
    kv[:, 575] = 1.0
    batch.kv = W.bf16_bits_from_f32(kv)
    idx = np.array([sorted(random.Random(5).sample(range(30), 16))], dtype=np.int32)
    out1, lse1 = oracle.sparse_mla(batch, idx)
    q = W.f32_from_bf16_bits(batch.q).reshape(1, 64, 576).copy()
    q[0, :, 575] += 32.0
    batch.q = W.bf16_bits_from_f32(q)
    out2, lse2 = oracle.sparse_mla(batch, idx)
    np.testing.assert_allclose(out2, out1, rtol=1e-11, atol=1e-13)
    assert not np.allclose(lse2, lse1)


def test_attention_mask_form_equals_gather_form():
    batch = W.make_batch_np([50, 40], [3, 2], k=12, seed=53)
    rng = np.random.default_rng(9)
    pos = batch.positions()
    idx = np.full((batch.total_q, 12), -1, dtype=np.int32)
    for r, (b, t) in enumerate(pos):
        m = min(12, t + 1)
        idx[r, :m] = np.sort(rng.choice(t + 1, size=m, replace=False))
    o1, l1 = oracle.sparse_mla(batch, idx)
    o2, l2 = oracle.masked_mla(batch, idx)
    np.testing.assert_allclose(o1, o2, rtol=1e-11, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=1e-12)


def test_attention_full_path_on_tiny_prefill_is_dense_below_k():
    # oracle scores -> oracle top-k -> oracle attention: rows with t < k select
    # everything and so equal dense causal attention (mask form, all ones).
    batch = W.make_batch_np([40], [40], k=16, seed=59)
    sc = oracle.indexer_scores(batch).astype(np.float32)
    idx = oracle.topk(batch, np.nan_to_num(sc, nan=0.0), k=16)
    o, _ = oracle.sparse_mla(batch, idx)
    dense_idx = np.full((40, 40), -1, dtype=np.int32)
    for t in range(40):
        dense_idx[t, :t + 1] = np.arange(t + 1)
    od, _ = oracle.masked_mla(batch, dense_idx)
    np.testing.assert_allclose(o[:16], od[:16], rtol=1e-11, atol=1e-13)
    assert not np.allclose(o[30:], od[30:])


def test_oracle_wrapper_refuses_batches_larger_than_their_arrays():
    # a batch description naming more sequences than the arrays hold must be
    # refused before the C code runs (it would read past the arrays)
    small = W.make_batch_np([16], [1], k=4, seed=61)
    big = W.Batch(B=3, stride=16, q_off=np.arange(4, dtype=np.int32), ctx_len=np.full(3, 16, np.int32),
                  q_idx=small.q_idx, w=small.w, k_idx=small.k_idx, q=small.q, kv=small.kv, k=4,
                  sm_scale=W.SM_SCALE)
    with pytest.raises(ValueError):
        oracle.indexer_scores(big)
    with pytest.raises(ValueError):
        oracle.sparse_mla(big, np.zeros((3, 4), np.int32))
    with pytest.raises(ValueError):
        oracle.topk(small, np.zeros((1, 8), np.float32), k=4)     # row shorter than t + 1 = 16
