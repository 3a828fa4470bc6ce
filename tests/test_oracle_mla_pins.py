"""CPU pins of the oracle's MLA routines around the path (the pages' expanded
kv_b_proj / o_proj path and the absorbed form), against closed forms, an
independent numpy evaluation, and each other (the absorption identity)."""

import numpy as np
import pytest

import oracle
import workloads as W


@pytest.fixture(scope="module")
def weights():
    return W.make_mla_weights_np(7)


def _wf(bits):
    return W.f32_from_bf16_bits(bits).astype(np.float64)


def test_absorb_q_one_hot_picks_a_row_of_w_uk(weights):
    T = 2
    q_nope = np.zeros((T, 64, 192), np.uint16)
    q_nope[1, 3, 5] = W.bf16_bits_from_f32(np.array([1.0], np.float32))[0]
    _, q_pe = W.make_mla_queries_np(T, 1)
    out = oracle.mla_absorb_q(q_nope, q_pe, weights.w_kvb)
    wk = _wf(weights.w_kvb)
    assert np.array_equal(out[1, 3, :512], wk[3 * 448 + 5])       # W_UK[3]^T e_5 = row 5 of W_UK[3]
    assert np.all(out[0, :, :512] == 0) and np.all(out[1, :3, :512] == 0) and np.all(out[1, 4:, :512] == 0)
    assert np.array_equal(out[:, :, 512:], _wf(q_pe))                # q_pe passes through


def test_absorb_q_matches_numpy(weights):
    qn, qp = W.make_mla_queries_np(3, 2)
    out = oracle.mla_absorb_q(qn, qp, weights.w_kvb)
    wk = _wf(weights.w_kvb).reshape(64, 448, 512)[:, :192, :]      # W_UK[h]: [192, 512]
    ref = np.einsum("thi,hid->thd", _wf(qn), wk)
    assert np.allclose(out[:, :, :512], ref, rtol=1e-12, atol=1e-12)


def test_output_one_hot_and_numpy(weights):
    T = 2
    o_lat = np.zeros((T, 64, 512))
    o_lat[0, 7, 11] = 1.0
    o_lat[1] = np.random.default_rng(3).standard_normal((64, 512))
    o_mid, y = oracle.mla_output(o_lat, weights.w_kvb, weights.w_o)
    wk = _wf(weights.w_kvb).reshape(64, 448, 512)
    wo = _wf(weights.w_o)
    assert np.array_equal(o_mid[0, 7], wk[7, 192:, 11])             # W_UV[7] e_11 = column 11 of W_UV[7]
    assert np.all(o_mid[0, :7] == 0) and np.all(o_mid[0, 8:] == 0)
    ref_mid = np.einsum("hed,hd->he", wk[:, 192:, :], o_lat[1])
    assert np.allclose(o_mid[1], ref_mid, rtol=1e-12, atol=1e-12)
    assert np.allclose(y, o_mid.reshape(T, -1) @ wo.T, rtol=1e-10, atol=1e-12)


def _one_hot_uv(h0, e0, d0):
    """kv_b_proj whose only non-zero entry is W_UV[h0][e0, d0] = 1 (head h0
    holds rows 448 h0 .. 448 h0 + 447; its last 256 rows are W_UV[h0])."""
    w = np.zeros((64 * 448, 512), np.uint16)
    w[448 * h0 + 192 + e0, d0] = W.bf16_bits_from_f32(np.array([1.0], np.float32))[0]
    return w


def test_o_proj_reads_head_major_columns(weights):
    """o_proj's input is the attention output reshaped head-major to
    [T, 64 x 256] ("GLM-5.1 架构深度拆解" §4.5 Step 8), so head h's value
    dimension e is column 256 h + e of W_o.  With o_mid one-hot at (h0, e0)
    the output is that column exactly; a dimension-major layout would read
    column 64 e0 + h0 instead."""
    h0, e0, d0 = 5, 17, 300
    w_kvb = _one_hot_uv(h0, e0, d0)
    o_lat = np.zeros((2, 64, 512))
    o_lat[0, h0, d0] = 1.0
    o_lat[1, h0, d0] = -3.0
    o_mid, y = oracle.mla_output(o_lat, w_kvb, weights.w_o)
    expect_mid = np.zeros((64, 256))
    expect_mid[h0, e0] = 1.0
    assert np.array_equal(o_mid[0], expect_mid)
    wo = _wf(weights.w_o)
    assert np.array_equal(y[0], wo[:, 256 * h0 + e0])
    assert np.array_equal(y[1], -3.0 * wo[:, 256 * h0 + e0])
    assert not np.array_equal(wo[:, 256 * h0 + e0], wo[:, 64 * e0 + h0])


def test_expanded_o_proj_reads_head_major_columns(weights):
    """The same closed form through the pages' expanded path: every query
    attends to one cached row s0 only, so o_mid[h0, e0] = c[s0][d0] and
    y = c[s0][d0] * W_o[:, 256 h0 + e0]."""
    h0, e0, d0 = 9, 200, 4
    w_kvb = _one_hot_uv(h0, e0, d0)
    bt, _ = _tiny_batch()
    idx = np.full((bt.total_q, 8), -1, np.int32)
    idx[:, 0] = 1
    qn, qp = W.make_mla_queries_np(bt.total_q, 95)
    o_mid, y = oracle.mla_expanded(bt, qn, qp, w_kvb, weights.w_o, idx)
    kv = _wf(bt.kv).reshape(-1, 576)
    wo = _wf(weights.w_o)
    for r, (b, t) in enumerate(bt.positions()):
        c = kv[b * bt.stride + 1, d0]
        assert c != 0.0
        expect_mid = np.zeros((64, 256))
        expect_mid[h0, e0] = c
        assert np.array_equal(o_mid[r], expect_mid)
        assert np.array_equal(y[r], c * wo[:, 256 * h0 + e0])


def _tiny_batch():
    # two sequences, ragged, selections with -1 holes; cached rows N(0,1)
    bt = W.make_batch_np([40, 23], [3, 2], k=8, seed=91)
    rng = np.random.default_rng(92)
    idx = np.full((bt.total_q, 8), -1, np.int32)
    for r, (b, t) in enumerate(bt.positions()):
        n = min(8, t + 1) - (r % 2)
        idx[r, :n] = np.sort(rng.choice(t + 1, size=n, replace=False))
    return bt, idx


def test_expanded_equals_absorbed(weights):
    """The absorption identity: the pages' expanded path (kv_b_proj applied to
    every attended latent row) equals absorb_q -> attention on the latent rows
    -> W_UV -> o_proj."""
    bt, idx = _tiny_batch()
    qn, qp = W.make_mla_queries_np(bt.total_q, 93)
    o_exp, y_exp = oracle.mla_expanded(bt, qn, qp, weights.w_kvb, weights.w_o, idx)
    q_abs = oracle.mla_absorb_q(qn, qp, weights.w_kvb)
    # attention on the absorbed query, evaluated in fp64 here (no bf16 rounding of q)
    kv = _wf(bt.kv).reshape(-1, 576)
    o_lat = np.zeros((bt.total_q, 64, 512))
    for r, (b, t) in enumerate(bt.positions()):
        rows = kv[b * bt.stride + idx[r][idx[r] >= 0]]
        l = bt.sm_scale * q_abs[r] @ rows.T
        p = np.exp(l - l.max(axis=1, keepdims=True))
        o_lat[r] = (p / p.sum(axis=1, keepdims=True)) @ rows[:, :512]
    o_mid, y = oracle.mla_output(o_lat, weights.w_kvb, weights.w_o)
    assert np.allclose(o_exp, o_mid, rtol=1e-9, atol=1e-12)
    assert np.allclose(y_exp, y, rtol=1e-9, atol=1e-12)
    # and through the oracle's own attention routine on a bf16-exact query
    assert np.isfinite(y_exp).all() and np.abs(y_exp).max() > 0


def test_expanded_single_row_is_its_value(weights):
    bt, _ = _tiny_batch()
    idx = np.full((bt.total_q, 8), -1, np.int32)
    idx[:, 0] = 0                                          # every query attends to position 0 only
    qn, qp = W.make_mla_queries_np(bt.total_q, 94)
    o_mid, y = oracle.mla_expanded(bt, qn, qp, weights.w_kvb, weights.w_o, idx)
    wk = _wf(weights.w_kvb).reshape(64, 448, 512)
    kv = _wf(bt.kv).reshape(-1, 576)
    for r, (b, t) in enumerate(bt.positions()):
        v = np.einsum("hed,d->he", wk[:, 192:, :], kv[b * bt.stride, :512])    # W_UV[h] c_0
        assert np.allclose(o_mid[r], v, rtol=1e-12, atol=1e-12)


def test_wrappers_refuse_wrong_weight_sizes(weights):
    qn, qp = W.make_mla_queries_np(1, 5)
    with pytest.raises(ValueError):
        oracle.mla_absorb_q(qn, qp, weights.w_kvb[:100])
    with pytest.raises(ValueError):
        oracle.mla_output(np.zeros((1, 64, 512)), weights.w_kvb, weights.w_o[:10])
