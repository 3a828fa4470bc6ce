"""CPU pins of the oracle's index-key producer (wk -> LayerNorm(128) -> RoPE on
the first 64 dims; weights_proj * 32^-1/2) against closed forms and an
independent numpy evaluation."""

import numpy as np
import pytest

import oracle
import workloads as W


@pytest.fixture(scope="module")
def params():
    return W.make_index_key_params_np(21)


def _wf(bits):
    return W.f32_from_bf16_bits(bits).astype(np.float64)


def test_layernorm_alone_has_zero_mean_unit_variance(params):
    T = 5
    x = W.make_hidden_np(T, 22)
    ones, zeros = np.ones(128), np.zeros(128)
    cos, sin = np.ones((T, 64)), np.zeros((T, 64))            # rotation by 0
    k, _ = oracle.index_key(x, params.wk, ones, zeros, 1e-5, cos, sin, params.ww)
    y = _wf(x) @ _wf(params.wk).T
    var_y = y.var(axis=1)
    assert np.allclose(k.mean(axis=1), 0.0, atol=1e-12)
    assert np.allclose(k.var(axis=1), var_y / (var_y + 1e-5), rtol=1e-12)


def test_rope_rotates_pairs_i_and_i_plus_32(params):
    T = 4
    x = W.make_hidden_np(T, 23)
    pos = [0, 1, 1000, 202751]
    cos, sin = W.rotary_rows(pos)
    k, _ = oracle.index_key(x, params.wk, params.gamma, params.beta, params.eps, cos, sin, params.ww)
    k0, _ = oracle.index_key(x, params.wk, params.gamma, params.beta, params.eps, np.ones((T, 64)),
                             np.zeros((T, 64)), params.ww)
    c, s = cos.astype(np.float64)[:, :32], sin.astype(np.float64)[:, :32]
    a, b = k0[:, :32], k0[:, 32:64]
    assert np.allclose(k[:, :32], a * c - b * s, rtol=1e-12, atol=1e-12)     # 2-D rotation of (a, b)
    assert np.allclose(k[:, 32:64], b * c + a * s, rtol=1e-12, atol=1e-12)
    assert np.array_equal(k[:, 64:], k0[:, 64:])                             # the nope half is untouched
    assert np.allclose(k[0], k0[0])                                          # position 0: no rotation
    # norms kept up to the fp32 rounding of the cos / sin rows (cos^2 + sin^2 = 1 within 1e-7)
    assert np.allclose(a ** 2 + b ** 2, k[:, :32] ** 2 + k[:, 32:64] ** 2, rtol=1e-6)


def test_index_key_matches_numpy(params):
    T = 6
    x = W.make_hidden_np(T, 24)
    cos, sin = W.rotary_rows(np.arange(T) * 37 + 5)
    k, w = oracle.index_key(x, params.wk, params.gamma, params.beta, params.eps, cos, sin, params.ww)
    xf = _wf(x)
    y = xf @ _wf(params.wk).T
    z = (y - y.mean(1, keepdims=True)) / np.sqrt(y.var(1, keepdims=True) + params.eps)
    z = z * params.gamma.astype(np.float64) + params.beta.astype(np.float64)
    rot = np.concatenate([-z[:, 32:64], z[:, :32]], axis=1)
    ref = z.copy()
    ref[:, :64] = z[:, :64] * cos + rot * sin
    assert np.allclose(k, ref, rtol=1e-10, atol=1e-12)
    assert np.allclose(w, xf @ _wf(params.ww).T / np.sqrt(32.0), rtol=1e-12, atol=1e-14)


def test_head_weights_one_hot_rows(params):
    """weights_proj rows that are one-hot, row h = a_h at column c_h, give
    w[t, h] = a_h * x[t, c_h] / sqrt(32) exactly ("GLM-5.1 架构深度拆解" §3.6
    Step 4: the head weight is weights_proj(x) times H_idx^-1/2 with
    H_idx = 32).  The columns differ per head and the factors per head, so a
    transposed weight, a reading of x by head index, or any other factor
    (1/32, sqrt(32), 1/sqrt(128)) fails."""
    T = 3
    x = W.make_hidden_np(T, 26)
    cols = (np.arange(32) * 193 + 7) % 6144
    a = np.array([(-1.0) ** h * 2.0 ** (h % 5 - 2) for h in range(32)], np.float32)
    ww = np.zeros((32, 6144), np.uint16)
    ww[np.arange(32), cols] = W.bf16_bits_from_f32(a)
    _, w = oracle.index_key(x, params.wk, params.gamma, params.beta, params.eps,
                            np.ones((T, 64)), np.zeros((T, 64)), ww)
    xf = _wf(x)
    for h in range(32):
        assert np.array_equal(w[:, h], a[h] * xf[:, cols[h]] / np.sqrt(32.0))
    # a one-hot token x = e_c reads column c of weights_proj: w[h] = ww[h, c] / sqrt(32)
    c = 4099
    xe = np.zeros((1, 6144), np.uint16)
    xe[0, c] = W.bf16_bits_from_f32(np.array([1.0], np.float32))[0]
    _, w1 = oracle.index_key(xe, params.wk, params.gamma, params.beta, params.eps,
                             np.ones((1, 64)), np.zeros((1, 64)), params.ww)
    assert np.array_equal(w1[0], _wf(params.ww)[:, c] / np.sqrt(32.0))


def test_wrapper_refuses_wrong_sizes(params):
    x = W.make_hidden_np(2, 25)
    cos, sin = W.rotary_rows([0, 1])
    with pytest.raises(ValueError):
        oracle.index_key(x, params.wk[:10], params.gamma, params.beta, 1e-5, cos, sin, params.ww)
    with pytest.raises(ValueError):
        oracle.index_key(x, params.wk, params.gamma, params.beta, 1e-5, cos[:1], sin, params.ww)
