"""GPU parity of the index-key producer (wk -> LayerNorm(128) -> rotate-half
RoPE on the first 64 dims -> cache append; weights_proj * 32^-1/2) against the
fp64 oracle, through the C ABI.

Tolerances: the projections accumulate in fp32 over 6144 terms (~1e-6
relative) and k is stored as bf16 (relative 2^-9), so k is checked at
|d| <= 8e-3 |ref| + 1e-3 and the fp32 w at |d| <= 1e-3 |ref| + 1e-5.  Every
cache row that is not a new token's must keep its bits.
"""

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_gb300 as dsa
import workloads as W
from dsa_case import bf16_dev

pytestmark = pytest.mark.gpu

SENTINEL = 0x3F80          # bf16 1.0: a value the producer never writes by chance


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_attention_gb300 import build as B
    B.build()
    dsa.load_library()


@pytest.fixture(scope="module")
def params():
    p = W.make_index_key_params_np(31)
    dev = dict(wk=bf16_dev(p.wk), ww=bf16_dev(p.ww), gamma=torch.from_numpy(p.gamma).cuda(),
               beta=torch.from_numpy(p.beta).cuda())
    return p, dev


def _close(got, ref, rtol, atol, what):
    err = np.abs(got - ref) - (atol + rtol * np.abs(ref))
    assert err.max() <= 0, f"{what}: worst excess {err.max():.3g} at {np.unravel_index(np.argmax(err), err.shape)}"


def _run(params, ctx, new, stride, seed, check_rows=None):
    p, dev = params
    B = len(ctx)
    q_off = np.concatenate([[0], np.cumsum(new)]).astype(np.int32)
    T = int(q_off[-1])
    pos = np.concatenate([np.arange(c - n, c) for c, n in zip(ctx, new)])
    seq = np.concatenate([np.full(n, b) for b, n in enumerate(new)])
    x = W.make_hidden_np(T, seed)
    cos, sin = W.rotary_rows(pos)
    b = dsa.make_batch(q_off, ctx, max(new), max(ctx), stride)
    cache = torch.full((B * stride, 128), 0, dtype=torch.int16, device="cuda")
    cache.fill_(SENTINEL)
    k_idx = cache.view(torch.bfloat16)
    w_out = torch.full((T, 32), float("nan"), dtype=torch.float32, device="cuda")
    ws = dsa.index_key_workspace(T)
    dsa.index_key_producer(b, bf16_dev(x), dev["wk"], dev["gamma"], dev["beta"], p.eps, torch.from_numpy(cos).cuda(),
                           torch.from_numpy(sin).cuda(), dev["ww"], k_idx, w_out, ws)
    assert dsa.read_device_status(ws) == 0
    got = cache.cpu().numpy().view(np.uint16)
    rows = np.arange(T) if check_rows is None else np.asarray(check_rows)
    k_ref, w_ref = oracle.index_key(x[rows], p.wk, p.gamma, p.beta, p.eps, cos[rows], sin[rows], p.ww)
    cache_rows = seq[rows] * stride + pos[rows]
    _close(W.f32_from_bf16_bits(got[cache_rows]).astype(np.float64), k_ref, 8e-3, 1e-3, "k")
    _close(w_out.cpu().numpy()[rows].astype(np.float64), w_ref, 1e-3, 1e-5, "w")
    # every other row of the cache keeps its bits
    written = np.zeros(B * stride, bool)
    written[seq * stride + pos] = True
    assert np.all(got[~written] == SENTINEL)
    return got


def test_ragged_batch(params):
    # 136 new tokens over three sequences (two 128-row tiles, a single-token sequence)
    _run(params, ctx=[40, 77, 300], new=[5, 1, 130], stride=320, seed=41)


def test_decode_shape_splits_k(params):
    # 64 sequences, one new token each: few rows, so the products split over K
    _run(params, ctx=[32768 - j for j in range(64)], new=[1] * 64, stride=32768, seed=42)


def test_prefill_shape(params):
    T = 16384
    rows = sorted({0, 1, 127, 128, 4095, 8192, T - 1} | set(np.random.default_rng(43).choice(T, 9).tolist()))
    _run(params, ctx=[T], new=[T], stride=T, seed=43, check_rows=rows)
