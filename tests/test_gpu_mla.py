"""GPU parity of the MLA projections around the attention (absorbed query,
W_UV and o_proj) against the fp64 oracle, through the C ABI, and the whole
layer (absorb -> indexer -> top-k -> attention -> W_UV -> o_proj) against the
oracle's expanded path (kv_b_proj applied to every attended latent row).

Tolerances: each GEMM accumulates in fp32 and rounds its result to bf16
(relative 2^-9), so a projection is checked at |d| <= 4e-3 |ref| + 1e-4;
o_proj reads the bf16-rounded o_mid, whose rounding reaches y[t] in
proportion to the rms of row t (about 2^-9 / sqrt(3) of it per element), so
y is checked tightly against o_proj of the GPU's own o_mid and at
1e-2 |ref| + 2e-2 rms(row) against the oracle's y; the whole layer chains
five bf16 roundings and is checked at 2e-2 |ref| + 3e-2 rms(row).
"""

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_gb300 as dsa
import workloads as W
from dsa_case import Staged, bf16_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_attention_gb300 import build as B
    B.build()
    dsa.load_library()


@pytest.fixture(scope="module")
def weights():
    wn = W.make_mla_weights_np(11)
    return wn, bf16_dev(wn.w_kvb), bf16_dev(wn.w_o)


def _ws(T):
    return dsa.mla_workspace(T)


def _bits(t):
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _close(got, ref, rtol, atol, what):
    err = np.abs(got - ref) - (atol + rtol * np.abs(ref))
    assert err.max() <= 0, f"{what}: worst excess {err.max():.3g} at {np.unravel_index(np.argmax(err), err.shape)}"


@pytest.mark.parametrize("T", [1, 64, 300])
def test_absorb_q(weights, T):
    wn, w_kvb, _ = weights
    qn, qp = W.make_mla_queries_np(T, 100 + T)
    q_out = torch.full((T, 64, 576), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = _ws(T)
    dsa.mla_absorb_q(bf16_dev(qn), bf16_dev(qp), w_kvb, q_out, ws)
    assert dsa.read_device_status(ws) == 0
    ref = oracle.mla_absorb_q(qn, qp, wn.w_kvb)
    got = _f64(q_out)
    _close(got[:, :, :512], ref[:, :, :512], 4e-3, 1e-4, "q_lat")
    assert np.array_equal(_bits(q_out)[:, :, 512:], qp)          # the rope part is copied bit for bit


@pytest.mark.parametrize("T", [1, 64, 300, 700])
def test_output(weights, T):
    wn, w_kvb, w_o = weights
    rng = np.random.default_rng(200 + T)
    o_lat = W.bf16_bits_from_f32(rng.standard_normal((T, 64, 512), dtype=np.float32) * 0.3)
    o_mid = torch.full((T, 64 * 256), float("nan"), dtype=torch.bfloat16, device="cuda")
    y = torch.full((T, 6144), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = _ws(T)
    dsa.mla_output(bf16_dev(o_lat), w_kvb, w_o, o_mid, y, ws)
    assert dsa.read_device_status(ws) == 0
    ref_mid, ref_y = oracle.mla_output(W.f32_from_bf16_bits(o_lat).astype(np.float64), wn.w_kvb, wn.w_o)
    _close(_f64(o_mid).reshape(T, 64, 256), ref_mid, 4e-3, 1e-4, "o_mid")
    # o_proj of the GPU's own bf16 o_mid (numpy fp64), then the oracle's y
    y_own = _f64(o_mid) @ W.f32_from_bf16_bits(wn.w_o).astype(np.float64).T
    _close(_f64(y), y_own, 4e-3, 1e-4, "y vs o_proj(o_mid)")
    rms = np.sqrt(np.mean(ref_y ** 2, axis=1, keepdims=True))
    _close(_f64(y), ref_y, 1e-2, 2e-2 * rms, "y vs oracle")


def test_layer_against_the_expanded_path(weights):
    """absorb_q -> dsa_forward -> mla_output equals the pages' expanded path
    (kv_b_proj on every attended latent row, masked attention, o_proj) on the
    GPU's own selections."""
    wn, w_kvb, w_o = weights
    bt = W.make_batch_np([300, 129, 40], [5, 4, 3], k=32, seed=301, key_kind="lowrank16")
    qn, qp = W.make_mla_queries_np(bt.total_q, 302)
    st = Staged(bt)
    T = bt.total_q
    ws = _ws(T)
    q = torch.empty((T, 64, 576), dtype=torch.bfloat16, device="cuda")
    dsa.mla_absorb_q(bf16_dev(qn), bf16_dev(qp), w_kvb, q, ws)
    st.q = q
    out, lse, idx, _ = st.forward()
    assert st.status() == 0
    o_mid = torch.empty((T, 64 * 256), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((T, 6144), dtype=torch.bfloat16, device="cuda")
    dsa.mla_output(out, w_kvb, w_o, o_mid, y, ws)
    assert dsa.read_device_status(ws) == 0
    ref_mid, ref_y = oracle.mla_expanded(bt, qn, qp, wn.w_kvb, wn.w_o, idx.cpu().numpy())
    rms_mid = np.sqrt(np.mean(ref_mid ** 2, axis=(1, 2), keepdims=True))
    rms_y = np.sqrt(np.mean(ref_y ** 2, axis=1, keepdims=True))
    _close(_f64(o_mid).reshape(T, 64, 256), ref_mid, 2e-2, 3e-2 * rms_mid, "o_mid vs expanded")
    _close(_f64(y), ref_y, 2e-2, 3e-2 * rms_y, "y vs expanded")


@pytest.mark.parametrize("T", [64, 16384])
def test_projections_full_size(weights, T):
    """Decode (64 tokens) and prefill (16384 tokens) shapes; oracle on sampled rows."""
    wn, w_kvb, w_o = weights
    qn_t, qp_t = W.make_mla_queries_torch(T, 400 + T)
    q_out = torch.empty((T, 64, 576), dtype=torch.bfloat16, device="cuda")
    ws = _ws(T)
    dsa.mla_absorb_q(qn_t, qp_t, w_kvb, q_out, ws)
    g = torch.Generator(device="cuda")
    g.manual_seed(500 + T)
    o_lat = (torch.randn(T, 64, 512, generator=g, device="cuda") * 0.3).to(torch.bfloat16)
    o_mid = torch.empty((T, 64 * 256), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((T, 6144), dtype=torch.bfloat16, device="cuda")
    dsa.mla_output(o_lat, w_kvb, w_o, o_mid, y, ws)
    torch.cuda.synchronize()
    assert dsa.read_device_status(ws) == 0
    cand = {0, 1, 127, 128, T // 2, T - 2, T - 1} | set(np.random.default_rng(T).choice(T, 9).tolist())
    rows = sorted(r for r in cand if 0 <= r < T)
    assert rows and max(rows) < T                      # checked on the host before any device indexing
    ri = torch.tensor(rows, device="cuda")
    ref = oracle.mla_absorb_q(_bits(qn_t[ri]), _bits(qp_t[ri]), wn.w_kvb)
    _close(_f64(q_out[ri])[:, :, :512], ref[:, :, :512], 4e-3, 1e-4, "q_lat")
    ref_mid, ref_y = oracle.mla_output(_f64(o_lat[ri]), wn.w_kvb, wn.w_o)
    _close(_f64(o_mid[ri]).reshape(len(rows), 64, 256), ref_mid, 4e-3, 1e-4, "o_mid")
    rms = np.sqrt(np.mean(ref_y ** 2, axis=1, keepdims=True))
    _close(_f64(y[ri]), ref_y, 1e-2, 2e-2 * rms, "y")
