"""GPU parity of the E4M3 index-key path against the fp64 oracle, through the
C ABI: the row quantizer bit for bit (codes and fp32 scales), indexer scores
on the quantized queries / keys within 1e-3 (1 + |ref|), top-k bit-exact on
the GPU's scores, attention on the selections, forward == steps.  (Which FP8
recipe the method uses is a reading -- the pages give none; its arithmetic
is what is checked here.)"""

import numpy as np
import pytest
import torch

import oracle
import sparse_attention_gb300 as dsa
import workloads as W
from dsa_case import SCORE_RTOL, Staged, check_attention

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from sparse_attention_gb300 import build as B
    B.build()
    dsa.load_library()


def _quant(x_dev, rows):
    codes = torch.empty((rows, 128), dtype=torch.uint8, device="cuda")
    scale = torch.empty(rows, dtype=torch.float32, device="cuda")
    dsa.quantize_fp8(x_dev, codes, scale)
    return codes, scale


def test_quantizer_bit_exact():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((300, 128)).astype(np.float32) * rng.uniform(1e-3, 1e3, (300, 1)).astype(np.float32)
    x[5] = 0.0                                           # an all-zero row
    x[6] = 0.0
    x[6, 3] = -2.5                                       # one nonzero value: it maps to -448
    x[7] = np.linspace(-1, 1, 128)                       # many values between codes
    bits = W.bf16_bits_from_f32(x)
    codes, scale = _quant(torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16), 300)
    ref_c, ref_s = oracle.quantize_fp8(bits, 128)
    got_c = codes.cpu().numpy()
    bad = np.argwhere(got_c != ref_c)
    assert len(bad) == 0, f"{len(bad)} codes differ, first at {bad[0]}: {got_c[tuple(bad[0])]:#x} vs {ref_c[tuple(bad[0])]:#x}"
    assert np.array_equal(scale.cpu().numpy().astype(np.float64), ref_s)
    assert got_c[6, 3] == 0xFE and ref_s[5] == 1.0


def _fp8_case(bt):
    st = Staged(bt)
    T = bt.total_q
    q8, qs = _quant(st.q_idx, T * 32)
    k8, ks = _quant(st.k_idx, bt.B * bt.stride)
    return st, q8, qs, k8, ks


@pytest.mark.parametrize("shape", ["ragged_prefill", "decode"])
def test_fp8_path(shape):
    if shape == "ragged_prefill":
        bt = W.make_batch_np([300, 190, 1, 129, 257], [300, 2, 1, 64, 19], k=64, seed=61, key_kind="lowrank16")
    else:
        bt = W.make_batch_np([1000, 2500, 128, 4097], [1] * 4, k=512, seed=62, key_kind="zipf")
    st, q8, qs, k8, ks = _fp8_case(bt)
    sc = st.new_scores()
    dsa.indexer_scores_fp8(st.b, q8, qs, st.w, k8, ks, sc, ws=st.ws)
    assert st.status() == 0
    ref = oracle.indexer_scores_fp8(bt, q8.cpu().numpy().reshape(-1), qs.cpu().numpy().astype(np.float64),
                                    k8.cpu().numpy().reshape(-1), ks.cpu().numpy().astype(np.float64), ld=st.ld)
    got = sc.cpu().numpy().astype(np.float64)
    for r, (_, t) in enumerate(bt.positions()):
        d = np.abs(got[r, :t + 1] - ref[r, :t + 1])
        assert np.all(d <= SCORE_RTOL * (1 + np.abs(ref[r, :t + 1]))), f"row {r}: max err {d.max():.3g}"
        assert np.all(np.isnan(got[r, t + 1:]))
    # the fused call equals the step calls; top-k on the GPU's scores; attention
    out = torch.empty((bt.total_q, 64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((bt.total_q, 64), dtype=torch.float32, device="cuda")
    idx = torch.empty((bt.total_q, bt.k), dtype=torch.int32, device="cuda")
    sc2 = st.new_scores()
    dsa.forward_fp8(st.b, q8, qs, st.w, k8, ks, st.q, st.kv, bt.k, bt.sm_scale, out, lse, idx_out=idx, scores_out=sc2,
                    ws=st.ws)
    assert st.status() == 0
    for r, (_, t) in enumerate(bt.positions()):
        assert torch.equal(sc2[r, :t + 1], sc[r, :t + 1])
    assert np.array_equal(idx.cpu().numpy(), oracle.topk(bt, np.nan_to_num(got.astype(np.float32), nan=0.0), k=bt.k))
    check_attention(st, idx, out, lse)


def test_fp8_decode_full_size():
    wl = W.WORKLOADS["decode_B64_ctx32768"]
    bt = W.make_batch_torch([wl.ctx] * wl.B, [1] * wl.B, wl.k, wl.seed, key_kind=wl.key_kind)
    b = dsa.Batch(bt.q_off, bt.ctx_len, 1, wl.ctx, bt.stride, total_q=wl.B)
    q8, qs = _quant(bt.q_idx, wl.B * 32)
    k8, ks = _quant(bt.k_idx, wl.B * bt.stride)
    ws = dsa.workspace(b, wl.k)
    out = torch.empty((wl.B, 64, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((wl.B, 64), dtype=torch.float32, device="cuda")
    idx = torch.empty((wl.B, wl.k), dtype=torch.int32, device="cuda")
    sc = torch.full((wl.B, wl.ctx), float("nan"), dtype=torch.float32, device="cuda")
    dsa.forward_fp8(b, q8, qs, bt.w, k8, ks, bt.q, bt.kv, wl.k, bt.sm_scale, out, lse, idx_out=idx, scores_out=sc,
                    ws=ws)
    torch.cuda.synchronize()
    assert dsa.read_device_status(ws) == 0
    # top-k on every row; scores of three rows against the oracle
    lay = W.Batch(B=wl.B, stride=bt.stride, q_off=np.arange(wl.B + 1, dtype=np.int32),
                  ctx_len=np.full(wl.B, wl.ctx, np.int32), q_idx=None, w=bt.w.cpu().numpy(), k_idx=None, q=None,
                  kv=None, k=wl.k, sm_scale=W.SM_SCALE)
    got = sc.cpu().numpy()
    assert np.array_equal(idx.cpu().numpy(), oracle.topk(lay, got, k=wl.k))
    rows = [0, 31, 63]
    k8h, ksh = k8.cpu().numpy().reshape(-1), ks.cpu().numpy().astype(np.float64)
    ref = oracle.indexer_scores_fp8(lay, q8.cpu().numpy().reshape(-1), qs.cpu().numpy().astype(np.float64), k8h, ksh,
                                    rows=rows, ld=wl.ctx)
    for j, r in enumerate(rows):
        assert np.all(np.abs(got[r] - ref[j]) <= SCORE_RTOL * (1 + np.abs(ref[j])))
