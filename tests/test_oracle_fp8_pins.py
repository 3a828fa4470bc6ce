"""CPU pins of the oracle's reduced-precision index keys: the E4M3 codec
against the format's definition (every code), rounding (midpoints, ties to
even, saturation), the absmax quantization, and the FP8 scores against the
bf16 scores within the quantization error.  The recipe itself (E4M3,
per-key / per-(token, head) absmax scales) is a reading: the pages give no
FP8 recipe for the indexer, so which quantization the method uses is
unpinned; its arithmetic is pinned here."""

import numpy as np

import oracle
import workloads as W


def test_every_e4m3_code_decodes_by_definition():
    codes = np.arange(256, dtype=np.uint8)
    v = oracle.e4m3_decode(codes)
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            assert np.isnan(v[c])
            continue
        mag = (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        assert v[c] == (-mag if s else mag), c
    finite = v[~np.isnan(v)]
    assert finite.max() == 448.0 and finite.min() == -448.0
    assert np.sum(np.isnan(v)) == 2                       # 0x7F and 0xFF


def test_encode_round_trips_and_rounds_to_nearest_even():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    v = oracle.e4m3_decode(codes)
    back = oracle.e4m3_encode(v)
    assert np.array_equal(oracle.e4m3_decode(back), v)    # exact values encode to themselves (+-0 equal)
    pos = np.sort(np.unique(v[v >= 0]))
    mids = (pos[:-1] + pos[1:]) / 2
    enc = oracle.e4m3_encode(mids)
    lo = oracle.e4m3_encode(pos[:-1])
    hi = oracle.e4m3_encode(pos[1:])
    # a midpoint goes to whichever neighbour has the even code
    assert np.all(enc == np.where(lo % 2 == 0, lo, hi))
    # just off the midpoint it goes to the nearer neighbour
    assert np.array_equal(oracle.e4m3_encode(mids * (1 - 1e-9)), lo)
    assert np.array_equal(oracle.e4m3_encode(mids * (1 + 1e-9)), hi)
    assert oracle.e4m3_decode(oracle.e4m3_encode([1e6, -1e6, 449.0])).tolist() == [448.0, -448.0, 448.0]


def test_quantize_scales_to_448_and_bounds_the_error():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((50, 128)).astype(np.float32) * rng.uniform(0.01, 10, (50, 1)).astype(np.float32)
    x[7] = 0.0
    bits = W.bf16_bits_from_f32(x)
    codes, scale = oracle.quantize_fp8(bits, 128)
    xf = W.f32_from_bf16_bits(bits).astype(np.float64)
    deq = oracle.e4m3_decode(codes) * scale[:, None]
    assert scale[7] == 1.0 and np.all(codes[7] == 0)
    amax = np.abs(xf).max(axis=1)
    ok = amax > 0
    # the largest maps to +-448; the single-precision scale keeps 448 * scale within 2^-23 of amax
    assert np.allclose(np.abs(deq[ok]).max(axis=1), amax[ok], rtol=2.0 ** -22)
    # nearest rounding: within half a step (2^-4 relative for normals, 2^-10 * scale for subnormals)
    err = np.abs(deq - xf)
    assert np.all(err <= np.maximum(np.abs(xf) * 2.0 ** -4, scale[:, None] * 2.0 ** -10) * (1 + 1e-12))


def test_fp8_scores_follow_the_bf16_scores():
    bt = W.make_batch_np([200], [6], k=16, seed=9)
    q8, qs = oracle.quantize_fp8(bt.q_idx, 128)
    k8, ks = oracle.quantize_fp8(bt.k_idx, 128)
    ref = oracle.indexer_scores(bt)
    got = oracle.indexer_scores_fp8(bt, q8.reshape(-1), qs, k8.reshape(-1), ks)
    # exact identity with the dequantised values fed to the bf16 formula
    deq_q = oracle.e4m3_decode(q8) * qs[:, None]
    deq_k = oracle.e4m3_decode(k8) * ks[:, None]
    w = bt.w.astype(np.float64)
    for j, (_, t) in enumerate(bt.positions()):
        d = deq_q.reshape(bt.total_q, 32, 128)[j] @ deq_k[:t + 1].T
        assert np.allclose(got[j, :t + 1], (w[j][:, None] * np.maximum(d, 0)).sum(0), rtol=1e-12, atol=1e-14)
    # and close to the unquantised scores (3 mantissa bits on both operands)
    for j, (_, t) in enumerate(bt.positions()):
        e = np.abs(got[j, :t + 1] - ref[j, :t + 1])
        assert np.median(e / (np.abs(ref[j, :t + 1]) + 1e-3)) < 0.1
