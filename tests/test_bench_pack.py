"""bench.py's end-to-end leg packs a step's host data (inputs of several
dtypes, then the new cache rows taken from strided views) into one block
that one copy moves: each tensor read back from the block must equal the
original bit for bit, start on a 256-byte boundary and be contiguous."""
import os
import sys

import pytest
import torch

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_pack_roundtrip_bits_and_alignment():
    g = torch.Generator().manual_seed(7)
    B, stride = 5, 9
    kv = torch.randn(B * stride, 576, generator=g).to(torch.bfloat16)
    ks = torch.randn(B * stride, generator=g)
    srcs = [("q_idx", torch.randn(B, 32, 128, generator=g).to(torch.bfloat16)),
            ("w", torch.randn(B, 32, generator=g)),
            ("q", torch.randn(B, 64, 576, generator=g).to(torch.bfloat16)),
            ("idx", torch.randint(-1, 1000, (B, 7), generator=g, dtype=torch.int32)),
            ("row:kv", kv.view(B, stride, 576)[:, stride - 1].contiguous()),
            ("row:ks", ks.view(B, stride)[:, stride - 1].contiguous())]
    segs, nbytes = bench.pack_layout(srcs)
    assert nbytes % 256 == 0
    blk = torch.full((nbytes,), 0xA5, dtype=torch.uint8)
    bench.pack_into(blk, segs, srcs)
    prev_end = 0
    for n, t in srcs:
        v = bench.seg_view(blk, segs, n)
        o0 = segs[n][0]
        assert o0 % 256 == 0 and o0 >= prev_end
        prev_end = o0 + segs[n][1]
        assert v.is_contiguous() and v.dtype == t.dtype and v.shape == t.shape
        assert torch.equal(v.reshape(-1).view(torch.uint8), t.reshape(-1).view(torch.uint8)), n
    assert prev_end <= nbytes


def test_scatter_of_staged_rows_touches_only_those_rows():
    B, stride, width = 4, 6, 16
    cache = torch.arange(B * stride * width, dtype=torch.float32).view(B * stride, width)
    before = cache.clone()
    new = torch.full((B, width), -1.0)
    segs, nbytes = bench.pack_layout([("row:c", new)])
    blk = torch.zeros(nbytes, dtype=torch.uint8)
    bench.pack_into(blk, segs, [("row:c", new)])
    row = cache.view(B, stride, width)[:, stride - 1]
    row.copy_(bench.seg_view(blk, segs, "row:c"))
    c3, b3 = cache.view(B, stride, width), before.view(B, stride, width)
    assert torch.equal(c3[:, stride - 1], new)
    assert torch.equal(c3[:, :stride - 1], b3[:, :stride - 1])


@pytest.mark.parametrize("align", [16, 256])
def test_layout_of_empty_and_odd_sizes(align):
    srcs = [("a", torch.zeros(0, dtype=torch.float32)), ("b", torch.zeros(3, dtype=torch.uint8)),
            ("c", torch.zeros(5, dtype=torch.bfloat16))]
    segs, nbytes = bench.pack_layout(srcs, align)
    assert segs["a"][0] == 0 and segs["a"][1] == 0
    assert segs["b"][0] == 0 and segs["c"][0] == align
    assert nbytes == 2 * align
