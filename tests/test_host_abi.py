"""CPU-only checks of the C ABI: the library builds and loads, exports every
symbol include/dsa.h declares, and its host-side argument checks reject bad
calls before any CUDA work (no compute call runs here)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_gb300 import build as B
    B.build()
    import sparse_attention_gb300 as dsa
    return dsa.load_library()


def _declared_symbols():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            names.update(re.findall(r"DSA_API\s+[\w\s\*]+?\b(dsa_\w+)\s*\(", text))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = _declared_symbols()
    assert {"dsa_indexer_scores", "dsa_topk", "dsa_sparse_mla_fwd", "dsa_forward"} <= names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_strings(lib):
    assert lib.dsa_status_string(0) == b"DSA_OK"
    for code in range(1, 9):
        assert lib.dsa_status_string(code).startswith(b"DSA_ERR_")
    assert lib.dsa_status_string(99) == b"unknown dsa_status"


def _batch(B=1, total_q=4, max_q=4, max_ctx=16, stride=16, q_off=0x10000, ctx=0x20000):
    import sparse_attention_gb300 as dsa
    return dsa.DsaBatch(B, total_q, max_q, max_ctx, stride, q_off, ctx)


def _ws_size(lib, b, k):
    n = ctypes.c_size_t(0)
    rc = lib.dsa_workspace_size(ctypes.byref(b), k, ctypes.byref(n))
    return rc, n.value


def test_workspace_size_checks(lib):
    rc, n = _ws_size(lib, _batch(), 8)
    assert rc == 0 and n >= 256 and n % 256 == 0
    assert _ws_size(lib, _batch(B=0), 8)[0] == 1
    assert _ws_size(lib, _batch(), 0)[0] == 1
    assert _ws_size(lib, _batch(), 2049)[0] == 1
    assert _ws_size(lib, _batch(stride=8), 8)[0] == 1          # stride < max_ctx
    assert _ws_size(lib, _batch(q_off=0), 8)[0] == 1           # null device array
    # decode batch: 64 sequences x 32768, k = 2048 -> split-K partials included
    rc, n = _ws_size(lib, _batch(B=64, total_q=64, max_q=1, max_ctx=32768, stride=32768), 2048)
    assert rc == 0 and n > 64 * 32768 * 4


def test_compute_entry_points_reject_bad_host_arguments(lib):
    b = _batch()
    rc, n = _ws_size(lib, b, 8)
    ws = 0x7f0000000000          # never dereferenced: every call below fails its host check
    p = 0x7f0000100000
    bad = p + 8                  # not 16-byte aligned
    B = ctypes.byref(b)
    # workspace missing / too small
    assert lib.dsa_topk(B, p, 16, 8, p, None, n, None) == 3
    assert lib.dsa_sparse_mla_fwd(B, p, p, p, 8, ctypes.c_float(0.0625), p, None, ws, n - 256, None) == 3
    # bad k, misaligned pointers, short ld, bad scale
    assert lib.dsa_topk(B, p, 16, 0, p, ws, n, None) == 1
    assert lib.dsa_topk(B, bad, 16, 8, p, ws, n, None) == 1
    assert lib.dsa_topk(B, p, 12, 8, p, ws, n, None) == 1              # ld < max_ctx
    assert lib.dsa_topk(B, p, 18, 8, p, ws, n, None) == 1              # ld % 4 != 0
    assert lib.dsa_indexer_scores(B, bad, p, p, p, 16, ws, n, None) == 1
    assert lib.dsa_indexer_scores(B, p, p, None, p, 16, ws, n, None) == 1
    assert lib.dsa_sparse_mla_fwd(B, p, p, p, 8, ctypes.c_float(-1.0), p, None, ws, n, None) == 1
    assert lib.dsa_forward(B, p, p, p, p, p, 8, ctypes.c_float(0.0625), bad, None, None, None, 0, ws, n, None) == 1
    # an empty batch is a no-op
    e = _batch(total_q=0, max_q=0)
    assert lib.dsa_forward(ctypes.byref(e), p, p, p, p, p, 8, ctypes.c_float(0.0625), p, None, None, None, 0,
                           ws, _ws_size(lib, e, 8)[1], None) == 0
    # MLA projections: bad sizes, missing workspace, null or misaligned pointers
    assert lib.dsa_mla_absorb_q(-1, p, p, p, p, ws, 256, None) == 1
    assert lib.dsa_mla_absorb_q(4, p, p, p, p, None, 0, None) == 3
    assert lib.dsa_mla_absorb_q(4, None, p, p, p, ws, 256, None) == 1
    assert lib.dsa_mla_absorb_q(4, p, bad, p, p, ws, 256, None) == 1
    assert lib.dsa_mla_absorb_q(0, None, None, None, None, ws, 256, None) == 0
    m = ctypes.c_size_t(0)
    assert lib.dsa_mla_workspace_size(4, ctypes.byref(m)) == 0
    assert lib.dsa_mla_output(1 << 26, p, p, p, p, p, ws, m.value, None) == 1
    assert lib.dsa_mla_output(4, p, p, p, p, None, ws, m.value, None) == 1
    assert lib.dsa_mla_output(4, p, p, p, p, p, ws, 100, None) == 3
    assert lib.dsa_mla_workspace_size(64, ctypes.byref(m)) == 0 and m.value > 64 * 6144 * 4   # split-K partials
    assert lib.dsa_mla_output(64, p, p, p, p, p, ws, m.value - 256, None) == 3
    assert lib.dsa_mla_workspace_size(-1, ctypes.byref(m)) == 1
    # index-key producer: workspace, pointers, eps
    assert lib.dsa_index_key_workspace_size(4, ctypes.byref(m)) == 0 and m.value >= 256
    assert lib.dsa_index_key_producer(B, p, p, p, p, ctypes.c_float(1e-5), p, p, p, p, p, ws, 100, None) == 3
    assert lib.dsa_index_key_producer(B, p, p, p, p, ctypes.c_float(0.0), p, p, p, p, p, ws, m.value, None) == 1
    assert lib.dsa_index_key_producer(B, p, None, p, p, ctypes.c_float(1e-5), p, p, p, p, p, ws, m.value, None) == 1
    assert lib.dsa_index_key_producer(B, p, p, p, bad, ctypes.c_float(1e-5), p, p, p, p, p, ws, m.value, None) == 1
    # FP8 index keys: quantizer and forward host checks
    assert lib.dsa_quantize_fp8(-1, p, p, p, None) == 1
    assert lib.dsa_quantize_fp8(4, bad, p, p, None) == 1
    assert lib.dsa_quantize_fp8(0, None, None, None, None) == 0
    assert lib.dsa_indexer_scores_fp8(B, p, p, p, p, None, p, 16, ws, n, None) == 1
    assert lib.dsa_forward_fp8(B, p, p, p, p, p, p, p, 8, ctypes.c_float(0.0625), p, None, None, None, 0, ws, n - 256,
                               None) == 3
    # status word helpers check their pointers on the host
    assert lib.dsa_read_device_status(None, None, None) == 1
    assert lib.dsa_reset_device_status(None, None) == 3


def test_product_has_no_oracle_dependency():
    """The product package neither imports nor links the oracle."""
    pkg = os.path.join(ROOT, "sparse_attention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "liboracle" not in text and "oracle.c" not in text, f


def test_noalloc_host_checks_and_error_record(lib):
    """The allocation-free attention call rejects bad arguments on the host,
    refuses partials beyond its static array before any CUDA call, and a
    failing CUDA call is reported by dsa_last_cuda_error like every other
    entry point's."""
    import torch
    b = _batch()
    p = 0x7f0000100000
    B = ctypes.byref(b)
    f = lib.dsa_sparse_mla_fwd_noalloc
    assert f(B, p, p, p, 0, ctypes.c_float(0.0625), p, None, None, None) == 1          # k < 1
    assert f(B, p + 8, p, p, 8, ctypes.c_float(0.0625), p, None, None, None) == 1      # misaligned q
    assert f(B, p, p, p, 8, ctypes.c_float(0.0), p, None, None, None) == 1             # bad scale
    big = _batch(total_q=100, max_q=100, max_ctx=4096, stride=4096)
    assert f(ctypes.byref(big), p, p, p, 2047, ctypes.c_float(0.0625), p, None, None, None) == 3
    if torch.cuda.is_available():
        pytest.skip("the error-record check needs a host without a CUDA device")
    # no device here: the address lookup fails before anything is launched
    assert f(B, p, p, p, 8, ctypes.c_float(0.0625), p, None, None, None) == 4          # DSA_ERR_CUDA
    assert lib.dsa_last_cuda_error() != b"no error"
