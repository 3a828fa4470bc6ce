"""Python binding of libdsa.so -- the GLM-5 DSA attention hot path
(lightning indexer -> causal top-k -> sparse MLA) on one GB300.

Argument marshalling only: every step runs in the CUDA kernels of
``libdsa.so`` (C ABI in ``include/dsa.h``).  PyTorch supplies device memory
and the current stream.  There is no fallback: if the library is missing or
no CUDA device is present the calls raise.

    import sparse_attention_gb300 as dsa
    b  = dsa.make_batch(q_off, ctx_len, max_q, max_ctx, cache_stride)
    ws = dsa.workspace(b, k)
    dsa.forward(b, q_idx, w, k_idx, q, kv, k, sm_scale, out, lse, ws=ws)
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")

H_IDX, D_IDX, H, D_QK, D_V, MAX_TOPK = 32, 128, 64, 576, 512, 2048

STATUS = {
    0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_UNSUPPORTED", 3: "DSA_ERR_WORKSPACE",
    4: "DSA_ERR_CUDA", 5: "DSA_ERR_TIMEOUT", 6: "DSA_ERR_BAD_BATCH", 7: "DSA_ERR_BAD_INDEX", 8: "DSA_ERR_INTERNAL",
}

EXPORTS = ("dsa_status_string", "dsa_last_cuda_error", "dsa_kernel_launch_count", "dsa_workspace_size", "dsa_reset_device_status", "dsa_read_device_status",
           "dsa_selftest_wait_timeout", "dsa_indexer_scores", "dsa_topk", "dsa_sparse_mla_fwd",
           "dsa_sparse_mla_fwd_noalloc", "dsa_forward", "dsa_mla_absorb_q", "dsa_mla_workspace_size", "dsa_mla_output", "dsa_index_key_workspace_size",
           "dsa_index_key_producer", "dsa_quantize_fp8", "dsa_indexer_scores_fp8", "dsa_forward_fp8")


class DsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = f"{where}: {STATUS.get(code, code)}"
        if code == 4 and _lib is not None:
            msg += f" ({_lib.dsa_last_cuda_error().decode()})"
        super().__init__(msg)


class DsaBatch(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("total_q", ctypes.c_int32), ("max_q", ctypes.c_int32),
                ("max_ctx", ctypes.c_int32), ("cache_stride", ctypes.c_int64),
                ("q_off", ctypes.c_void_p), ("ctx_len", ctypes.c_void_p)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libdsa.so (build it first with ``python -m sparse_attention_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libdsa.so not found at {path}; build it with "
                           f"`python -m sparse_attention_gb300.build` (no CPU fallback exists)")
    lib = ctypes.CDLL(path)
    P, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    BP = ctypes.POINTER(DsaBatch)
    lib.dsa_status_string.restype = ctypes.c_char_p
    lib.dsa_status_string.argtypes = [i32]
    lib.dsa_last_cuda_error.restype = ctypes.c_char_p
    lib.dsa_last_cuda_error.argtypes = []
    lib.dsa_kernel_launch_count.restype = ctypes.c_uint64
    lib.dsa_kernel_launch_count.argtypes = []
    lib.dsa_workspace_size.argtypes = [BP, i32, ctypes.POINTER(sz)]
    lib.dsa_reset_device_status.argtypes = [P, P]
    lib.dsa_read_device_status.argtypes = [P, P, ctypes.POINTER(ctypes.c_int)]
    lib.dsa_indexer_scores.argtypes = [BP, P, P, P, P, i64, P, sz, P]
    lib.dsa_topk.argtypes = [BP, P, i64, i32, P, P, sz, P]
    lib.dsa_sparse_mla_fwd.argtypes = [BP, P, P, P, i32, f32, P, P, P, sz, P]
    lib.dsa_sparse_mla_fwd_noalloc.argtypes = [BP, P, P, P, i32, f32, P, P, P, P]
    lib.dsa_selftest_wait_timeout.argtypes = [P, ctypes.c_uint32, P]
    lib.dsa_forward.argtypes = [BP, P, P, P, P, P, i32, f32, P, P, P, P, i64, P, sz, P]
    lib.dsa_mla_absorb_q.argtypes = [i32, P, P, P, P, P, sz, P]
    lib.dsa_mla_output.argtypes = [i32, P, P, P, P, P, P, sz, P]
    lib.dsa_mla_workspace_size.argtypes = [i32, ctypes.POINTER(sz)]
    lib.dsa_index_key_workspace_size.argtypes = [i32, ctypes.POINTER(sz)]
    lib.dsa_index_key_producer.argtypes = [BP, P, P, P, P, f32, P, P, P, P, P, P, sz, P]
    lib.dsa_quantize_fp8.argtypes = [i64, P, P, P, P]
    lib.dsa_indexer_scores_fp8.argtypes = [BP, P, P, P, P, P, P, i64, P, sz, P]
    lib.dsa_forward_fp8.argtypes = [BP, P, P, P, P, P, P, P, i32, f32, P, P, P, P, i64, P, sz, P]
    for name in EXPORTS:
        if name not in ("dsa_status_string", "dsa_last_cuda_error", "dsa_kernel_launch_count"):
            getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


class Batch:
    """Host handle of a dsa_batch.  Keeps the device q_off / ctx_len alive."""

    def __init__(self, q_off: torch.Tensor, ctx_len: torch.Tensor, max_q: int, max_ctx: int, cache_stride: int,
                 total_q: Optional[int] = None):
        assert q_off.dtype == torch.int32 and ctx_len.dtype == torch.int32
        assert q_off.is_cuda and ctx_len.is_cuda and q_off.is_contiguous() and ctx_len.is_contiguous()
        self.q_off, self.ctx_len = q_off, ctx_len
        B = ctx_len.numel()
        if total_q is None:
            total_q = int(q_off[-1].item())
        self.c = DsaBatch(B, int(total_q), int(max_q), int(max_ctx), int(cache_stride),
                          q_off.data_ptr(), ctx_len.data_ptr())

    @property
    def B(self) -> int:
        return self.c.batch

    @property
    def total_q(self) -> int:
        return self.c.total_q

    @property
    def max_q(self) -> int:
        return self.c.max_q

    @property
    def max_ctx(self) -> int:
        return self.c.max_ctx


def make_batch(q_off, ctx_len, max_q: int, max_ctx: int, cache_stride: int, total_q: Optional[int] = None,
               device="cuda") -> Batch:
    q_off = torch.as_tensor(q_off, dtype=torch.int32).to(device).contiguous()
    ctx_len = torch.as_tensor(ctx_len, dtype=torch.int32).to(device).contiguous()
    return Batch(q_off, ctx_len, max_q, max_ctx, cache_stride, total_q)


def _check(code: int, where: str) -> None:
    if code != 0:
        raise DsaError(code, where)


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("device tensor expected")
    if not t.is_contiguous():
        raise ValueError("contiguous tensor expected")
    return t.data_ptr()


def _bf16(t: torch.Tensor):
    if t.dtype != torch.bfloat16:
        raise TypeError(f"bf16 tensor expected, got {t.dtype}")
    return _p(t)


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def kernel_launch_count() -> int:
    """Kernels launched by libdsa.so in this process so far."""
    return int(load_library().dsa_kernel_launch_count())


def workspace_size(batch: Batch, k: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load_library().dsa_workspace_size(ctypes.byref(batch.c), int(k), ctypes.byref(n)), "dsa_workspace_size")
    return int(n.value)


def workspace(batch: Batch, k: int, device="cuda") -> torch.Tensor:
    """A fresh workspace (uint8 tensor) with a cleared status word."""
    ws = torch.empty(max(workspace_size(batch, k), 256), dtype=torch.uint8, device=device)
    reset_device_status(ws)
    return ws


def reset_device_status(ws: torch.Tensor, stream=None) -> None:
    _check(load_library().dsa_reset_device_status(_p(ws), _stream(stream)), "dsa_reset_device_status")


def read_device_status(ws: torch.Tensor, stream=None) -> int:
    v = ctypes.c_int(0)
    _check(load_library().dsa_read_device_status(_p(ws), _stream(stream), ctypes.byref(v)), "dsa_read_device_status")
    return int(v.value)


def selftest_wait_timeout(ws: torch.Tensor, limit_us: int = 2000, stream=None) -> None:
    """Launch the bounded-wait diagnostic (see dsa_selftest_wait_timeout)."""
    _check(load_library().dsa_selftest_wait_timeout(_p(ws), int(limit_us), _stream(stream)),
           "dsa_selftest_wait_timeout")


def indexer_scores(batch: Batch, q_idx, w, k_idx, scores, ld: Optional[int] = None, ws=None, stream=None):
    assert w.dtype == torch.float32 and scores.dtype == torch.float32
    ld = int(ld if ld is not None else scores.shape[-1])
    _check(load_library().dsa_indexer_scores(ctypes.byref(batch.c), _bf16(q_idx), _p(w), _bf16(k_idx), _p(scores),
                                             ld, _p(ws), ws.numel() if ws is not None else 0, _stream(stream)),
           "dsa_indexer_scores")
    return scores


def topk(batch: Batch, scores, k: int, idx, ld: Optional[int] = None, ws=None, stream=None):
    assert scores.dtype == torch.float32 and idx.dtype == torch.int32
    ld = int(ld if ld is not None else scores.shape[-1])
    _check(load_library().dsa_topk(ctypes.byref(batch.c), _p(scores), ld, int(k), _p(idx), _p(ws),
                                   ws.numel() if ws is not None else 0, _stream(stream)), "dsa_topk")
    return idx


def sparse_mla_fwd(batch: Batch, q, kv, idx, k: int, sm_scale: float, out, lse=None, ws=None, stream=None):
    assert idx.dtype == torch.int32 and (lse is None or lse.dtype == torch.float32)
    _check(load_library().dsa_sparse_mla_fwd(ctypes.byref(batch.c), _bf16(q), _bf16(kv), _p(idx), int(k),
                                             float(sm_scale), _bf16(out), _p(lse), _p(ws),
                                             ws.numel() if ws is not None else 0, _stream(stream)),
           "dsa_sparse_mla_fwd")
    return out


def sparse_mla_fwd_noalloc(batch: Batch, q, kv, idx, k: int, sm_scale: float, out, lse=None, device_status=None,
                           stream=None):
    """dsa_sparse_mla_fwd without a workspace: the split-K partials live in
    the library's static device scratch (for callers that cannot allocate).
    Calls that overlap on the GPU race; the first call on a device should
    come before any stream capture."""
    assert idx.dtype == torch.int32 and (lse is None or lse.dtype == torch.float32)
    assert device_status is None or device_status.dtype == torch.int32
    _check(load_library().dsa_sparse_mla_fwd_noalloc(ctypes.byref(batch.c), _bf16(q), _bf16(kv), _p(idx), int(k),
                                                     float(sm_scale), _bf16(out), _p(lse), _p(device_status),
                                                     _stream(stream)), "dsa_sparse_mla_fwd_noalloc")
    return out


def forward(batch: Batch, q_idx, w, k_idx, q, kv, k: int, sm_scale: float, out, lse=None, idx_out=None,
            scores_out=None, ld: int = 0, ws=None, stream=None):
    if scores_out is not None and not ld:
        ld = scores_out.shape[-1]
    _check(load_library().dsa_forward(ctypes.byref(batch.c), _bf16(q_idx), _p(w), _bf16(k_idx), _bf16(q), _bf16(kv),
                                      int(k), float(sm_scale), _bf16(out), _p(lse), _p(idx_out), _p(scores_out),
                                      int(ld), _p(ws), ws.numel() if ws is not None else 0, _stream(stream)),
           "dsa_forward")
    return out


def mla_absorb_q(q_nope, q_pe, w_kv_b, q_out, ws, stream=None):
    """q_out[t, h] = [W_UK[h]^T q_nope[t, h] | q_pe[t, h]] (see dsa_mla_absorb_q)."""
    total_q = q_nope.shape[0]
    assert q_pe.shape[0] == total_q and q_out.shape[0] == total_q
    _check(load_library().dsa_mla_absorb_q(int(total_q), _bf16(q_nope), _bf16(q_pe), _bf16(w_kv_b), _bf16(q_out),
                                           _p(ws), ws.numel(), _stream(stream)), "dsa_mla_absorb_q")
    return q_out


def mla_workspace(total_q: int, device="cuda") -> torch.Tensor:
    """A workspace for dsa_mla_output / dsa_mla_absorb_q with a cleared status word."""
    n = ctypes.c_size_t(0)
    _check(load_library().dsa_mla_workspace_size(int(total_q), ctypes.byref(n)), "dsa_mla_workspace_size")
    ws = torch.empty(max(int(n.value), 256), dtype=torch.uint8, device=device)
    reset_device_status(ws)
    return ws


def mla_output(o_lat, w_kv_b, w_o, o_mid, y, ws, stream=None):
    """o_mid[t, h] = W_UV[h] o_lat[t, h]; y[t] = w_o o_mid[t] (see dsa_mla_output)."""
    total_q = o_lat.shape[0]
    assert o_mid.shape[0] == total_q and y.shape[0] == total_q
    _check(load_library().dsa_mla_output(int(total_q), _bf16(o_lat), _bf16(w_kv_b), _bf16(w_o), _bf16(o_mid),
                                         _bf16(y), _p(ws), ws.numel(), _stream(stream)), "dsa_mla_output")
    return y


def index_key_workspace(total_q: int, device="cuda") -> torch.Tensor:
    n = ctypes.c_size_t(0)
    _check(load_library().dsa_index_key_workspace_size(int(total_q), ctypes.byref(n)),
           "dsa_index_key_workspace_size")
    ws = torch.empty(max(int(n.value), 256), dtype=torch.uint8, device=device)
    reset_device_status(ws)
    return ws


def index_key_producer(batch: Batch, x, wk, gamma, beta, eps: float, cos, sin, w_proj, k_idx, w_out, ws,
                       stream=None):
    """Index keys of the batch's new tokens appended to k_idx, and their head
    weights in w_out (see dsa_index_key_producer)."""
    for t in (gamma, beta, cos, sin, w_out):
        assert t.dtype == torch.float32
    _check(load_library().dsa_index_key_producer(ctypes.byref(batch.c), _bf16(x), _bf16(wk), _p(gamma), _p(beta),
                                                 float(eps), _p(cos), _p(sin), _bf16(w_proj), _bf16(k_idx),
                                                 _p(w_out), _p(ws), ws.numel(), _stream(stream)),
           "dsa_index_key_producer")
    return k_idx


def quantize_fp8(x, codes, scale, stream=None):
    """E4M3 codes and per-row scales of bf16 rows of 128 (see dsa_quantize_fp8)."""
    assert codes.dtype == torch.uint8 and scale.dtype == torch.float32
    rows = x.numel() // 128
    _check(load_library().dsa_quantize_fp8(int(rows), _bf16(x), _p(codes), _p(scale), _stream(stream)),
           "dsa_quantize_fp8")
    return codes, scale


def indexer_scores_fp8(batch: Batch, q8, qs, w, k8, ks, scores, ld: Optional[int] = None, ws=None, stream=None):
    ld = int(ld if ld is not None else scores.shape[-1])
    _check(load_library().dsa_indexer_scores_fp8(ctypes.byref(batch.c), _p(q8), _p(qs), _p(w), _p(k8), _p(ks),
                                                 _p(scores), ld, _p(ws), ws.numel() if ws is not None else 0,
                                                 _stream(stream)), "dsa_indexer_scores_fp8")
    return scores


def forward_fp8(batch: Batch, q8, qs, w, k8, ks, q, kv, k: int, sm_scale: float, out, lse=None, idx_out=None,
                scores_out=None, ld: int = 0, ws=None, stream=None):
    if scores_out is not None and not ld:
        ld = scores_out.shape[-1]
    _check(load_library().dsa_forward_fp8(ctypes.byref(batch.c), _p(q8), _p(qs), _p(w), _p(k8), _p(ks), _bf16(q),
                                          _bf16(kv), int(k), float(sm_scale), _bf16(out), _p(lse), _p(idx_out),
                                          _p(scores_out), int(ld), _p(ws), ws.numel() if ws is not None else 0,
                                          _stream(stream)), "dsa_forward_fp8")
    return out
