"""fp64 CPU oracle for the DSA hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  The product library never calls it
and shares no code with it: the arithmetic lives in ``oracle.c`` (plain C,
OpenMP over query rows), compiled here with gcc into ``_build/liboracle.so``.

Functions (all take numpy arrays; bf16 tensors as uint16 bit patterns):
  indexer_scores(batch, rows)          -> float64 [len(rows), ld]
  topk(batch, scores_f32, rows, k)     -> int32   [len(rows), k]
  sparse_mla(batch, idx, rows)         -> (float64 [n, 64, 512], float64 [n, 64])
  masked_mla(batch, idx, rows)         -> same, written in the pages' mask form
  mla_absorb_q(q_nope, q_pe, w_kvb)    -> float64 [T, 64, 576]
  mla_output(o_lat, w_kvb, w_o)        -> (float64 [T, 64, 256], float64 [T, 6144])
  mla_expanded(batch, q_nope, q_pe, w_kvb, w_o, idx, rows) -> same pair, the pages' expanded path
  index_key(x, wk, gamma, beta, eps, cos, sin, ww) -> (float64 [T, 128], float64 [T, 32])
  e4m3_decode(codes) / e4m3_encode(values)       -> the OCP FP8 E4M3 format
  quantize_fp8(rows_bf16)              -> (uint8 codes, float64 scale per row)
  indexer_scores_fp8(batch, q8, qs, k8, ks, rows) -> float64 [len(rows), ld]
See ``oracle.c`` for what each computes and the passages it follows.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

H_IDX, D_IDX, H, D_QK, D_V = 32, 128, 64, 576, 512
D_NOPE, D_ROPE, D_VH, KVB_ROWS, HIDDEN = 192, 64, 256, 64 * 448, 6144


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (-O2, OpenMP, no fast-math, no contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            P = ctypes.c_void_p
            i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            lib.oracle_indexer_scores.argtypes = [i32, P, P, i64, P, P, P, i32, P, P, i64]
            lib.oracle_topk.argtypes = [i32, P, P, P, i64, i32, P, i32, P]
            lib.oracle_sparse_mla.argtypes = [i32, P, P, i64, P, P, P, i32, dbl, i32, P, P, P]
            lib.oracle_masked_mla.argtypes = [i32, P, P, i64, P, P, P, i32, dbl, i32, P, P, P]
            lib.oracle_mla_absorb_q.argtypes = [i32, P, P, P, P]
            lib.oracle_mla_output.argtypes = [i32, P, P, P, P, P]
            lib.oracle_mla_expanded.argtypes = [i32, P, P, i64, P, P, P, P, P, P, i32, dbl, i32, P, P, P]
            lib.oracle_index_key.argtypes = [i32, P, P, P, P, dbl, P, P, P, P, P]
            lib.oracle_e4m3_decode_array.argtypes = [i64, P, P]
            lib.oracle_e4m3_encode_array.argtypes = [i64, P, P]
            lib.oracle_quantize_fp8.argtypes = [i64, ctypes.c_int, P, P, P]
            lib.oracle_indexer_scores_fp8.argtypes = [i32, P, P, i64, P, P, P, P, P, i32, P, P, i64]
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _np(x, dtype) -> np.ndarray:
    if hasattr(x, "detach"):          # a torch tensor (CPU copy is taken)
        x = x.detach().cpu()
        if str(x.dtype) == "torch.bfloat16":
            import torch
            x = x.view(torch.int16)
        x = x.numpy()
    a = np.asarray(x)
    if a.dtype != dtype:
        if dtype == np.uint16 and a.dtype == np.int16:
            a = a.view(np.uint16)          # bf16 bit patterns
        else:
            a = a.astype(dtype)
    return np.ascontiguousarray(a)


def _rows(batch, rows: Optional[Sequence[int]]) -> np.ndarray:
    if rows is None:
        rows = range(batch.total_q)
    r = np.ascontiguousarray(np.asarray(list(rows), dtype=np.int32))
    if len(r) and (r.min() < 0 or r.max() >= batch.total_q):
        raise ValueError("row index outside the batch")
    return r


def _check_layout(batch, **arrays) -> None:
    """Refuse a batch description larger than the arrays it points into, so
    that the C code can never read past them."""
    q_off = np.asarray(_np(batch.q_off, np.int32))
    ctx = np.asarray(_np(batch.ctx_len, np.int32))
    if len(q_off) != batch.B + 1 or len(ctx) != batch.B or q_off[0] != 0:
        raise ValueError("q_off / ctx_len do not match B")
    nq = np.diff(q_off)
    if np.any(nq < 0) or np.any(nq > ctx) or np.any(ctx > batch.stride) or int(q_off[-1]) != batch.total_q:
        raise ValueError("inconsistent batch layout")
    need = {"q_idx": batch.total_q * H_IDX * D_IDX, "w": batch.total_q * H_IDX,
            "k_idx": batch.B * batch.stride * D_IDX, "q": batch.total_q * H * D_QK,
            "kv": batch.B * batch.stride * D_QK}
    for name, a in arrays.items():
        if a.size < need[name]:
            raise ValueError(f"{name} holds {a.size} elements, the batch needs {need[name]}")


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def indexer_scores(batch, rows: Optional[Sequence[int]] = None, ld: Optional[int] = None) -> np.ndarray:
    """Lightning-indexer scores; entries s > t of each row are NaN."""
    lib = _load()
    r = _rows(batch, rows)
    ld = int(ld if ld is not None else max(batch.max_ctx, 1))
    out = np.full((len(r), ld), np.nan, dtype=np.float64)
    q_off, ctx = _np(batch.q_off, np.int32), _np(batch.ctx_len, np.int32)
    qi, w, ki = _np(batch.q_idx, np.uint16), _np(batch.w, np.float32), _np(batch.k_idx, np.uint16)
    _check_layout(batch, q_idx=qi, w=w, k_idx=ki)
    lib.oracle_indexer_scores(batch.B, _ptr(q_off), _ptr(ctx), int(batch.stride), _ptr(qi), _ptr(w),
                              _ptr(ki), len(r), _ptr(r), _ptr(out), ld)
    return out


def topk(batch, scores: np.ndarray, rows: Optional[Sequence[int]] = None, k: Optional[int] = None) -> np.ndarray:
    """Causal top-k of fp32 score rows (row j of ``scores`` belongs to rows[j])."""
    lib = _load()
    r = _rows(batch, rows)
    k = int(k if k is not None else batch.k)
    s = np.ascontiguousarray(np.asarray(scores, dtype=np.float32))
    assert s.ndim == 2 and s.shape[0] == len(r)
    out = np.empty((len(r), k), dtype=np.int32)
    q_off, ctx = _np(batch.q_off, np.int32), _np(batch.ctx_len, np.int32)
    _check_layout(batch)
    pos = ctx[np.searchsorted(q_off, r, side="right") - 1] - np.diff(q_off)[np.searchsorted(q_off, r, side="right") - 1] \
        + (r - q_off[np.searchsorted(q_off, r, side="right") - 1])
    if len(r) and int(pos.max()) + 1 > s.shape[1]:
        raise ValueError("score rows shorter than the positions they cover")
    lib.oracle_topk(batch.B, _ptr(q_off), _ptr(ctx), _ptr(s), s.shape[1], len(r), _ptr(r), k, _ptr(out))
    return out


def _mla(fn, batch, idx, rows, sm_scale) -> Tuple[np.ndarray, np.ndarray]:
    r = _rows(batch, rows)
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int32))
    assert idx.ndim == 2 and idx.shape[0] == len(r)
    k = idx.shape[1]
    out = np.empty((len(r), H, D_V), dtype=np.float64)
    lse = np.empty((len(r), H), dtype=np.float64)
    q_off, ctx = _np(batch.q_off, np.int32), _np(batch.ctx_len, np.int32)
    q, kv = _np(batch.q, np.uint16), _np(batch.kv, np.uint16)
    _check_layout(batch, q=q, kv=kv)
    if idx.size and int(idx.max()) >= batch.stride:
        raise ValueError("index outside the cache")
    scale = float(sm_scale if sm_scale is not None else batch.sm_scale)
    fn(batch.B, _ptr(q_off), _ptr(ctx), int(batch.stride), _ptr(q), _ptr(kv), _ptr(idx), k, scale,
       len(r), _ptr(r), _ptr(out), _ptr(lse))
    return out, lse


def sparse_mla(batch, idx, rows=None, sm_scale=None):
    """Absorbed-form attention over the selected latent rows (gather form)."""
    return _mla(_load().oracle_sparse_mla, batch, idx, rows, sm_scale)


def masked_mla(batch, idx, rows=None, sm_scale=None):
    """The same attention in the pages' dense-mask form."""
    return _mla(_load().oracle_masked_mla, batch, idx, rows, sm_scale)


def _weights(w_kvb, w_o=None):
    wk = _np(w_kvb, np.uint16)
    if wk.size != KVB_ROWS * D_V:
        raise ValueError(f"kv_b_proj weight holds {wk.size} elements, expected {KVB_ROWS * D_V}")
    if w_o is None:
        return wk, None
    wo = _np(w_o, np.uint16)
    if wo.size != HIDDEN * H * D_VH:
        raise ValueError(f"o_proj weight holds {wo.size} elements, expected {HIDDEN * H * D_VH}")
    return wk, wo


def mla_absorb_q(q_nope, q_pe, w_kvb) -> np.ndarray:
    """The absorbed 576-wide query: [W_UK[h]^T q_nope[h] | q_pe[h]] per head."""
    qn, qp = _np(q_nope, np.uint16), _np(q_pe, np.uint16)
    T = qn.size // (H * D_NOPE)
    if qn.size != T * H * D_NOPE or qp.size != T * H * D_ROPE:
        raise ValueError("q_nope / q_pe sizes do not match")
    wk, _ = _weights(w_kvb)
    out = np.empty((T, H, D_QK), dtype=np.float64)
    _load().oracle_mla_absorb_q(T, _ptr(qn), _ptr(qp), _ptr(wk), _ptr(out))
    return out


def mla_output(o_lat, w_kvb, w_o) -> Tuple[np.ndarray, np.ndarray]:
    """Head outputs W_UV[h] o_lat[h] and the o_proj output y."""
    ol = np.ascontiguousarray(np.asarray(o_lat, dtype=np.float64))
    T = ol.size // (H * D_V)
    if ol.size != T * H * D_V:
        raise ValueError("o_lat size is not a multiple of 64 x 512")
    wk, wo = _weights(w_kvb, w_o)
    o_mid = np.empty((T, H, D_VH), dtype=np.float64)
    y = np.empty((T, HIDDEN), dtype=np.float64)
    _load().oracle_mla_output(T, _ptr(ol), _ptr(wk), _ptr(wo), _ptr(o_mid), _ptr(y))
    return o_mid, y


def mla_expanded(batch, q_nope, q_pe, w_kvb, w_o, idx, rows=None, sm_scale=None) -> Tuple[np.ndarray, np.ndarray]:
    """The pages' expanded path (kv_b_proj applied to every attended cached
    row, masked attention, o_proj) for the given rows and selections."""
    r = _rows(batch, rows)
    idx = np.ascontiguousarray(np.asarray(idx, dtype=np.int32))
    assert idx.ndim == 2 and idx.shape[0] == len(r)
    qn, qp = _np(q_nope, np.uint16), _np(q_pe, np.uint16)
    if qn.size < batch.total_q * H * D_NOPE or qp.size < batch.total_q * H * D_ROPE:
        raise ValueError("q_nope / q_pe hold fewer rows than the batch")
    kv = _np(batch.kv, np.uint16)
    _check_layout(batch, kv=kv)
    wk, wo = _weights(w_kvb, w_o)
    q_off, ctx = _np(batch.q_off, np.int32), _np(batch.ctx_len, np.int32)
    scale = float(sm_scale if sm_scale is not None else batch.sm_scale)
    o_mid = np.empty((len(r), H, D_VH), dtype=np.float64)
    y = np.empty((len(r), HIDDEN), dtype=np.float64)
    _load().oracle_mla_expanded(batch.B, _ptr(q_off), _ptr(ctx), int(batch.stride), _ptr(qn), _ptr(qp), _ptr(kv),
                                _ptr(wk), _ptr(wo), _ptr(idx), idx.shape[1], scale, len(r), _ptr(r), _ptr(o_mid),
                                _ptr(y))
    return o_mid, y


def index_key(x, wk, gamma, beta, eps, cos, sin, ww) -> Tuple[np.ndarray, np.ndarray]:
    """Index keys of new tokens (wk, LayerNorm(128), RoPE on the first 64
    dims with the given cos / sin rows) and their head weights
    (weights_proj * 32^-1/2)."""
    xb = _np(x, np.uint16)
    T = xb.size // HIDDEN
    if xb.size != T * HIDDEN:
        raise ValueError("x is not [T, 6144]")
    wkb, wwb = _np(wk, np.uint16), _np(ww, np.uint16)
    if wkb.size != D_IDX * HIDDEN or wwb.size != H_IDX * HIDDEN:
        raise ValueError("wk must be [128, 6144] and weights_proj [32, 6144]")
    g = np.ascontiguousarray(np.asarray(gamma, dtype=np.float64))
    b = np.ascontiguousarray(np.asarray(beta, dtype=np.float64))
    c = np.ascontiguousarray(np.asarray(cos, dtype=np.float64))
    s = np.ascontiguousarray(np.asarray(sin, dtype=np.float64))
    if g.size != D_IDX or b.size != D_IDX or c.size != T * 64 or s.size != T * 64:
        raise ValueError("gamma / beta must hold 128 values, cos / sin [T, 64]")
    k = np.empty((T, D_IDX), dtype=np.float64)
    w = np.empty((T, H_IDX), dtype=np.float64)
    _load().oracle_index_key(T, _ptr(xb), _ptr(wkb), _ptr(g), _ptr(b), float(eps), _ptr(c), _ptr(s), _ptr(wwb),
                             _ptr(k), _ptr(w))
    return k, w


def e4m3_decode(codes) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_e4m3_decode_array(c.size, _ptr(c), _ptr(out))
    return out


def e4m3_encode(values) -> np.ndarray:
    x = np.ascontiguousarray(np.asarray(values, dtype=np.float64))
    out = np.empty(x.shape, dtype=np.uint8)
    _load().oracle_e4m3_encode_array(x.size, _ptr(x), _ptr(out))
    return out


def quantize_fp8(rows_bf16, n: int) -> Tuple[np.ndarray, np.ndarray]:
    """Rows of n bf16 values -> (E4M3 codes [rows, n], scale [rows]) with
    scale = amax / 448 (1 for an all-zero row)."""
    v = _np(rows_bf16, np.uint16)
    rows = v.size // n
    if v.size != rows * n:
        raise ValueError("size is not a multiple of n")
    codes = np.empty((rows, n), dtype=np.uint8)
    scale = np.empty(rows, dtype=np.float64)
    _load().oracle_quantize_fp8(rows, n, _ptr(v), _ptr(codes), _ptr(scale))
    return codes, scale


def indexer_scores_fp8(batch, q8, qs, k8, ks, rows: Optional[Sequence[int]] = None,
                       ld: Optional[int] = None) -> np.ndarray:
    """Lightning-indexer scores on E4M3 queries / keys with per-(token, head)
    and per-key scales; entries s > t are NaN."""
    r = _rows(batch, rows)
    ld = int(ld if ld is not None else max(batch.max_ctx, 1))
    q8a, k8a = np.ascontiguousarray(q8, dtype=np.uint8), np.ascontiguousarray(k8, dtype=np.uint8)
    qsa, ksa = np.ascontiguousarray(qs, dtype=np.float64), np.ascontiguousarray(ks, dtype=np.float64)
    w = _np(batch.w, np.float32)
    if q8a.size < batch.total_q * H_IDX * D_IDX or qsa.size < batch.total_q * H_IDX or \
            k8a.size < batch.B * batch.stride * D_IDX or ksa.size < batch.B * batch.stride:
        raise ValueError("FP8 arrays smaller than the batch")
    _check_layout(batch, w=w)
    out = np.full((len(r), ld), np.nan, dtype=np.float64)
    q_off, ctx = _np(batch.q_off, np.int32), _np(batch.ctx_len, np.int32)
    _load().oracle_indexer_scores_fp8(batch.B, _ptr(q_off), _ptr(ctx), int(batch.stride), _ptr(q8a), _ptr(qsa),
                                      _ptr(w), _ptr(k8a), _ptr(ksa), len(r), _ptr(r), _ptr(out), ld)
    return out
