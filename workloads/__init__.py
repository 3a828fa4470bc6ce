"""Seeded synthetic inputs for the DSA (lightning indexer -> causal top-k ->
sparse MLA) hot path.

This module is shared by the oracle side and the CUDA side of the tests and
the benchmark.  It holds no arithmetic of the method itself: it only draws
random tensors with the shapes, scales and structure of the GLM-5 DSA layer
("GLM-5.1 架构深度拆解", CH3 "DSA" and CH4 "MLA"; the GLM-5 explainer page,
indexer and cache tables) and rounds them to the bf16 storage format.

Two back ends draw the same *recipe*, not the same numbers:
  * ``numpy`` (CPU, PCG64) for the parity sizes the oracle finishes in seconds;
  * ``torch`` (any device) for the full-size workloads, drawn on the GPU so
    that a 2.4 GB latent cache does not take a minute of host time.

Layouts (row-major, packed over query rows of all sequences):
  q_idx  bf16 [total_q, 32, 128]   post-RoPE indexer queries
  w      fp32 [total_q, 32]        indexer head weights (the 32**-0.5 factor
                                   of the pages is already folded in)
  k_idx  bf16 [B * stride, 128]    one index key per cached token
  q      bf16 [total_q, 64, 576]   absorbed MLA queries (512 latent || 64 rope)
  kv     bf16 [B * stride, 576]    latent cache rows (512 latent || 64 rope)
  q_off  int32 [B + 1]             prefix offsets of each sequence's queries
  ctx_len int32 [B]                cached tokens per sequence, this call's
                                   queries included (the last query of
                                   sequence b sits at position ctx_len[b]-1)
"""

from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence

import numpy as np

H_IDX = 32      # index_n_heads
D_IDX = 128     # index_head_dim
H = 64          # attention heads
D_QK = 576      # kv_lora_rank 512 + qk_rope_head_dim 64
D_V = 512       # kv_lora_rank (V is the latent part of the cached row)
TOPK = 2048     # index_topk
SM_SCALE = 1.0 / 16.0   # (192 nope + 64 rope) ** -0.5
MAX_POS = 202752        # max_position_embeddings
D_NOPE = 192    # qk_nope_head_dim
D_ROPE = 64     # qk_rope_head_dim
D_VH = 256      # v_head_dim
HIDDEN = 6144   # hidden size (o_proj output)


def bf16_bits_from_f32(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even) and return
    the 16-bit patterns as uint16.  Storage-format conversion of the inputs."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Batch:
    """One call's worth of inputs (numpy arrays or torch tensors)."""
    B: int
    stride: int                 # cache rows reserved per sequence
    q_off: object               # int32 [B+1]
    ctx_len: object             # int32 [B]
    q_idx: object
    w: object
    k_idx: object
    q: object
    kv: object
    k: int
    sm_scale: float
    name: str = ""

    @property
    def total_q(self) -> int:
        return int(self.q_off[-1])

    @property
    def max_q(self) -> int:
        qo = [int(v) for v in self.q_off]
        return max([qo[i + 1] - qo[i] for i in range(self.B)] + [0])

    @property
    def max_ctx(self) -> int:
        return max([int(v) for v in self.ctx_len] + [0])

    def positions(self) -> List[tuple]:
        """(sequence, position t) of every packed query row, in row order."""
        out = []
        qo = [int(v) for v in self.q_off]
        cl = [int(v) for v in self.ctx_len]
        for b in range(self.B):
            nq = qo[b + 1] - qo[b]
            for i in range(nq):
                out.append((b, cl[b] - nq + i))
        return out


# --------------------------------------------------------------------------
# index-key structure recipes
# --------------------------------------------------------------------------

def _np_index_keys(rng: np.random.Generator, n: int, kind: str) -> np.ndarray:
    if kind == "iid":
        return rng.standard_normal((n, D_IDX), dtype=np.float32) / math.sqrt(D_IDX)
    if kind == "lowrank16":
        # k[s] = (g_s + A z_s) / 16 with g ~ N(0, I_128), z ~ N(0, I_16) and a
        # fixed A ~ N(0,1)/4 of shape [128, 16]: per-element variance 1/128,
        # plus a shared rank-16 component so that scores are not near-tied.
        A = rng.standard_normal((D_IDX, 16), dtype=np.float32) / 4.0
        g = rng.standard_normal((n, D_IDX), dtype=np.float32)
        z = rng.standard_normal((n, 16), dtype=np.float32)
        return (g + z @ A.T) / 16.0
    if kind == "zipf":
        # k[s] = base_s * sqrt(b_s), base ~ N(0,1)/sqrt(128), b_s a discrete
        # Pareto (Zipf-like, exponent 1.5) magnitude boost, capped at 64.
        base = rng.standard_normal((n, D_IDX), dtype=np.float32) / math.sqrt(D_IDX)
        u = 1.0 - rng.random(n)              # (0, 1]
        b = np.minimum(np.floor(u ** (-1.0 / 0.5)), 64.0).astype(np.float32)
        return base * np.sqrt(b)[:, None]
    raise ValueError(kind)


def make_batch_np(ctx_len: Sequence[int], n_new: Sequence[int], k: int, seed: int,
                  key_kind: str = "iid", stride: Optional[int] = None,
                  sm_scale: float = SM_SCALE, name: str = "") -> Batch:
    """Numpy (CPU) inputs: sequence b has ctx_len[b] cached tokens of which
    the last n_new[b] are this call's queries."""
    B = len(ctx_len)
    assert len(n_new) == B
    for c, n in zip(ctx_len, n_new):
        assert 0 <= n <= c
    stride = int(stride if stride is not None else max(max(ctx_len), 1))
    rng = np.random.Generator(np.random.PCG64(seed))
    q_off = np.zeros(B + 1, dtype=np.int32)
    q_off[1:] = np.cumsum(np.asarray(n_new, dtype=np.int64)).astype(np.int32)
    total_q = int(q_off[-1])
    q_idx = rng.standard_normal((total_q, H_IDX, D_IDX), dtype=np.float32) / math.sqrt(D_IDX)
    w = (rng.standard_normal((total_q, H_IDX), dtype=np.float32) / math.sqrt(H_IDX)).astype(np.float32)
    k_idx = np.zeros((B * stride, D_IDX), dtype=np.float32)
    kv = np.zeros((B * stride, D_QK), dtype=np.float32)
    for b in range(B):
        n = ctx_len[b]
        k_idx[b * stride: b * stride + n] = _np_index_keys(rng, n, key_kind)
        kv[b * stride: b * stride + n] = rng.standard_normal((n, D_QK), dtype=np.float32)
    q = rng.standard_normal((total_q, H, D_QK), dtype=np.float32)
    return Batch(B=B, stride=stride, q_off=q_off, ctx_len=np.asarray(ctx_len, dtype=np.int32),
                 q_idx=bf16_bits_from_f32(q_idx), w=w, k_idx=bf16_bits_from_f32(k_idx),
                 q=bf16_bits_from_f32(q), kv=bf16_bits_from_f32(kv), k=k, sm_scale=sm_scale,
                 name=name)


# --------------------------------------------------------------------------
# torch back end (full-size workloads, drawn on the device)
# --------------------------------------------------------------------------

def make_batch_torch(ctx_len: Sequence[int], n_new: Sequence[int], k: int, seed: int,
                     key_kind: str = "iid", stride: Optional[int] = None,
                     sm_scale: float = SM_SCALE, device: str = "cuda", name: str = "") -> Batch:
    import torch
    B = len(ctx_len)
    stride = int(stride if stride is not None else max(max(ctx_len), 1))
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    q_off = [0]
    for n in n_new:
        q_off.append(q_off[-1] + int(n))
    total_q = q_off[-1]
    bf = torch.bfloat16

    def randn(*shape, scale=1.0):
        return (torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * scale)

    q_idx = randn(total_q, H_IDX, D_IDX, scale=1 / math.sqrt(D_IDX)).to(bf)
    w = randn(total_q, H_IDX, scale=1 / math.sqrt(H_IDX))
    q = randn(total_q, H, D_QK).to(bf)
    kv = torch.zeros(B * stride, D_QK, dtype=bf, device=device)
    k_idx = torch.zeros(B * stride, D_IDX, dtype=bf, device=device)
    A = randn(D_IDX, 16, scale=0.25) if key_kind == "lowrank16" else None
    for b in range(B):
        n = int(ctx_len[b])
        base = b * stride
        kv[base: base + n] = randn(n, D_QK).to(bf)
        if key_kind == "iid":
            kk = randn(n, D_IDX, scale=1 / math.sqrt(D_IDX))
        elif key_kind == "lowrank16":
            kk = (randn(n, D_IDX) + randn(n, 16) @ A.T) / 16.0
        elif key_kind == "zipf":
            u = 1.0 - torch.rand(n, generator=g, device=device, dtype=torch.float64)
            boost = torch.clamp(torch.floor(u ** (-2.0)), max=64.0).to(torch.float32)
            kk = randn(n, D_IDX, scale=1 / math.sqrt(D_IDX)) * boost.sqrt()[:, None]
        else:
            raise ValueError(key_kind)
        k_idx[base: base + n] = kk.to(bf)
    return Batch(B=B, stride=stride,
                 q_off=torch.tensor(q_off, dtype=torch.int32, device=device),
                 ctx_len=torch.tensor(list(ctx_len), dtype=torch.int32, device=device),
                 q_idx=q_idx, w=w, k_idx=k_idx, q=q, kv=kv, k=k, sm_scale=sm_scale, name=name)


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------

@dataclasses.dataclass
class Workload:
    name: str
    kind: str                   # "prefill" | "decode" | "chunked_prefill"
    B: int
    ctx: int                    # final context length of each sequence
    n_new: int                  # queries per call per sequence
    k: int
    key_kind: str
    seed: int
    steps: int = 1              # decode steps (long decode) or chunks (chunked prefill)

    @property
    def mla(self) -> bool:
        """The MLA projections around the path are part of the step."""
        return self.kind.startswith("mla_")

    @property
    def fp8(self) -> bool:
        """The index keys are cached as E4M3 codes with per-key scales."""
        return self.kind.startswith("fp8_")

    @property
    def base(self) -> str:
        """The kind of the DSA part of the step."""
        return self.kind[4:] if (self.mla or self.fp8) else self.kind

    def describe(self) -> Dict[str, object]:
        return dataclasses.asdict(self)


WORKLOADS: Dict[str, Workload] = {
    # T=512 tiny prefill, k=128 (parity sized)
    "tiny_prefill_T512_k128": Workload("tiny_prefill_T512_k128", "prefill", 1, 512, 512, 128, "iid", 20260),
    # decode: 64 sequences x 32768 context, one new token each, top-2048
    "decode_B64_ctx32768": Workload("decode_B64_ctx32768", "decode", 64, 32768, 1, TOPK, "iid", 20261),
    # prefill: one sequence of 16384 tokens, top-2048, rank-16 index keys
    "prefill_T16384": Workload("prefill_T16384", "prefill", 1, 16384, 16384, TOPK, "lowrank16", 20262),
    # chunked prefill: 65536 tokens in 8 chunks of 8192 queries
    "chunked_prefill_T65536_c8192": Workload("chunked_prefill_T65536_c8192", "chunked_prefill", 1, 65536, 8192,
                                             TOPK, "lowrank16", 20263, steps=8),
    # IndexShare window on the decode shape: one full layer (indexer, top-k,
    # attention) and three shared layers reusing its indices (steps = layers)
    "indexshare_decode_B64_ctx32768_w4": Workload("indexshare_decode_B64_ctx32768_w4", "indexshare", 64, 32768, 1,
                                                  TOPK, "iid", 20265, steps=4),
    # the decode and prefill workloads with the MLA projections around the
    # path: absorb the query (W_UK), then W_UV and o_proj on the output
    "mla_decode_B64_ctx32768": Workload("mla_decode_B64_ctx32768", "mla_decode", 64, 32768, 1, TOPK, "iid", 20266),
    "mla_prefill_T16384": Workload("mla_prefill_T16384", "mla_prefill", 1, 16384, 16384, TOPK, "lowrank16", 20267),
    # the decode workload with E4M3 index keys (per-key scales) and E4M3
    # indexer queries (per (token, head) scales), quantized each step
    "decode_B64_ctx32768_fp8keys": Workload("decode_B64_ctx32768_fp8keys", "fp8_decode", 64, 32768, 1, TOPK, "iid",
                                            20268),
    # long decode: 8 sequences at 202752 context, 4 decode steps
    "long_decode_B8_ctx202752": Workload("long_decode_B8_ctx202752", "decode", 8, MAX_POS, 1, TOPK, "zipf",
                                         20264, steps=4),
}



# --------------------------------------------------------------------------
# MLA around the path: un-absorbed queries and random-init projection weights
# --------------------------------------------------------------------------

@dataclasses.dataclass
class MlaWeights:
    """kv_b_proj weight [64 * 448, 512] (per head: 192 rows of W_UK, then 256
    rows of W_UV) and o_proj weight [6144, 64 * 256], bf16 bit patterns
    (numpy) or bf16 tensors (torch); random init with variance 1/fan_in."""
    w_kvb: object
    w_o: object


def make_mla_weights_np(seed: int) -> MlaWeights:
    rng = np.random.default_rng(seed)
    w_kvb = rng.standard_normal((H * (D_NOPE + D_VH), D_V), dtype=np.float32) / math.sqrt(D_V)
    w_o = rng.standard_normal((HIDDEN, H * D_VH), dtype=np.float32) / math.sqrt(H * D_VH)
    return MlaWeights(bf16_bits_from_f32(w_kvb), bf16_bits_from_f32(w_o))


def make_mla_weights_torch(seed: int, device: str = "cuda") -> MlaWeights:
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    w_kvb = torch.randn(H * (D_NOPE + D_VH), D_V, generator=g, device=device) / math.sqrt(D_V)
    w_o = torch.randn(HIDDEN, H * D_VH, generator=g, device=device) / math.sqrt(H * D_VH)
    return MlaWeights(w_kvb.to(torch.bfloat16), w_o.to(torch.bfloat16))


def make_mla_queries_np(total_q: int, seed: int):
    """q_nope [total_q, 64, 192] and q_pe [total_q, 64, 64] (post-RoPE), bf16 bits."""
    rng = np.random.default_rng(seed)
    q_nope = rng.standard_normal((total_q, H, D_NOPE), dtype=np.float32)
    q_pe = rng.standard_normal((total_q, H, D_ROPE), dtype=np.float32)
    return bf16_bits_from_f32(q_nope), bf16_bits_from_f32(q_pe)


def make_mla_queries_torch(total_q: int, seed: int, device: str = "cuda"):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    q_nope = torch.randn(total_q, H, D_NOPE, generator=g, device=device).to(torch.bfloat16)
    q_pe = torch.randn(total_q, H, D_ROPE, generator=g, device=device).to(torch.bfloat16)
    return q_nope, q_pe


# --------------------------------------------------------------------------
# the index-key producer: hidden states, wk / k_norm / weights_proj, rotary rows
# --------------------------------------------------------------------------

ROPE_THETA = 10000.0    # synthetic rotary base (the tables are inputs of the producer)


@dataclasses.dataclass
class IndexKeyParams:
    """wk [128, 6144] and weights_proj [32, 6144] (bf16 bits / tensors),
    k_norm gamma / beta [128] (fp32), eps."""
    wk: object
    ww: object
    gamma: object
    beta: object
    eps: float = 1e-5


def rotary_rows(positions, dim: int = 64, theta: float = ROPE_THETA):
    """cos / sin rows [n, dim] of the rotate-half rotary table at the given
    positions (frequencies repeated over the two halves), fp32 numpy."""
    pos = np.asarray(positions, dtype=np.float64)[:, None]
    inv = theta ** (-np.arange(0, dim, 2, dtype=np.float64) / dim)
    ang = pos * np.concatenate([inv, inv])[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def make_index_key_params_np(seed: int) -> IndexKeyParams:
    rng = np.random.default_rng(seed)
    wk = rng.standard_normal((D_IDX, HIDDEN), dtype=np.float32) / math.sqrt(HIDDEN)
    ww = rng.standard_normal((H_IDX, HIDDEN), dtype=np.float32) / math.sqrt(HIDDEN)
    gamma = (1.0 + 0.1 * rng.standard_normal(D_IDX)).astype(np.float32)
    beta = (0.1 * rng.standard_normal(D_IDX)).astype(np.float32)
    return IndexKeyParams(bf16_bits_from_f32(wk), bf16_bits_from_f32(ww), gamma, beta)


def make_hidden_np(total_q: int, seed: int) -> np.ndarray:
    """Hidden states [total_q, 6144] ~ N(0, 1), bf16 bits."""
    rng = np.random.default_rng(seed)
    return bf16_bits_from_f32(rng.standard_normal((total_q, HIDDEN), dtype=np.float32))
