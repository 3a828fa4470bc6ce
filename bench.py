#!/usr/bin/env python
"""Benchmark of the DSA hot path (lightning indexer -> causal top-k ->
sparse MLA attention) through libdsa.so on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl dsa|reference]

One step is one pass of the whole path over one batch of synthetic input:
  decode_B64_ctx32768 (default): one decode step of 64 sequences at context
      32768 (one new query each), top-2048 -> metric "decode steps/s";
  long_decode_B8_ctx202752: one decode step of 8 sequences near 202752;
  prefill_T16384, tiny_prefill_T512_k128: a whole prefill -> tokens/s;
  chunked_prefill_T65536_c8192: 8 chunks of 8192 queries -> tokens/s.
Inputs are drawn on the device (seeded) and stay resident in HBM; the
decode working set (2.96 GB of caches) is far larger than L2, so no flush
is needed between steps.  Rank 0 prints ONE JSON line.

--impl reference times the fp64 CPU oracle (the method written out plainly,
tests/ pins it) on the host cores on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

DEFAULT_WORKLOAD = "decode_B64_ctx32768"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
NOMINAL_PEAKS = {"hbm_gbs": 7900.0, "bf16_tflops": 2250.0}     # GB300 data-sheet figures, for context
# workloads timed beside the default decode line (details.other_workloads)
SIDE_WORKLOADS = ("prefill_T16384", "long_decode_B8_ctx202752")

# algorithmic work per unit
IDX_FLOP_PER_PAIR = 2 * 32 * 128            # 8192
IDX_BYTES_PER_KEY = 128 * 2                 # one bf16 index key
IDX_BYTES_PER_QUERY = 32 * 128 * 2 + 32 * 4  # q_idx + w
IDX8_BYTES_PER_KEY = 128 + 4                # one E4M3 index key and its scale
IDX8_BYTES_PER_QUERY = 32 * 128 + 32 * 4 + 32 * 4   # E4M3 q_idx + scales + w
ATT_FLOP_PER_SEL = 2 * 64 * 576 + 2 * 64 * 512   # 139264
ATT_BYTES_PER_SEL = 576 * 2                 # one gathered latent row
ATT_BYTES_PER_QUERY = 64 * 576 * 2 + 64 * 512 * 2  # q in + out
# MLA projections around the path, per token (and the weights, once per call)
ABS_FLOP_PER_TOKEN = 2 * 64 * 192 * 512
ABS_BYTES_PER_TOKEN = 64 * 192 * 2 + 64 * 64 * 2 + 64 * 576 * 2
ABS_WEIGHT_BYTES = 64 * 192 * 512 * 2
OUT_FLOP_PER_TOKEN = 2 * 64 * 512 * 256 + 2 * 64 * 256 * 6144
OUT_BYTES_PER_TOKEN = 64 * 512 * 2 + 6144 * 2
OUT_WEIGHT_BYTES = (64 * 256 * 512 + 6144 * 64 * 256) * 2
IK_FLOP_PER_TOKEN = 2 * 6144 * (128 + 32)                  # wk and weights_proj
IK_BYTES_PER_TOKEN = 6144 * 2 + 128 * 2 + 32 * 4 + 64 * 8   # x in, key and w out, cos / sin rows
IK_WEIGHT_BYTES = (128 + 32) * 6144 * 2


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=None)
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS))
    p.add_argument("--impl", default="dsa", choices=["dsa", "reference"])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--kernel-reps", type=int, default=20)
    p.add_argument("--no-side", action="store_true", help="skip the prefill / long-decode sets of the default line")
    p.add_argument("--clock-hold-s", type=float, default=0.5,
                   help="seconds of untimed repeats after the timed steps, for clock samples (0: none)")
    return p.parse_args()


def default_steps(wl: W.Workload):
    return (300, 10) if wl.base in ("decode", "indexshare") else (20, 3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained")}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------- workloads --

def metric_for(wl: W.Workload):
    if wl.mla:
        what = "index-key producer, absorbed query, indexer, top-k, attention, W_UV, o_proj"
        if wl.base == "decode":
            return f"MLA layer decode steps/s ({wl.B} seqs x {wl.ctx} ctx, top-{wl.k}; {what})", "steps/s"
        return f"MLA layer prefill tokens/s (T={wl.ctx}, top-{wl.k}; {what})", "tokens/s"
    if wl.fp8:
        return (f"decode steps/s with E4M3 index keys ({wl.B} seqs x {wl.ctx} ctx, top-{wl.k}; % of HBM roofline)",
                "steps/s")
    if wl.base == "indexshare":
        return (f"IndexShare decode window steps/s ({wl.B} seqs x {wl.ctx} ctx, 1 full + {wl.steps - 1} shared "
                f"layers, top-{wl.k})", "steps/s")
    if wl.base == "decode":
        return f"decode steps/s ({wl.B} seqs x {wl.ctx} ctx, top-{wl.k}; % of HBM roofline)", "steps/s"
    if wl.base == "prefill":
        return f"prefill tokens/s (T={wl.ctx}, top-{wl.k}; % of bf16 tensor roofline)", "tokens/s"
    return f"chunked prefill tokens/s (T={wl.ctx} in {wl.ctx // wl.n_new} chunks, top-{wl.k})", "tokens/s"


def base_config(wl: W.Workload, world: int):
    return {"workload": wl.name, "batch": wl.B, "ctx": wl.ctx, "queries_per_seq": wl.n_new, "topk": wl.k,
            "l2": "no flush: inputs larger than L2" if wl.base in ("decode", "indexshare") else
            "no flush: the one sequence's keys and latent cache are L2-resident by design",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


class Case:
    """The device inputs of one workload and its step function."""

    def __init__(self, wl: W.Workload, seed: int, device):
        import torch

        import sparse_attention_gb300 as dsa
        self.wl, self.dev = wl, device
        self.calls = []          # (batch, slices) per dsa_forward call of one step
        if wl.base == "decode":
            self.bt = W.make_batch_torch([wl.ctx] * wl.B, [1] * wl.B, wl.k, seed, key_kind=wl.key_kind,
                                         device=device, name=wl.name)
            bt = self.bt
            # decode steps cycle over the last `steps` positions of the cache
            self.ctx_variants = [torch.full((wl.B,), wl.ctx - wl.steps + 1 + j, dtype=torch.int32, device=device)
                                 for j in range(wl.steps)]
            self.batches = [dsa.Batch(bt.q_off, c, 1, wl.ctx, bt.stride, total_q=wl.B) for c in self.ctx_variants]
            self.positions = [[wl.ctx - wl.steps + j] * wl.B for j in range(wl.steps)]
            self.units_per_step = 1            # one decode step of the whole batch
        elif wl.base == "indexshare":
            # layer 0 is full; layers 1.. reuse its indices with their own q and latent cache
            self.bt = W.make_batch_torch([wl.ctx] * wl.B, [1] * wl.B, wl.k, seed, key_kind=wl.key_kind,
                                         device=device, name=wl.name)
            bt = self.bt
            self.shared = []
            for layer in range(1, wl.steps):
                lb = W.make_batch_torch([wl.ctx] * wl.B, [1] * wl.B, wl.k, seed + 17 * layer, key_kind="iid",
                                        device=device)
                self.shared.append((lb.q, lb.kv))
                del lb
            self.batches = [dsa.Batch(bt.q_off, bt.ctx_len, 1, wl.ctx, bt.stride, total_q=wl.B)]
            self.positions = [[wl.ctx - 1] * wl.B]
            self.units_per_step = 1            # one decode step of the whole window
            self.share_idx = torch.empty((wl.B, wl.k), dtype=torch.int32, device=device)
        elif wl.base == "prefill":
            self.bt = W.make_batch_torch([wl.ctx], [wl.n_new], wl.k, seed, key_kind=wl.key_kind, device=device,
                                         name=wl.name)
            bt = self.bt
            self.batches = [dsa.Batch(bt.q_off, bt.ctx_len, wl.n_new, wl.ctx, bt.stride, total_q=wl.n_new)]
            self.positions = [list(range(wl.ctx - wl.n_new, wl.ctx))]
            self.units_per_step = wl.n_new
        else:  # chunked prefill
            T, C = wl.ctx, wl.n_new
            self.bt = W.make_batch_torch([T], [T], wl.k, seed, key_kind=wl.key_kind, device=device, name=wl.name)
            bt = self.bt
            self.batches, self.positions = [], []
            for c in range(T // C):
                qo = torch.tensor([0, C], dtype=torch.int32, device=device)
                cl = torch.tensor([C * (c + 1)], dtype=torch.int32, device=device)
                self.batches.append(dsa.Batch(qo, cl, C, C * (c + 1), bt.stride, total_q=C))
                self.positions.append(list(range(C * c, C * (c + 1))))
            self.units_per_step = T
        self.metric, self.unit = metric_for(wl)
        self.max_rows = max(b.total_q for b in self.batches)
        if wl.mla:
            # un-absorbed queries and random-init kv_b_proj / o_proj weights
            T = self.max_rows
            self.mw = W.make_mla_weights_torch(seed + 1, device=device)
            self.q_nope, self.q_pe = W.make_mla_queries_torch(T, seed + 2, device=device)
            self.o_mid = torch.empty((T, 64 * 256), dtype=torch.bfloat16, device=device)
            self.y = torch.empty((T, 6144), dtype=torch.bfloat16, device=device)
            self.mla_ws = dsa.mla_workspace(T, device=device)
            # the index-key producer: hidden states, wk / k_norm / weights_proj, rotary rows
            ip = W.make_index_key_params_np(seed + 3)
            g = torch.Generator(device=device)
            g.manual_seed(seed + 4)
            self.x = torch.randn(T, W.HIDDEN, generator=g, device=device).to(torch.bfloat16)
            self.ik = {"wk": torch.from_numpy(ip.wk.view(np.int16)).to(device).view(torch.bfloat16),
                       "ww": torch.from_numpy(ip.ww.view(np.int16)).to(device).view(torch.bfloat16),
                       "gamma": torch.from_numpy(ip.gamma).to(device), "beta": torch.from_numpy(ip.beta).to(device),
                       "eps": ip.eps}
            self.rope = []
            for pos in self.positions:
                c, sn = W.rotary_rows(pos)
                self.rope.append((torch.from_numpy(c).to(device), torch.from_numpy(sn).to(device)))
            self.ik_ws = [dsa.index_key_workspace(b.total_q, device=device) for b in self.batches]
        if wl.fp8:
            # the cache holds E4M3 keys (quantized once, as a cache append
            # would); the queries are quantized in every step
            nk = wl.B * self.bt.stride
            self.k8 = torch.empty((nk, 128), dtype=torch.uint8, device=device)
            self.ks = torch.empty(nk, dtype=torch.float32, device=device)
            dsa.quantize_fp8(self.bt.k_idx, self.k8, self.ks)
            self.q8 = torch.empty((self.max_rows * 32, 128), dtype=torch.uint8, device=device)
            self.qs = torch.empty(self.max_rows * 32, dtype=torch.float32, device=device)
        self.out = torch.empty((self.max_rows, 64, 512), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((self.max_rows, 64), dtype=torch.float32, device=device)
        # one workspace for every call, as a decode or chunked-prefill loop
        # on one stream reuses it (a call's indexer launch waits for the
        # previous call's kernels); its status word then covers every call.
        # (A workspace per context length made the 8 x 202,752 decode step
        # ~2 us slower: four sets of score rows cycle through L2.)
        sizes = [dsa.workspace_size(b, wl.k) for b in self.batches]
        ws = dsa.workspace(self.batches[sizes.index(max(sizes))], wl.k, device=device)
        self.ws = [ws] * len(self.batches)
        self.dsa = dsa

    def _slices(self, j):
        """query-side tensors of call j (chunked prefill slices the queries)."""
        bt, wl = self.bt, self.wl
        if self.wl.base == "chunked_prefill":
            C = wl.n_new
            s = slice(C * j, C * (j + 1))
            return bt.q_idx[s], bt.w[s], bt.q[s]
        return bt.q_idx, bt.w, bt.q

    def step(self, i=0):
        """One step of the workload: every dsa_forward call it needs."""
        wl = self.wl
        if wl.base == "indexshare":
            b = self.batches[0]
            self.dsa.forward(b, self.bt.q_idx, self.bt.w, self.bt.k_idx, self.bt.q, self.bt.kv, wl.k,
                             self.bt.sm_scale, self.out, self.lse, idx_out=self.share_idx, ws=self.ws[0])
            for q, kv in self.shared:
                self.dsa.sparse_mla_fwd(b, q, kv, self.share_idx, wl.k, self.bt.sm_scale, self.out, self.lse,
                                        ws=self.ws[0])
            return
        if wl.base == "decode":
            j = i % len(self.batches)
            calls = [j]
        else:
            calls = range(len(self.batches))
        if wl.mla:
            for j in calls:
                self._index_key(j)
            self.dsa.mla_absorb_q(self.q_nope, self.q_pe, self.mw.w_kvb, self.bt.q, self.mla_ws)
        for j in calls:
            q_idx, w, q = self._slices(j)
            b = self.batches[j]
            if wl.fp8:
                self.dsa.quantize_fp8(q_idx, self.q8, self.qs)
                self.dsa.forward_fp8(b, self.q8, self.qs, w, self.k8, self.ks, q, self.bt.kv, wl.k,
                                     self.bt.sm_scale, self.out[:b.total_q], self.lse[:b.total_q], ws=self.ws[j])
                continue
            self.dsa.forward(b, q_idx, w, self.bt.k_idx, q, self.bt.kv, wl.k, self.bt.sm_scale,
                             self.out[:b.total_q], self.lse[:b.total_q], ws=self.ws[j])
        if wl.mla:
            self.dsa.mla_output(self.out, self.mw.w_kvb, self.mw.w_o, self.o_mid, self.y, self.mla_ws)

    def _index_key(self, j):
        """The new tokens' index keys (appended to the cache) and head weights."""
        b, (c, sn), ik = self.batches[j], self.rope[j], self.ik
        self.dsa.index_key_producer(b, self.x[:b.total_q], ik["wk"], ik["gamma"], ik["beta"], ik["eps"], c, sn,
                                    ik["ww"], self.bt.k_idx, self.bt.w[:b.total_q], self.ik_ws[j])

    # algorithmic work of one step
    def work(self):
        wl = self.wl
        calls = [0] if wl.base in ("decode", "indexshare") else range(len(self.batches))
        idx_flop = idx_bytes = att_flop = att_bytes = topk_bytes = 0
        for j in calls:
            pos = self.positions[j]
            pairs = sum(t + 1 for t in pos)
            sel = sum(min(wl.k, t + 1) for t in pos)
            idx_flop += IDX_FLOP_PER_PAIR * pairs
            att_flop += ATT_FLOP_PER_SEL * sel
            att_bytes += ATT_BYTES_PER_SEL * sel + ATT_BYTES_PER_QUERY * len(pos)
            topk_bytes += 4 * pairs + 4 * wl.k * len(pos)
            if wl.base == "indexshare":   # the shared layers repeat the attention only
                att_flop *= wl.steps
                att_bytes *= wl.steps
            if wl.fp8:
                idx_bytes += IDX8_BYTES_PER_KEY * sum(t + 1 for t in pos) + IDX8_BYTES_PER_QUERY * len(pos)
            elif wl.base in ("decode", "indexshare"):
                idx_bytes += IDX_BYTES_PER_KEY * sum(t + 1 for t in pos) + IDX_BYTES_PER_QUERY * len(pos)
            else:   # one sequence: keys read once per call (they stay in L2 across query groups)
                idx_bytes += IDX_BYTES_PER_KEY * (max(pos) + 1) + IDX_BYTES_PER_QUERY * len(pos)
        mla_flop = mla_bytes = 0
        if wl.mla:
            T = self.max_rows
            mla_flop = (ABS_FLOP_PER_TOKEN + OUT_FLOP_PER_TOKEN + IK_FLOP_PER_TOKEN) * T
            mla_bytes = ((ABS_BYTES_PER_TOKEN + OUT_BYTES_PER_TOKEN + IK_BYTES_PER_TOKEN) * T + ABS_WEIGHT_BYTES
                         + OUT_WEIGHT_BYTES + IK_WEIGHT_BYTES)
        return dict(idx_flop=idx_flop, idx_bytes=idx_bytes, att_flop=att_flop, att_bytes=att_bytes,
                    topk_bytes=topk_bytes, mla_flop=mla_flop, mla_bytes=mla_bytes)

    def kernel_times_us(self, reps: int):
        """Average device time of each step call (indexer, top-k, attention):
        `reps` back-to-back calls between two CUDA events on the launching
        stream, so host submission overlaps the device work."""
        import torch
        dsa, wl = self.dsa, self.wl
        stream = torch.cuda.current_stream()
        j = 0
        b = self.batches[j]
        q_idx, w, q = self._slices(j)
        ld = (b.max_ctx + 3) // 4 * 4
        scores = torch.empty((b.total_q, ld), dtype=torch.float32, device=self.dev)
        idx = torch.empty((b.total_q, wl.k), dtype=torch.int32, device=self.dev)
        calls = {
            "indexer": (lambda: dsa.indexer_scores_fp8(b, self.q8, self.qs, w, self.k8, self.ks, scores, ld=ld,
                                                      ws=self.ws[j])) if wl.fp8 else
                       (lambda: dsa.indexer_scores(b, q_idx, w, self.bt.k_idx, scores, ld=ld, ws=self.ws[j])),
            "topk": lambda: dsa.topk(b, scores, wl.k, idx, ld=ld, ws=self.ws[j]),
            "sparse_mla": lambda: dsa.sparse_mla_fwd(b, q, self.bt.kv, idx, wl.k, self.bt.sm_scale,
                                                     self.out[:b.total_q], self.lse[:b.total_q], ws=self.ws[j]),
        }
        if wl.mla:
            calls["index_key"] = lambda: self._index_key(0)
            calls["mla_absorb"] = lambda: dsa.mla_absorb_q(self.q_nope, self.q_pe, self.mw.w_kvb, self.bt.q,
                                                           self.mla_ws)
            calls["mla_output"] = lambda: dsa.mla_output(self.out, self.mw.w_kvb, self.mw.w_o, self.o_mid, self.y,
                                                         self.mla_ws)
        times = {}
        for name, fn in calls.items():
            fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            times[name] = e0.elapsed_time(e1) * 1e3 / reps
        return times

    def kernel_work_one_call(self):
        """Algorithmic work of the calls timed by kernel_times_us (call 0)."""
        wl = self.wl
        pos = self.positions[0]
        pairs = sum(t + 1 for t in pos)
        sel = sum(min(wl.k, t + 1) for t in pos)
        if wl.fp8:
            ib = IDX8_BYTES_PER_KEY * pairs + IDX8_BYTES_PER_QUERY * len(pos)
        elif wl.base in ("decode", "indexshare"):
            ib = IDX_BYTES_PER_KEY * pairs + IDX_BYTES_PER_QUERY * len(pos)
        else:
            ib = IDX_BYTES_PER_KEY * (max(pos) + 1) + IDX_BYTES_PER_QUERY * len(pos)
        work = {
            "indexer": dict(flop=IDX_FLOP_PER_PAIR * pairs, bytes=ib),
            "topk": dict(flop=0, bytes=4 * pairs + 4 * wl.k * len(pos)),
            "sparse_mla": dict(flop=ATT_FLOP_PER_SEL * sel,
                               bytes=ATT_BYTES_PER_SEL * sel + ATT_BYTES_PER_QUERY * len(pos)),
        }
        if wl.mla:
            T = self.max_rows
            nt = len(pos)
            work["index_key"] = dict(flop=IK_FLOP_PER_TOKEN * nt, bytes=IK_BYTES_PER_TOKEN * nt + IK_WEIGHT_BYTES)
            work["mla_absorb"] = dict(flop=ABS_FLOP_PER_TOKEN * T, bytes=ABS_BYTES_PER_TOKEN * T + ABS_WEIGHT_BYTES)
            work["mla_output"] = dict(flop=OUT_FLOP_PER_TOKEN * T, bytes=OUT_BYTES_PER_TOKEN * T + OUT_WEIGHT_BYTES)
        return work


def step_roofline(case: "Case", ms_step: float, peaks):
    """The whole step against its roofline: algorithmic bytes (HBM-bound
    decode) or flops (tensor-bound prefill) of one step over the step's
    time, as a fraction of the measured peak and of the nominal one."""
    wk, wl = case.work(), case.wl
    if wl.base in ("decode", "indexshare"):
        b = wk["idx_bytes"] + wk["att_bytes"] + wk["mla_bytes"]
        ach = b / (ms_step * 1e-3) / 1e9
        return {"bound": "hbm", "algorithmic": b, "achieved": ach, "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "frac_nominal": ach / NOMINAL_PEAKS["hbm_gbs"]}
    f = wk["idx_flop"] + wk["att_flop"] + wk["mla_flop"]
    ach = f / (ms_step * 1e-3) / 1e12
    return {"bound": "tensor", "algorithmic": f, "achieved": ach, "unit": "TFLOP/s",
            "frac": ach / peaks["bf16_tflops"], "frac_nominal": ach / NOMINAL_PEAKS["bf16_tflops"]}


def timed_steps(case: "Case", K: int, stream):
    """K steps between CUDA events on the launching stream (one event after
    every step): total milliseconds and the per-step times."""
    import torch
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    evs[0].record(stream)
    for i in range(K):
        case.step(i)
        evs[i + 1].record(stream)
    return evs


def per_step_ms(evs):
    return [evs[i].elapsed_time(evs[i + 1]) for i in range(len(evs) - 1)]


def side_workload(name: str, dev, peaks, reps: int):
    """One more workload timed in the same run (warm-up 3, then 10 steps for
    a prefill or 200 for a decode step), with its kernel times and its
    whole-step roofline fraction."""
    import torch
    wl = W.WORKLOADS[name]
    case = Case(wl, wl.seed, dev)
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    for i in range(3):
        case.step(i)
    torch.cuda.synchronize()
    K = 200 if wl.base == "decode" else 10
    t0 = time.time()
    evs = timed_steps(case, K, stream)
    torch.cuda.synchronize()
    clocks.timed(t0, time.time())
    ms = evs[0].elapsed_time(evs[-1])
    steps = per_step_ms(evs)
    t0 = time.time()
    for i in range(max(1, int(0.3 / (ms / K / 1e3)))):
        case.step(i)
    torch.cuda.synchronize()
    clocks.hold(t0, time.time())
    times = case.kernel_times_us(reps)
    clk = clocks.stop()
    status = case.dsa.read_device_status(case.ws[0])
    res = {"metric": case.metric, "value": case.units_per_step * K / (ms / 1e3), "unit": case.unit, "steps": K,
           "warmup": 3, "ms_per_step": ms / K, "ms_per_step_median": statistics.median(steps),
           "step_roofline": step_roofline(case, ms / K, peaks),
           "kernel_us": {k: round(v, 2) for k, v in times.items()}, "device_status": status, "clocks": clk}
    del case
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi samples (every 50 ms) around the timed region; the summary
    uses the samples whose timestamps fall inside it."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.window = None
        self.hold_window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50",
                 "-i", str(self.gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def timed(self, t0: float, t1: float):
        self.window = (t0, t1)

    def hold(self, t0: float, t1: float):
        self.hold_window = (t0, t1)

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        import datetime
        samples = []
        for line in out.strip().splitlines():
            r = [x.strip() for x in line.split(",")]
            if len(r) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                samples.append((ts, float(r[1]), float(r[2]), tuple(r[5:9])))
            except ValueError:
                continue
        def within(w):
            return [x for x in samples if w and w[0] - 0.05 <= x[0] <= w[1] + 0.05]

        inside = within(self.window)
        scope = "timed region"
        if len(inside) < 2:
            # a short timed region: add the ~0.5 s repeat of the same steps
            # that follows it
            inside = sorted(set(inside) | set(within(self.hold_window)))
            scope = "timed region and a 0.5 s repeat of the same steps right after it"
        if len(inside) < 2:
            inside, scope = samples, "warm-up, timed region and per-kernel timing"
        sm = [x[1] for x in inside]
        reasons = sorted({n for x in inside for n, v in zip(self.REASONS, x[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(x[2] for x in inside) if inside else None,
                "reasons": reasons, "samples": len(sm), "scope": scope}


# ------------------------------------------------------------- cpu oracle --

def host_sample(case: Case, n_seq: int):
    """Copy a sample of the workload to the host as a numpy Batch (decode: the
    first n_seq sequences; prefill: evenly spaced query rows)."""
    import torch
    bt, wl = case.bt, case.wl

    def bits(t):
        return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

    if wl.base == "decode":
        ctx = wl.ctx
        n_seq = min(n_seq, wl.B)
        rows = slice(0, n_seq)
        cache = slice(0, n_seq * bt.stride)
        b = W.Batch(B=n_seq, stride=bt.stride, q_off=np.arange(n_seq + 1, dtype=np.int32),
                    ctx_len=np.full(n_seq, ctx, np.int32), q_idx=bits(bt.q_idx[rows]),
                    w=bt.w[rows].cpu().numpy(), k_idx=bits(bt.k_idx[cache]), q=bits(bt.q[rows]),
                    kv=bits(bt.kv[cache]), k=wl.k, sm_scale=bt.sm_scale)
        return b, list(range(n_seq)), n_seq / wl.B, f"{n_seq} of {wl.B} sequences of one decode step"
    T = wl.ctx
    b = W.Batch(B=1, stride=bt.stride, q_off=np.array([0, T], np.int32), ctx_len=np.array([T], np.int32),
                q_idx=bits(bt.q_idx), w=bt.w.cpu().numpy(), k_idx=bits(bt.k_idx), q=bits(bt.q), kv=bits(bt.kv),
                k=wl.k, sm_scale=bt.sm_scale)
    rows = sorted(set(int(x) for x in np.linspace(0, T - 1, min(n_seq, T))))
    return b, rows, len(rows), f"{len(rows)} evenly spaced query rows of the {T}-token prefill"


def oracle_path_seconds(b, rows, attention_layers: int = 1, mla=None, ik=None, fp8=None):
    """The oracle's whole path on `rows`; attention_layers > 1 repeats the
    attention on the same indices (IndexShare's shared layers); mla =
    (q_nope, q_pe, w_kv_b, w_o) of those rows adds the projections around it,
    ik = (x, IndexKeyParams, cos, sin) the index-key producer."""
    import oracle
    t0 = time.perf_counter()
    if ik is not None:
        x, p, c, sn = ik
        oracle.index_key(x, p.wk, p.gamma, p.beta, p.eps, c, sn, p.ww)
    if mla is not None:
        oracle.mla_absorb_q(mla[0], mla[1], mla[2])
    if fp8 is not None:          # (k8, ks) of the cache: the queries are quantized here
        q8, qs = oracle.quantize_fp8(b.q_idx, 128)
        sc = oracle.indexer_scores_fp8(b, q8.reshape(-1), qs, fp8[0], fp8[1], rows)
    else:
        sc = oracle.indexer_scores(b, rows)
    ix = oracle.topk(b, np.nan_to_num(sc.astype(np.float32), nan=0.0), rows=rows, k=b.k)
    for _ in range(attention_layers):
        o, _ = oracle.sparse_mla(b, ix, rows=rows)
    if mla is not None:
        oracle.mla_output(o, mla[2], mla[3])
    return time.perf_counter() - t0


def _bits(t):
    import torch
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def cpu_baseline(case: Case, unit: str):
    import oracle
    n = 64 if case.wl.base == "decode" else 48      # decode: every sequence of the step (B <= 64)
    b, rows, units, sample = host_sample(case, n)
    mla = ik = None
    if case.wl.mla:
        import torch
        ri = torch.tensor(rows, dtype=torch.long, device=case.q_nope.device)
        mla = (_bits(case.q_nope[ri]), _bits(case.q_pe[ri]), _bits(case.mw.w_kvb), _bits(case.mw.w_o))
        ip = W.IndexKeyParams(_bits(case.ik["wk"]), _bits(case.ik["ww"]), case.ik["gamma"].cpu().numpy(),
                              case.ik["beta"].cpu().numpy(), case.ik["eps"])
        c, sn = W.rotary_rows([case.positions[0][r] for r in rows])
        ik = (_bits(case.x[ri]), ip, c, sn)
        sample += "; with the index-key producer and the MLA projections"
    fp8 = None
    if case.wl.fp8:
        nk = b.B * b.stride
        fp8 = (case.k8[:nk].cpu().numpy().reshape(-1), case.ks[:nk].cpu().numpy().astype(np.float64))
        sample += "; E4M3 keys of the cache, queries quantized by the oracle"
    secs = oracle_path_seconds(b, rows, mla=mla, ik=ik, fp8=fp8)
    # units: decode -> fraction of one step; prefill -> query rows (tokens)
    return {"value": units / secs, "unit": unit, "cores": oracle.num_threads(), "kind": "oracle",
            "sample": sample + f" (full path: indexer, top-k, attention; {secs:.1f} s in fp64)"}


# --------------------------------------------------------------- reference --

def run_reference(args):
    """The oracle as the reference arm, on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    wl = W.WORKLOADS[args.workload]
    K, Wu = default_steps(wl)
    K = args.steps if args.steps is not None else K
    Wu = args.warmup if args.warmup is not None else Wu
    # one bounded sample per step, drawn with the numpy recipe: one query
    # row per host thread (the oracle runs its rows in parallel)
    shared_layers = wl.steps - 1 if wl.base == "indexshare" else 0
    threads = max(1, oracle.num_threads())
    if wl.base in ("decode", "indexshare"):
        ns = min(wl.B, threads)
        b = W.make_batch_np([wl.ctx] * ns, [1] * ns, wl.k, wl.seed, key_kind=wl.key_kind)
        rows = list(range(ns))
        frac = ns / wl.B
        sample = f"{ns} of {wl.B} sequences of one decode step per timed step"
    else:
        T = wl.ctx
        nq = threads
        b = W.make_batch_np([T], [T], wl.k, wl.seed, key_kind=wl.key_kind) if T <= 16384 else None
        if b is None:
            print(json.dumps({"impl": "reference", "unavailable": "oracle sample of this workload exceeds host memory"}))
            return
        rows = [int(x) for x in np.linspace(0, T - 1, nq)]
        frac = nq
        sample = f"{nq} evenly spaced query rows per timed step"
    mla = ik = None
    if wl.mla:
        mw = W.make_mla_weights_np(wl.seed + 1)
        qn, qp = W.make_mla_queries_np(len(rows), wl.seed + 2)
        mla = (qn, qp, mw.w_kvb, mw.w_o)
        c, sn = W.rotary_rows([wl.ctx - 1] * len(rows) if wl.base == "decode" else rows)
        ik = (W.make_hidden_np(len(rows), wl.seed + 4), W.make_index_key_params_np(wl.seed + 3), c, sn)
        sample += "; with the index-key producer and the MLA projections"

    fp8 = None
    if wl.fp8:                   # the cache's E4M3 keys, quantized once before timing
        k8, ks = oracle.quantize_fp8(b.k_idx, 128)
        fp8 = (k8.reshape(-1), ks)
        sample += "; E4M3 keys, queries quantized in each step"

    def one_step():
        oracle_path_seconds(b, rows, 1 + shared_layers, mla=mla, ik=ik, fp8=fp8)

    for _ in range(Wu):
        one_step()
    t0 = time.perf_counter()
    for _ in range(K):
        one_step()
    secs = (time.perf_counter() - t0) / K
    value = frac / secs
    metric, unit = metric_for(wl)
    line = {"impl": "reference", "metric": metric, "value": value, "unit": unit, "n_gpus": args.gpus,
            "steps": K, "warmup": Wu, "ms_per_step": 1e3 * secs,
            "ms_per_full_step_extrapolated": 1e3 / value if unit == "steps/s" else 1e3 * wl.ctx / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": base_config(wl, 1),
            "cpu_baseline": {"value": value, "unit": unit, "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------- multi-rank --

def max_over_ranks(x: float, device) -> float:
    """The largest of every rank's x (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_step_per_rank: float, steps: int, world: int, ms_max: float) -> float:
    """Units processed by all ranks per second of the slowest rank's time
    (weak scaling: every rank runs its own batch)."""
    return units_per_step_per_rank * steps * world / (ms_max / 1e3)


# --------------------------------------------------------------------- dsa --

def traffic_from_profiles(kernel: str, workload: str):
    """dram bytes per launch recorded by an ncu capture, if the kernel's
    source is unchanged since (profiles/ncu_traffic.txt)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    src = {"indexer": "indexer.cu", "topk": "topk.cu", "sparse_mla": "sparse_mla.cu", "mla_absorb": "mla_proj.cu",
           "mla_output": "mla_proj.cu", "index_key": "index_key.cu"}.get(kernel)
    if src is None:
        return None
    with open(os.path.join(ROOT, "sparse_attention_gb300", "csrc", src), "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    for line in open(path):
        kv = dict(x.split("=", 1) for x in line.split() if "=" in x)
        if kv.get("kernel") == kernel and kv.get("workload") == workload and kv.get("src_sha") == sha:
            return float(kv["dram_bytes_per_launch"])
    return None


def run_dsa(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from sparse_attention_gb300 import build as B
    if rank == 0 or world == 1:
        B.build()
    if world > 1:
        dist.barrier()
    import sparse_attention_gb300 as dsa
    dsa.load_library()

    wl = W.WORKLOADS[args.workload]
    K, Wu = default_steps(wl)
    K = args.steps if args.steps is not None else K
    Wu = max(3, args.warmup if args.warmup is not None else Wu)
    case = Case(wl, wl.seed + 1000 * rank, dev)
    stream = torch.cuda.current_stream()

    def barrier():
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()

    clocks = ClockSampler(local)
    clocks.start()
    for i in range(Wu):
        case.step(i)
    barrier()
    n0 = dsa.kernel_launch_count()
    barrier()
    t_start = time.time()
    evs = timed_steps(case, K, stream)
    barrier()
    clocks.timed(t_start, time.time())
    launches = dsa.kernel_launch_count() - n0
    ms = max_over_ranks(evs[0].elapsed_time(evs[-1]), dev)
    step_ms = per_step_ms(evs)
    status = dsa.read_device_status(case.ws[0])
    value = whole_job_value(case.units_per_step, K, world, ms)
    # a short timed region holds few clock samples: repeat the same steps
    # for about half a second under the sampler (not timed)
    t_hold = time.time()
    n_hold = int(args.clock_hold_s / max(ms / K / 1e3, 1e-6))
    for i in range(n_hold):
        case.step(i)
    barrier()
    clocks.hold(t_hold, time.time())

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e and wl.base != "indexshare":
        e2e = run_e2e(case, K, Wu, barrier, lambda x: max_over_ranks(x, dev), world)

    # per-kernel device times and the roofline of the dominant kernel
    times = case.kernel_times_us(args.kernel_reps)
    clk = clocks.stop()
    work = case.kernel_work_one_call()
    peaks, peak_src = load_peaks()
    dom = max(times, key=times.get)
    kw = work[dom]
    if wl.base not in ("decode", "indexshare") and dom in ("indexer", "sparse_mla", "mla_absorb", "mla_output",
                                                         "index_key"):
        achieved = kw["flop"] / (times[dom] * 1e-6) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"]}
    else:
        achieved = kw["bytes"] / (times[dom] * 1e-6) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"]}
    sr = step_roofline(case, ms / K, peaks)
    roof.update({"kernel": dom, "peak_source": f"{peak_src} ({'burst' if roof['bound'] == 'tensor' else 'copy'})",
                 "traffic": traffic_from_profiles(dom, wl.name),
                 "kernel_us": {k: round(v, 2) for k, v in times.items()},
                 "algorithmic_per_launch": kw,
                 "step_frac": sr["frac"], "step_frac_nominal": sr["frac_nominal"], "step": sr})

    if rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and world == 1 and wl.base != "indexshare":
        cpu = cpu_baseline(case, case.unit)
    case_metric, case_unit = case.metric, case.unit
    wk = case.work()
    cfg = base_config(wl, world)
    details = {"algorithmic_per_step": {"indexer_tflop": wk["idx_flop"] / 1e12,
                                        "attention_tflop": wk["att_flop"] / 1e12,
                                        "indexer_gb": wk["idx_bytes"] / 1e9, "attention_gb": wk["att_bytes"] / 1e9},
               "device_status": status}
    if wl.mla:
        details["algorithmic_per_step"].update({"mla_projection_tflop": wk["mla_flop"] / 1e12,
                                                "mla_projection_gb": wk["mla_bytes"] / 1e9})
        details["mla_device_status"] = dsa.read_device_status(case.mla_ws)
    if wl.base in ("decode", "indexshare"):
        details["tokens_per_s"] = value * wl.B
    details["ms_per_step_median"] = statistics.median(step_ms)
    if wl.name == DEFAULT_WORKLOAD and world == 1 and not args.no_side:
        # the metric's other half (prefill tokens/s) and the long-context
        # decode, timed in the same run
        del case
        torch.cuda.empty_cache()
        details["other_workloads"] = {n: side_workload(n, dev, peaks, args.kernel_reps) for n in SIDE_WORKLOADS}
    line = {"metric": case_metric, "value": value, "unit": case_unit, "n_gpus": world, "steps": K, "warmup": Wu,
            "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic", "config": cfg, "roofline": roof, "cpu_baseline": cpu,
            "e2e": e2e, "gpu_launches": launches, "clocks": clk, "details": details}
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def pack_layout(srcs, align: int = 256):
    """Byte layout of tensors packed one after another into one block:
    {name: (offset, nbytes, dtype, shape)} and the block's size; every
    offset is a multiple of `align`."""
    segs, nbytes = {}, 0
    for n, t in srcs:
        segs[n] = (nbytes, t.numel() * t.element_size(), t.dtype, t.shape)
        nbytes = (nbytes + segs[n][1] + align - 1) // align * align
    return segs, nbytes


def pack_into(blk, segs, srcs):
    """Copies each tensor's bytes to its place in the uint8 block."""
    import torch
    for n, t in srcs:
        o0, nb, _, _ = segs[n]
        blk[o0:o0 + nb].copy_(t.reshape(-1).view(torch.uint8).cpu())


def seg_view(blk, segs, n):
    """Tensor n as a view of the block (its dtype and shape)."""
    o0, nb, dt, shape = segs[n]
    return blk[o0:o0 + nb].view(dt).view(shape)


def run_e2e(case: Case, K: int, Wu: int, barrier, max_over_ranks, world: int):
    """Same metric through the public API with every step's inputs copied in
    from pinned host memory and its result read back to pinned host memory.
    Inputs and results are double-buffered: step i + 1's host-to-device copy
    (its own stream) overlaps step i's kernels, step i's read-back (a third
    stream) overlaps step i + 1's."""
    import torch
    wl, bt = case.wl, case.bt
    comp = torch.cuda.current_stream()
    h2d_s, d2h_s = torch.cuda.Stream(device=comp.device), torch.cuda.Stream(device=comp.device)
    # the step's inputs (holder, attribute) and result: the absorbed q and
    # the latent output, or (MLA layer) q_nope / q_pe / x and the o_proj
    # output y (that layer produces w and the new index keys itself)
    if wl.mla:
        names = {"q_idx": (bt, "q_idx"), "q_nope": (case, "q_nope"), "q_pe": (case, "q_pe"), "x": (case, "x")}
        res = (case, "y")
    else:
        names = {"q_idx": (bt, "q_idx"), "w": (bt, "w"), "q": (bt, "q")}
        res = (case, "out")
    decode = wl.base == "decode"
    if not decode:               # a prefill brings its whole caches
        names["kv"] = (bt, "kv")
        if not wl.mla:
            names["k_idx"] = (bt, "k_idx")
    own = {n: getattr(o, a) for n, (o, a) in names.items()}
    rbufs = [getattr(*res), torch.empty_like(getattr(*res))]
    out_h = [torch.empty(rbufs[0].shape, dtype=rbufs[0].dtype).pin_memory() for _ in range(2)]
    # A decode step appends the new token's cache rows.  The caches they go
    # into are double-buffered like the inputs: step i + 1's rows are copied
    # from pinned host memory (to a staging buffer, then into their rows) into
    # the other buffer while step i runs (both buffers hold the same cache),
    # so no copy waits on the kernels and none touches a row that a running
    # step reads.
    owners, caches, rows = [], [{}, {}], [[], []]
    if decode:
        owners = [(bt, "kv", 576)]
        if wl.fp8:
            owners += [(case, "k8", 128), (case, "ks", 0)]
        elif not wl.mla:          # (the MLA layer writes its index keys on the device)
            owners += [(bt, "k_idx", 128)]

        def row_of(t, width):
            v = t.view(wl.B, bt.stride, width) if width else t.view(wl.B, bt.stride)
            return v[:, wl.ctx - 1]
        for o, a, width in owners:
            t = getattr(o, a)
            caches[0][a], caches[1][a] = t, t.clone()
            rows[0].append(row_of(caches[0][a], width))
            rows[1].append(row_of(caches[1][a], width))
    # A step's host data (its inputs, then its new cache rows) is one pinned
    # block that one copy moves into one of two device blocks; the inputs
    # are views of that block (256-byte aligned) and the rows are staged in
    # it before being scattered into their cache rows.
    srcs = list(own.items()) + [(f"row:{a}", r.contiguous()) for (_, a, _), r in zip(owners, rows[0])]
    segs, nbytes = pack_layout(srcs)
    host_blk = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    pack_into(host_blk, segs, srcs)
    dev_blk = [torch.empty(nbytes, dtype=torch.uint8, device=comp.device) for _ in range(2)]
    bufs = [{n: seg_view(dev_blk[k], segs, n) for n in own} for k in range(2)]
    stage = [[seg_view(dev_blk[k], segs, f"row:{a}") for _, a, _ in owners] for k in range(2)]
    h2d = nbytes
    d2h = out_h[0].numel() * out_h[0].element_size()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_read = [torch.cuda.Event() for _ in range(2)]
    used = [False, False]

    def prefetch(i):
        k = i % 2
        with torch.cuda.stream(h2d_s):
            if used[k]:
                h2d_s.wait_event(ev_done[k])        # the step that last read buffer k has finished
            dev_blk[k].copy_(host_blk, non_blocking=True)
            for st, row in zip(stage[k], rows[k]):
                row.copy_(st, non_blocking=True)
            ev_in[k].record(h2d_s)

    def compute(i):
        k = i % 2
        comp.wait_event(ev_in[k])
        if used[k]:
            comp.wait_event(ev_read[k])             # the read-back of result buffer k has finished
        for n, (o, a) in names.items():
            setattr(o, a, bufs[k][n])
        for o, a, _ in owners:
            setattr(o, a, caches[k][a])
        setattr(res[0], res[1], rbufs[k])
        case.step(len(case.batches) - 1 if decode else i)
        ev_done[k].record(comp)
        used[k] = True

    def readback(i):
        k = i % 2
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(ev_done[k])
            out_h[k].copy_(rbufs[k], non_blocking=True)
            ev_read[k].record(d2h_s)

    def run(n):
        prefetch(0)
        for i in range(n):
            compute(i)
            if i + 1 < n:
                prefetch(i + 1)
            readback(i)
        comp.wait_stream(d2h_s)
        comp.wait_stream(h2d_s)

    run(Wu)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    run(K)
    e1.record(comp)
    barrier()
    ms = max_over_ranks(e0.elapsed_time(e1))
    for o, a, _ in owners:                  # the case's own caches and inputs again
        setattr(o, a, caches[0][a])
    for n, (o, a) in names.items():
        setattr(o, a, own[n])
    setattr(res[0], res[1], rbufs[0])
    del caches, dev_blk, bufs, stage
    value = whole_job_value(case.units_per_step, K, world, ms)
    api = ("sparse_attention_gb300.index_key_producer + mla_absorb_q + forward + mla_output" if wl.mla
           else "sparse_attention_gb300.forward")
    return {"value": value, "unit": case.unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "api": api,
            "overlap": "double-buffered: next step's copy-in (inputs and new cache rows as one pinned block, the "
                       "rows then scattered into the other of two cache buffers) and this step's read-back "
                       "overlap the kernels"}


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_dsa(args)


if __name__ == "__main__":
    main()
