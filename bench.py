#!/usr/bin/env python
"""Benchmark of the routed-MoE FFN with block-scaled FP4 experts on GB300.

Default workload: the Qwen-shaped decode stack -- 48 layers, each with 512
NVFP4 experts (H=2560, I=640, 2,764,800-byte records, ~68 GB resident in
HBM), top-10 routing, one token per step; each layer's input is the previous
layer's output, RMS-normalised.  A step runs router -> experts -> RMS chaining
for all 48 layers.  The metric is expert GB/s: the bytes of the records the
step selects divided by the step time, and its fraction of the HBM roofline.

The same run also measures the four other workloads, each under its own key
of the JSON line with its own roofline and oracle sample: ``config0`` (one
layer, one token, 64 experts), ``prompt`` (2451 tokens through one layer,
Zipf-skewed routing over 512 experts, the tensor-core path), ``config3``
(DeepSeek-shaped MXFP4 layer, 384 experts of 18,800,640 bytes, top-6, 40
calls with the L2 flushed between calls) and ``config4`` (32 tokens through
the 48-layer stack).

``--impl reference`` times the CPU oracle (float64 numpy) on a bounded sample
of the same workload instead.

One JSON line is printed by rank 0.  Multi-GPU runs (torchrun) are independent
replicas: each rank decodes its own tokens, no data-path collective.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "expert GB/s & fraction of HBM peak (decode); tokens/s per MoE layer (prompt)"
H, I, E, K_TOP, LAYERS = 2560, 640, 512, 10, 48
WORKLOAD_ID = 1
UNIQUE_EXPERTS = 1024


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"moe_bench_clocks_{os.getpid()}_{device_index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# the decode-stack workload on the GPU
# ---------------------------------------------------------------------------
class DecodeStack:
    def __init__(self, torch, moe, synth, device, rank: int, steps_total: int):
        self.torch, self.moe, self.synth = torch, moe, synth
        self.dev = device
        self.s = moe.shape(H, I, moe.FMT_NVFP4)
        self.rec_bytes = moe.moe_expert_record_bytes(self.s)
        t0 = time.time()
        uniq = torch.empty(UNIQUE_EXPERTS, self.rec_bytes, dtype=torch.uint8, device=device)
        for u in range(UNIQUE_EXPERTS):
            g, up, d = synth.expert_weights(H, I, synth.expert_seed(WORKLOAD_ID, 0, u), device=device)
            moe.fp4_pack_expert(g, up, d, self.s, record=uniq[u])
        # 48 x 512 slots, each its own physical copy of a seeded choice of record
        self.slots = torch.empty(LAYERS, E, self.rec_bytes, dtype=torch.uint8, device=device)
        self.choice = []
        for L in range(LAYERS):
            rng = np.random.default_rng(synth.seed_of(WORKLOAD_ID, L, synth.T_PERM))
            ch = rng.permutation(UNIQUE_EXPERTS)[:E]
            self.choice.append(ch)
            for e in range(E):  # one contiguous device-to-device copy per slot
                self.slots[L, e].copy_(uniq[int(ch[e])])
        del uniq
        self.ptrs = [moe.pointer_table([self.slots[L, e] for e in range(E)]) for L in range(LAYERS)]
        self.wr = torch.stack([synth.router_weights(E, H, synth.seed_of(WORKLOAD_ID, L, synth.T_ROUTER),
                                                    device=device) for L in range(LAYERS)])
        # one input token per step (distinct tokens, seeded)
        self.x0 = torch.cat([synth.activations(1, H, synth.seed_of(WORKLOAD_ID, 100 + s, synth.T_X),
                                               device=device) for s in range(steps_total)])
        self.x = torch.empty(1, H, dtype=torch.bfloat16, device=device)
        self.idx = torch.empty(1, K_TOP, dtype=torch.int32, device=device)
        self.w = torch.empty(1, K_TOP, dtype=torch.float32, device=device)
        self.logits = torch.empty(1, E, dtype=torch.float32, device=device)
        self.y = torch.empty(1, H, dtype=torch.float32, device=device)
        self.ws = torch.zeros(moe.moe_experts_decode_workspace(1, K_TOP, self.s), dtype=torch.uint8,
                              device=device)
        self.st = torch.zeros(1, dtype=torch.int32, device=device)
        self.setup_s = time.time() - t0
        self.kernels_per_step = LAYERS
        self.ev = None

    def expert_bytes_per_step(self):
        return LAYERS * K_TOP * self.rec_bytes

    def run_layers(self, timing_events=None):
        """One token through the 48 layers, one launch per layer: layer 0
        routes x0; every later layer RMS-chains the previous output inside
        its launch (y is overwritten in place)."""
        moe = self.moe
        for L in range(LAYERS):
            if timing_events is not None:
                timing_events[L][0].record()
            if L == 0:
                moe.moe_decode_layer(self.wr[L], None, K_TOP, self.ptrs[L], self.s, x=self.x, idx=self.idx,
                                     weights=self.w, logits=self.logits, y=self.y, workspace=self.ws,
                                     dev_status=self.st)
            else:
                moe.moe_decode_layer(self.wr[L], None, K_TOP, self.ptrs[L], self.s, y_prev=self.y, eps=1e-6,
                                     x_out=self.x, idx=self.idx, weights=self.w, logits=self.logits, y=self.y,
                                     workspace=self.ws, dev_status=self.st)
            if timing_events is not None:
                timing_events[L][1].record()

    def stack_buffers(self):
        """Outputs of the single-launch stack (moe_decode_stack)."""
        torch, moe = self.torch, self.moe
        if not hasattr(self, "stk"):
            self.stk = {"ptrs": torch.stack(self.ptrs),
                        "idx": torch.empty(LAYERS, 1, K_TOP, dtype=torch.int32, device=self.dev),
                        "w": torch.empty(LAYERS, 1, K_TOP, dtype=torch.float32, device=self.dev),
                        "ws": torch.zeros(moe.moe_experts_decode_workspace(1, K_TOP, self.s), dtype=torch.uint8,
                                          device=self.dev)}
        return self.stk

    def run_stack_kernel(self):
        """One token through the 48 layers in one launch of the persistent
        kernel (the same bits as run_layers)."""
        b = self.stack_buffers()
        self.moe.moe_decode_stack(self.x, self.wr, None, K_TOP, b["ptrs"], self.s, eps=1e-6, idx=b["idx"],
                                  weights=b["w"], logits=self.logits, x_out=self.xo if hasattr(self, "xo") else None,
                                  y=self.y, workspace=b["ws"], dev_status=self.st)

    def capture(self, with_events: bool):
        torch = self.torch
        self.x.copy_(self.x0[0:1])
        self.run_layers()  # warm, sets kernel attributes outside capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        ev = None
        if with_events:
            ev = [(torch.cuda.Event(enable_timing=True, external=True),
                   torch.cuda.Event(enable_timing=True, external=True)) for _ in range(LAYERS)]
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            self.run_layers(ev)
        return g, ev


def speculative_routing(torch, moe, wl, tokens=16):
    """Hit rate of speculative next-layer routing on the decode stack: layer
    L+1's router applied to layer L's input, against layer L+1's actual
    top-k (the pages guess the next layer's experts this way to start their
    copies early).  Reported for k guesses and for 16 guesses (fraction of the
    true top-k covered).  Random router weights have no layer-to-layer
    structure, so the expected rate is about k / E."""
    hits, hits16, n = 0, 0, 0
    for s in range(tokens):
        xs, idxs = [], []
        wl.x.copy_(wl.x0[s % wl.x0.shape[0]:s % wl.x0.shape[0] + 1])
        for L in range(LAYERS):
            if L == 0:
                moe.moe_decode_layer(wl.wr[L], None, K_TOP, wl.ptrs[L], wl.s, x=wl.x, idx=wl.idx, weights=wl.w,
                                     logits=wl.logits, y=wl.y, workspace=wl.ws, dev_status=wl.st)
                xs.append(wl.x.clone())
            else:
                moe.moe_decode_layer(wl.wr[L], None, K_TOP, wl.ptrs[L], wl.s, y_prev=wl.y, eps=1e-6, x_out=wl.x,
                                     idx=wl.idx, weights=wl.w, logits=wl.logits, y=wl.y, workspace=wl.ws,
                                     dev_status=wl.st)
                xs.append(wl.x.clone())
            idxs.append(wl.idx.clone())
        for L in range(LAYERS - 1):
            g10, _, _ = moe.moe_router_topk(xs[L], wl.wr[L + 1], None, K_TOP)
            g16, _, _ = moe.moe_router_topk(xs[L], wl.wr[L + 1], None, 16)
            true = set(idxs[L + 1].flatten().tolist())
            hits += len(true & set(g10.flatten().tolist()))
            hits16 += len(true & set(g16.flatten().tolist()))
            n += K_TOP
    return {"tokens": tokens, "layer_pairs": tokens * (LAYERS - 1),
            "hit_rate_top10": round(hits / n, 4), "coverage_top16": round(hits16 / n, 4),
            "chance_k_over_E": round(K_TOP / E, 4),
            "note": "router of layer L+1 on layer L's input vs layer L+1's own top-10; random router weights"}


class PromptLayer:
    """Qwen-shaped prompt through one MoE layer: T=2451 tokens, 512 NVFP4
    experts, top-10 with a Zipf(1.1) router bias; a step is router + the
    grouped tensor-core expert pass."""

    T = 2451
    WORKLOAD = 2

    def __init__(self, torch, moe, synth, device):
        self.torch, self.moe = torch, moe
        self.s = moe.shape(H, I, moe.FMT_NVFP4)
        rb = moe.moe_expert_record_bytes(self.s)
        self.pool = torch.empty(E, rb, dtype=torch.uint8, device=device)
        for e in range(E):
            g, up, d = synth.expert_weights(H, I, synth.expert_seed(self.WORKLOAD, 0, e), device=device)
            moe.fp4_pack_expert(g, up, d, self.s, record=self.pool[e])
        self.ptrs = moe.pointer_table([self.pool[e] for e in range(E)])
        self.x = synth.activations(self.T, H, synth.seed_of(self.WORKLOAD, 0, synth.T_X), device=device)
        self.wr = synth.router_weights(E, H, synth.seed_of(self.WORKLOAD, 0, synth.T_ROUTER), device=device)
        self.bias = synth.zipf_bias(E, synth.seed_of(self.WORKLOAD, 0, synth.T_BIAS)).to(device)
        self.idx = torch.empty(self.T, K_TOP, dtype=torch.int32, device=device)
        self.w = torch.empty(self.T, K_TOP, dtype=torch.float32, device=device)
        self.logits = torch.empty(self.T, E, dtype=torch.float32, device=device)
        self.y = torch.empty(self.T, H, dtype=torch.float32, device=device)
        self.ws = torch.empty(moe.moe_experts_grouped_workspace(self.T, K_TOP, E, self.s),
                              dtype=torch.uint8, device=device)
        self.st = torch.zeros(1, dtype=torch.int32, device=device)
        # L2 flush by reading (not writing) a 512 MB buffer: a write sweep would
        # leave the L2 full of dirty lines whose write-back lands in the next call
        self.flush = torch.ones(512 << 18, dtype=torch.int32, device=device)
        self.flush_out = torch.zeros((), dtype=torch.int64, device=device)

    def step(self):
        moe = self.moe
        moe.moe_router_topk(self.x, self.wr, self.bias, K_TOP, self.idx, self.w, self.logits)
        moe.moe_experts_grouped(self.x, self.idx, self.w, self.ptrs, self.s, self.y, self.ws, self.st)

    def measure(self, steps: int, warm: int):
        torch = self.torch
        for _ in range(warm):
            self.step()
        torch.cuda.synchronize()
        tot_step, tot_exp = 0.0, 0.0
        for i in range(steps):
            a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            torch.sum(self.flush, 0, out=self.flush_out)  # L2 flush (read sweep)
            _gpu_spacer(torch)
            a.record()
            self.moe.moe_router_topk(self.x, self.wr, self.bias, K_TOP, self.idx, self.w, self.logits)
            b.record()
            self.moe.moe_experts_grouped(self.x, self.idx, self.w, self.ptrs, self.s, self.y, self.ws,
                                         self.st)
            c.record()
            torch.cuda.synchronize()
            tot_step += a.elapsed_time(c)
            tot_exp += b.elapsed_time(c)
        ms, ms_exp = tot_step / steps, tot_exp / steps
        counts = torch.bincount(self.idx.flatten().long(), minlength=E)
        hit = int((counts > 0).sum().item())
        flops = 2.0 * self.T * K_TOP * 3 * H * I
        P = self.T * K_TOP
        # algorithmic bytes of the expert pass: every hit record once, X read,
        # the BF16 SwiGLU intermediate written and read, Y written
        nbytes = hit * self.pool.shape[1] + self.T * H * 2 + 2 * P * I * 2 + self.T * H * 4
        peak, kind = _peaks()
        achieved = nbytes / (ms_exp / 1e3) / 1e9
        return {"tokens_per_s": round(self.T / (ms / 1e3), 1), "ms_per_layer": round(ms, 4),
                "expert_pass_ms": round(ms_exp, 4),
                "expert_tflops": round(flops / (ms_exp / 1e3) / 1e12, 2),
                "expert_weight_gbs": round(hit * self.pool.shape[1] / (ms_exp / 1e3) / 1e9, 1),
                "experts_hit": hit, "max_tokens_per_expert": int(counts.max().item()),
                "tokens": self.T, "dev_status": int(self.st.item()),
                "roofline": {"bound": "hbm", "kernel": "moe_experts_grouped (bucketing + grouped_kernel phases 0 and 1)",
                             "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                             "peak_kind": kind + " (burst copy)", "frac": round(achieved / peak, 4),
                             "bytes_per_call": nbytes, "flops_per_call": flops,
                             "tensor_tflops": round(flops / (ms_exp / 1e3) / 1e12, 2),
                             "note": "HBM floor at the measured peak vs the FP16/BF16 tensor floor: bytes bound"},
                "l2": "flushed between steps by reading a 512 MB buffer"}


def _gpu_spacer(torch):
    """A ~1 ms spin kernel enqueued before a timed call's start event, so the
    host has enqueued the event and the call before the GPU reaches them: the
    timed interval then holds the call's own device time, not host launch
    gaps.  It touches no memory, so a preceding L2 flush stays in effect."""
    torch.cuda._sleep(2_000_000)


def _l2_flusher(torch, device):
    """A read sweep over 512 MB (four times the L2): evicts the L2 without
    leaving dirty lines whose write-back would land in the next timed call."""
    buf = torch.ones(512 << 18, dtype=torch.int32, device=device)
    out = torch.zeros((), dtype=torch.int64, device=device)
    return lambda: torch.sum(buf, 0, out=out)


def _roofline(nbytes, seconds, kernel, unit_note):
    peak, kind = _peaks()
    achieved = nbytes / seconds / 1e9
    return {"bound": "hbm", "kernel": kernel, "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "peak_kind": kind + " (burst copy)", "frac": round(achieved / peak, 4),
            "bytes_per_launch": int(nbytes), "avg_launch_us": round(seconds * 1e6, 3), "per": unit_note}


class SingleLayer:
    """One MoE layer for one token: 64 NVFP4 experts (H=2560, I=640), top-10,
    x ~ N(0,1) BF16, W_r ~ N(0,0.02).  One call = moe_decode_layer from x
    (router + expert pass in one launch); a fresh token per call and the L2
    flushed between calls."""

    WORKLOAD, NE = 0, 64

    def __init__(self, torch, moe, synth, device, calls):
        self.torch, self.moe = torch, moe
        self.s = moe.shape(H, I, moe.FMT_NVFP4)
        self.rb = moe.moe_expert_record_bytes(self.s)
        self.pool = torch.empty(self.NE, self.rb, dtype=torch.uint8, device=device)
        for e in range(self.NE):
            g, up, d = synth.expert_weights(H, I, synth.expert_seed(self.WORKLOAD, 0, e), device=device)
            moe.fp4_pack_expert(g, up, d, self.s, record=self.pool[e])
        self.ptrs = moe.pointer_table([self.pool[e] for e in range(self.NE)])
        self.wr = synth.router_weights(self.NE, H, synth.seed_of(self.WORKLOAD, 0, synth.T_ROUTER), device=device)
        self.xs = torch.cat([synth.activations(1, H, synth.seed_of(self.WORKLOAD, 100 + c, synth.T_X), device=device)
                             for c in range(calls)])
        self.idx = torch.empty(1, K_TOP, dtype=torch.int32, device=device)
        self.w = torch.empty(1, K_TOP, dtype=torch.float32, device=device)
        self.logits = torch.empty(1, self.NE, dtype=torch.float32, device=device)
        self.y = torch.empty(1, H, dtype=torch.float32, device=device)
        self.ws = torch.zeros(moe.moe_experts_decode_workspace(1, K_TOP, self.s), dtype=torch.uint8, device=device)
        self.st = torch.zeros(1, dtype=torch.int32, device=device)
        self.flush = _l2_flusher(torch, device)

    def call(self, c):
        self.moe.moe_decode_layer(self.wr, None, K_TOP, self.ptrs, self.s, x=self.xs[c:c + 1], idx=self.idx,
                                  weights=self.w, logits=self.logits, y=self.y, workspace=self.ws, dev_status=self.st)

    def measure(self, calls, warm):
        torch = self.torch
        for c in range(warm):
            self.call(c % self.xs.shape[0])
        torch.cuda.synchronize()
        tot = 0.0
        for c in range(calls):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            self.flush()
            _gpu_spacer(torch)
            a.record()
            self.call(c % self.xs.shape[0])
            b.record()
            torch.cuda.synchronize()
            tot += a.elapsed_time(b)
        sec = tot / calls / 1e3
        exp_bytes = K_TOP * self.rb
        nbytes = exp_bytes + self.NE * H * 2 + H * 2 + H * 4 + 2 * K_TOP * I * 4 + 2 * self.NE * 4
        return {"workload": "one MoE layer, one token: 64 NVFP4 experts (H=2560, I=640), top-10",
                "value": round(exp_bytes / sec / 1e9, 2), "unit": "GB/s", "us_per_layer": round(sec * 1e6, 3),
                "calls": calls, "l2": "flushed between calls (512 MB read sweep)",
                "dev_status": int(self.st.item()),
                "roofline": _roofline(nbytes, sec, "moe_decode_layer: oneshot_kernel", "one layer launch")}


class DeepSeekCalls:
    """DeepSeek-shaped layer: H=4096, I=2880, MXFP4 records of 18,800,640 B,
    384 experts, top-6; one weight set reused for 40 sequential calls, each
    with its own seeded router weights and token; L2 flushed between calls.
    One call = moe_router_topk + moe_experts_decode (the shape's per-SM share
    is larger than shared memory, so the expert pass is the ring kernel)."""

    WORKLOAD, NE, HD, ID, KD, CALLS = 3, 384, 4096, 2880, 6, 40

    def __init__(self, torch, moe, synth, device):
        self.torch, self.moe = torch, moe
        self.s = moe.shape(self.HD, self.ID, moe.FMT_MXFP4)
        self.rb = moe.moe_expert_record_bytes(self.s)
        self.pool = torch.empty(self.NE, self.rb, dtype=torch.uint8, device=device)
        for e in range(self.NE):
            g, up, d = synth.expert_weights(self.HD, self.ID, synth.expert_seed(self.WORKLOAD, 0, e), device=device)
            moe.fp4_pack_expert(g, up, d, self.s, record=self.pool[e])
        self.ptrs = moe.pointer_table([self.pool[e] for e in range(self.NE)])
        self.wr = [synth.router_weights(self.NE, self.HD, synth.seed_of(self.WORKLOAD, c, synth.T_ROUTER),
                                        device=device) for c in range(self.CALLS)]
        self.xs = [synth.activations(1, self.HD, synth.seed_of(self.WORKLOAD, c, synth.T_X), device=device)
                   for c in range(self.CALLS)]
        self.idx = torch.empty(1, self.KD, dtype=torch.int32, device=device)
        self.w = torch.empty(1, self.KD, dtype=torch.float32, device=device)
        self.logits = torch.empty(1, self.NE, dtype=torch.float32, device=device)
        self.y = torch.empty(1, self.HD, dtype=torch.float32, device=device)
        self.ws = torch.zeros(moe.moe_experts_decode_workspace(1, self.KD, self.s), dtype=torch.uint8, device=device)
        self.st = torch.zeros(1, dtype=torch.int32, device=device)
        self.flush = _l2_flusher(torch, device)

    def router(self, c):
        self.moe.moe_router_topk(self.xs[c], self.wr[c], None, self.KD, self.idx, self.w, self.logits)

    def experts(self, c):
        self.moe.moe_experts_decode(self.xs[c], self.idx, self.w, self.ptrs, self.s, self.y, self.ws, self.st)

    def measure(self, warm):
        torch = self.torch
        for c in range(warm):
            self.router(c % self.CALLS)
            self.experts(c % self.CALLS)
        torch.cuda.synchronize()
        tot, tot_exp = 0.0, 0.0
        for c in range(self.CALLS):
            a, b, d = (torch.cuda.Event(enable_timing=True) for _ in range(3))
            self.flush()
            _gpu_spacer(torch)
            a.record()
            self.router(c)
            b.record()
            self.experts(c)
            d.record()
            torch.cuda.synchronize()
            tot += a.elapsed_time(d)
            tot_exp += b.elapsed_time(d)
        sec, sec_exp = tot / self.CALLS / 1e3, tot_exp / self.CALLS / 1e3
        exp_bytes = self.KD * self.rb
        nbytes = exp_bytes + self.HD * 2 + self.HD * 4 + self.KD * self.ID * 4 * 2
        return {"workload": "DeepSeek-shaped layer: 384 MXFP4 experts (H=4096, I=2880, 18,800,640 B), top-6, "
                            "40 seeded calls on one weight set",
                "value": round(exp_bytes / sec / 1e9, 2), "unit": "GB/s", "us_per_call": round(sec * 1e6, 3),
                "us_expert_pass": round(sec_exp * 1e6, 3), "us_per_40_calls": round(40 * sec * 1e6, 1),
                "expert_bytes_per_call": exp_bytes, "l2": "flushed between calls (512 MB read sweep)",
                "dev_status": int(self.st.item()),
                "roofline": _roofline(nbytes, sec_exp, "moe_experts_decode: stream_kernel (TMA ring)",
                                      "one expert-pass launch")}


class BatchedStack:
    """32 tokens through the 48-layer stack of the decode pool (config of the
    decode stack, 512 experts per layer, top-10): per layer the router (layer
    0 from x, later layers RMS-chained from the previous output) and the
    expert pass for all 32 tokens; one step = 48 layers, captured in a CUDA
    graph.  Unique expert bytes per layer are counted from the routing."""

    T = 32

    def __init__(self, torch, moe, synth, stack, device, steps_total):
        self.torch, self.moe, self.st_ = torch, moe, stack
        T = self.T
        self.x0 = [synth.activations(T, H, synth.seed_of(4, 100 + s, synth.T_X), device=device)
                   for s in range(steps_total)]
        self.x = torch.empty(T, H, dtype=torch.bfloat16, device=device)
        self.idx = torch.empty(LAYERS, T, K_TOP, dtype=torch.int32, device=device)
        self.w = torch.empty(T, K_TOP, dtype=torch.float32, device=device)
        self.logits = torch.empty(T, E, dtype=torch.float32, device=device)
        self.y = torch.empty(T, H, dtype=torch.float32, device=device)
        self.ws = torch.zeros(moe.moe_experts_decode_workspace(T, K_TOP, stack.s), dtype=torch.uint8, device=device)
        self.st = torch.zeros(1, dtype=torch.int32, device=device)

    def run_layers(self):
        moe, st = self.moe, self.st_
        for L in range(LAYERS):
            if L == 0:
                moe.moe_router_topk(self.x, st.wr[L], None, K_TOP, self.idx[L], self.w, self.logits)
            else:
                moe.moe_rmsnorm_router_topk(self.y, st.wr[L], None, K_TOP, 1e-6, self.x, self.idx[L], self.w,
                                            self.logits)
            moe.moe_experts_decode(self.x, self.idx[L], self.w, st.ptrs[L], st.s, self.y, self.ws, self.st)

    def measure(self, steps, warm):
        torch = self.torch
        self.x.copy_(self.x0[0])
        self.run_layers()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            self.run_layers()
        for s in range(warm):
            self.x.copy_(self.x0[s % len(self.x0)])
            g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        uniq = 0
        a.record()
        for s in range(steps):
            self.x.copy_(self.x0[(warm + s) % len(self.x0)])
            g.replay()
        b.record()
        torch.cuda.synchronize()
        sec = a.elapsed_time(b) / steps / 1e3
        # unique records of the last step's 48 layers (the routing of every step is of the same kind)
        for L in range(LAYERS):
            uniq += int(torch.unique(self.idx[L]).numel())
        exp_bytes = uniq * self.st_.rec_bytes
        del g
        nbytes = exp_bytes + LAYERS * (E * H * 2 + self.T * H * (2 + 4 + 4) + 2 * self.T * K_TOP * I * 4)
        return {"workload": "batched decode: 32 tokens x 48 layers x 512 NVFP4 experts, top-10",
                "value": round(self.T / sec, 1), "unit": "tokens/s", "ms_per_step": round(sec * 1e3, 4),
                "unique_experts_per_layer": round(uniq / LAYERS, 1), "expert_bytes_per_step": exp_bytes,
                "expert_gbs": round(exp_bytes / sec / 1e9, 1),
                "l2": "inputs larger than L2 (~0.66 GB of distinct records per layer)",
                # per layer: RMS chaining (layers 1-47), logits, top-k, the ring kernel's expert pass
                "launches_per_step": LAYERS * 4 - 1, "dev_status": int(self.st.item()),
                "roofline": _roofline(nbytes, sec, "whole step (router kernels + ring-kernel expert pass), "
                                      "unique-record bytes", "one 48-layer step")}


def measure_host_tier(torch, moe, synth, device, calls: int = 40):
    """The host-memory expert tier: 64 NVFP4 experts (177 MB) in pinned host
    memory, one token top-10 per call through moe_experts_decode_host (plain
    loads over the device's address space: NVLink-C2C on a Grace machine);
    the same records in HBM through the same call for comparison.  A fresh
    token per call, L2 flushed between calls."""
    s = moe.shape(H, I, moe.FMT_NVFP4)
    rb = moe.moe_expert_record_bytes(s)
    NE = 64
    dev_pool = torch.empty(NE, rb, dtype=torch.uint8, device=device)
    for e in range(NE):
        g, up, d = synth.expert_weights(H, I, synth.expert_seed(0, 0, e), device=device)
        moe.fp4_pack_expert(g, up, d, s, record=dev_pool[e])
    host_pool = torch.empty(NE, rb, dtype=torch.uint8, pin_memory=True)
    host_pool.copy_(dev_pool)
    torch.cuda.synchronize()
    tables = {"host": torch.tensor([host_pool[e].data_ptr() for e in range(NE)], dtype=torch.int64, device=device),
              "hbm": moe.pointer_table([dev_pool[e] for e in range(NE)])}
    wr = synth.router_weights(NE, H, synth.seed_of(0, 0, synth.T_ROUTER), device=device)
    flush = _l2_flusher(torch, device)
    ws = torch.zeros(moe.moe_experts_decode_workspace(1, K_TOP, s), dtype=torch.uint8, device=device)
    y = torch.empty(1, H, dtype=torch.float32, device=device)
    out = {}
    for name, ptrs in tables.items():
        tot = 0.0
        for c in range(calls + 3):
            x = synth.activations(1, H, synth.seed_of(0, 300 + c, synth.T_X), device=device)
            idx, w, _ = moe.moe_router_topk(x, wr, None, K_TOP)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            flush()
            _gpu_spacer(torch)
            a.record()
            moe.moe_experts_decode_host(x, idx, w, ptrs, s, y, ws)
            b.record()
            torch.cuda.synchronize()
            if c >= 3:
                tot += a.elapsed_time(b)
        sec = tot / calls / 1e3
        out[name] = {"us_per_call": round(sec * 1e6, 2), "expert_gbs": round(K_TOP * rb / sec / 1e9, 1)}
    del host_pool
    return {"workload": "one token, top-10 of 64 NVFP4 experts (H=2560, I=640); records in pinned host memory vs HBM",
            "entry": "moe_experts_decode_host (two kernels, plain 16-byte loads)", **out}


def measure_fp8_gemv(torch, moe, synth, device, reps: int = 20):
    """FP8 row-scaled GEMV on the two proposed shapes; GB/s of W + x + y per
    call: single calls with the L2 flushed before each, and back-to-back calls
    on distinct matrices (more bytes than the L2 holds) replayed from a CUDA
    graph, as a model's consecutive matrices would run."""
    out = {}
    flush = torch.ones(512 << 18, dtype=torch.int32, device=device)   # read sweep evicts the L2
    flush_out = torch.zeros((), dtype=torch.int64, device=device)
    for M, K in ((8192, 2560), (2560, 4096)):
        # enough distinct matrices that consecutive calls never share L2 lines
        n = max(16, (256 << 20) // (M * K) + 1)
        ws = [synth.expert_matrix((M, K), seed=M + K + i, device=device).to(torch.float8_e4m3fn)
              .view(torch.uint8) for i in range(n)]
        s = synth.uniform((M,), seed=M, lo=0.5, hi=2.0, device=device)
        x = synth.activations(1, K, seed=K, device=device)[0]
        y = torch.empty(M, dtype=torch.float32, device=device)
        for i in range(3):
            moe.fp8_rowscale_gemv(ws[i % n], s, x, y)
        tot = 0.0
        for i in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.sum(flush, 0, out=flush_out)
            _gpu_spacer(torch)
            a.record()
            moe.fp8_rowscale_gemv(ws[i % n], s, x, y)
            b.record()
            torch.cuda.synchronize()
            tot += a.elapsed_time(b)
        us = tot / reps * 1e3
        nbytes = M * K + M * 4 + K * 2 + M * 4
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(n):
                moe.fp8_rowscale_gemv(ws[i], s, x, y)
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        _gpu_spacer(torch)
        a.record()
        for _ in range(5):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        gus = a.elapsed_time(b) / (5 * n) * 1e3
        out[f"{M}x{K}"] = {"us": round(us, 2), "gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                           "graph_us": round(gus, 2), "graph_gbs": round(nbytes / (gus * 1e-6) / 1e9, 1),
                           "graph_launches": n}
        del g, ws
    return out


def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """The largest value over all ranks (the slowest rank's time)."""
    import torch
    if dist is None or not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# the sources the one-shot decode kernel is compiled from: a DRAM capture
# stays valid while these files are unchanged
ONESHOT_SOURCES = ("common.cuh", "decode_math.cuh", "decode_oneshot.cu", "decode_oneshot.h", "router_math.cuh",
                   "tcgen05.cuh")


def _hash_sources(names=ONESHOT_SOURCES):
    h = hashlib.sha256()
    d = os.path.join(ROOT, "block_scaled_fp4_softmax_gb300", "csrc")
    for n in sorted(names):
        with open(os.path.join(d, n), "rb") as f:
            h.update(n.encode() + f.read())
    return h.hexdigest()[:16]


def _traffic_from_profiles(kernel_key: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current sources of the kernel (the files of ONESHOT_SOURCES)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        ent = d.get(kernel_key)
        if ent and ent.get("sources") == _hash_sources():
            return ent["bytes_per_launch"]
    except Exception:
        pass
    return None


def run_ours(args):
    import torch
    import torch.distributed as dist

    from block_scaled_fp4_softmax_gb300 import build, moe, synth

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    moe.load()

    steps, warm = args.steps, args.warmup
    wl = DecodeStack(torch, moe, synth, dev, rank, steps + warm)
    graph, _ = wl.capture(with_events=False)
    stream = torch.cuda.current_stream()

    def one_step(s):
        wl.x.copy_(wl.x0[s:s + 1])
        graph.replay()

    for s in range(warm):
        one_step(s)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    sampler = ClockSampler(local)
    sampler.start()
    # the clock sampler polls every 200 ms: run the same step back to back for
    # 1.5 s right before the timed region, so the clocks it records (over that
    # run and the timed region) are those of this workload under load
    t_soak = time.time()
    n_soak = 0
    while time.time() - t_soak < 1.5:
        for _ in range(50):
            one_step(n_soak % (steps + warm))
            n_soak += 1
        torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_start.record(stream)
    for s in range(steps):
        one_step(warm + s)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if clocks is not None:
        clocks["window"] = "a 1.5 s back-to-back run of the same step right before the timed region, and the region"
    ms = t_start.elapsed_time(t_end) / steps
    if world > 1:
        ms = max_over_ranks(ms, dist, dev)
        dist.barrier()
    st = int(wl.st.item())

    # the same steps through the persistent 48-layer kernel (one launch per
    # token), timed the same way: A/B against the per-layer launches
    persistent = None
    try:
        for s_ in range(warm):
            wl.x.copy_(wl.x0[s_:s_ + 1])
            wl.run_stack_kernel()
        torch.cuda.synchronize()
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record(stream)
        for s_ in range(steps):
            wl.x.copy_(wl.x0[warm + s_:warm + s_ + 1])
            wl.run_stack_kernel()
        p1.record(stream)
        torch.cuda.synchronize()
        pms = p0.elapsed_time(p1) / steps
        persistent = {"entry": "moe_decode_stack (one persistent launch per 48-layer step)",
                      "ms_per_step": round(pms, 4),
                      "value": round(wl.expert_bytes_per_step() / (pms / 1e3) / 1e9, 2), "unit": "GB/s",
                      "vs_per_layer_launches": round(ms / pms, 4), "dev_status": int(wl.st.item())}
    except Exception as exc:  # report, do not hide
        persistent = {"error": repr(exc)[:300]}

    # dominant kernel (the expert pass) timed with events inside the graph
    kern_ms = None
    try:
        g2, ev = wl.capture(with_events=True)
        samples = []
        for s in range(steps):
            wl.x.copy_(wl.x0[(warm + s) % (steps + warm):(warm + s) % (steps + warm) + 1])
            g2.replay()
            torch.cuda.synchronize()
            samples += [a.elapsed_time(b) for a, b in ev]
        kern_ms = statistics.mean(samples)
        del g2
    except Exception as exc:  # events inside graphs unsupported: time eagerly
        print(f"# graph events unavailable ({exc}); timing the expert pass eagerly", file=sys.stderr)
        samples = []
        flush = torch.ones(256 << 18, dtype=torch.int32, device=dev)
        flush_out = torch.zeros((), dtype=torch.int64, device=dev)
        for s in range(steps):
            L = s % LAYERS
            torch.sum(flush, 0, out=flush_out)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            moe.moe_experts_decode(wl.x, wl.idx, wl.w, wl.ptrs[L], wl.s, wl.y, wl.ws, wl.st)
            b.record()
            torch.cuda.synchronize()
            samples.append(a.elapsed_time(b))
        kern_ms = statistics.mean(samples)

    # end to end through the library's API with host buffers: every step
    # copies the token in from pinned host memory, runs the 48 layers and
    # copies the output back, timed on the host clock.  Two ways a caller
    # drives the layers: the 48 moe_decode_layer calls captured once in a CUDA
    # graph through the Python binding and replayed per token (the figure
    # reported), and the same calls made eagerly (kept beside it).
    e2e = None
    if not args.no_e2e:
        x_host = wl.x0.cpu().pin_memory()
        y_host = torch.empty(1, H, dtype=torch.float32).pin_memory()
        e_steps = max(3, min(steps, 20))

        def e2e_wall(run):
            for s in range(2):
                wl.x.copy_(x_host[s:s + 1], non_blocking=True)
                run()
                y_host.copy_(wl.y, non_blocking=True)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            for s in range(e_steps):
                wl.x.copy_(x_host[s % x_host.shape[0]:s % x_host.shape[0] + 1], non_blocking=True)
                run()
                y_host.copy_(wl.y, non_blocking=True)
            torch.cuda.synchronize()
            return (time.perf_counter() - t0) / e_steps

        wall_eager = e2e_wall(wl.run_layers)
        wall = e2e_wall(graph.replay)
        e2e = {"value": round(wl.expert_bytes_per_step() / wall / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": H * 2, "d2h_bytes_per_step": H * 4,
               "ms_per_step": round(wall * 1e3, 4),
               "api": "48 moe_decode_layer calls captured once in a CUDA graph through the binding, replayed per token",
               "eager": {"value": round(wl.expert_bytes_per_step() / wall_eager / 1e9, 2), "unit": "GB/s",
                         "ms_per_step": round(wall_eager * 1e3, 4), "api": "the same 48 calls made eagerly"}}

    spec = None
    if not args.no_others:
        try:
            spec = speculative_routing(torch, moe, wl)
        except Exception as exc:  # report, do not hide
            spec = {"error": repr(exc)[:300]}

    # the other workloads, one key each
    others = {}
    if not args.no_others:
        jobs = (("config4", lambda: BatchedStack(torch, moe, synth, wl, dev, 8).measure(max(3, min(steps, 10)), 3)),
                ("host_tier", lambda: measure_host_tier(torch, moe, synth, dev)),
                ("config0", lambda: SingleLayer(torch, moe, synth, dev, 64).measure(max(20, min(steps, 200)), 5)),
                ("config3", lambda: DeepSeekCalls(torch, moe, synth, dev).measure(5)))
        for key, job in jobs:
            try:
                others[key] = job()
            except Exception as exc:  # report, do not hide
                others[key] = {"error": repr(exc)[:300]}
            torch.cuda.empty_cache()

    prompt = None
    if not args.no_prompt:
        del wl.slots
        torch.cuda.empty_cache()
        try:
            pl = PromptLayer(torch, moe, synth, dev)
            prompt = pl.measure(max(3, min(steps, 20)), 3)
            del pl
        except Exception as exc:  # report, do not hide
            prompt = {"error": repr(exc)[:300]}

    fp8 = None
    if not args.no_prompt:
        try:
            fp8 = measure_fp8_gemv(torch, moe, synth, dev)
        except Exception as exc:
            fp8 = {"error": repr(exc)[:300]}


    peak, peak_kind = _peaks()
    value = wl.expert_bytes_per_step() * world / (ms / 1e3) / 1e9
    # one launch reads its 10 expert records and the router rows (W_r, E x H
    # BF16), reads y_prev and writes x and y, writes and reads h and the logits
    per_launch_bytes = (K_TOP * wl.rec_bytes + E * H * 2 + H * 4 + H * 2 + H * 4 + K_TOP * I * 4 * 2
                        + E * 4 * 2)
    achieved = per_launch_bytes / (kern_ms / 1e3) / 1e9
    out = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": warm,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e2m1+e4m3 weights, bf16 activations, f32 accumulate",
        "data": "synthetic (seeded N(0,0.02) FP32 experts packed to NVFP4 on device; "
                "1024 distinct experts copied into 24,576 physical slots)",
        "config": {"workload": "qwen_decode_stack: 48 layers x 512 NVFP4 experts "
                               "(H=2560, I=640, 2,764,800 B each, 68 GB resident), top-10, 1 token/step, "
                               "RMS-chained layers",
                   "tokens_per_step": 1, "layers": LAYERS, "experts": E, "top_k": K_TOP,
                   "expert_bytes_per_step": wl.expert_bytes_per_step(),
                   "l2": "inputs larger than L2: 1.33 GB of distinct expert records per step",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "launch": "CUDA graph, 1 kernel per layer (moe_decode_layer: RMS chaining, router logits and top-k, then the one-shot expert pass, in one launch), programmatic dependent launch"},
        "tokens_per_s": round(world * 1e3 / ms, 2),
        "hbm_frac": {"of_measured": round(value / world / peak, 4), "measured_gbs": peak,
                     "of_nominal_8000": round(value / world / 8000.0, 4)},
        "roofline": {"bound": "hbm", "kernel": "moe_decode_layer: oneshot_kernel (router logits + top-k, grid barrier, TMA bulk copies, gate/up, grid barrier, down)",
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "peak_kind": peak_kind + " (burst copy)",
                     "frac": round(achieved / peak, 4),
                     "bytes_per_launch": per_launch_bytes, "avg_launch_us": round(kern_ms * 1e3, 3),
                     "traffic": _traffic_from_profiles("moe_decode_layer")},
        "gpu_launches": wl.kernels_per_step * steps,
        "clocks": clocks,
        "e2e": e2e,
        "prompt": prompt,
        "fp8_gemv": fp8,
        "speculative_routing": spec,
        "persistent_stack": persistent,
        "dev_status": st,
        "setup_s": round(wl.setup_s, 1),
    }
    out.update(others)
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
        # the oracle on a bounded sample of each other workload, in that
        # workload's unit
        for key, fn in (("config0", cpu_baseline_config0), ("config3", cpu_baseline_config3),
                        ("config4", cpu_baseline_config4), ("prompt", cpu_baseline_prompt)):
            if isinstance(out.get(key), dict) and "error" not in out[key]:
                try:
                    out[key]["cpu_baseline"] = fn(args.cpu_seconds_other)
                except Exception as exc:  # report, do not hide
                    out[key]["cpu_baseline"] = {"error": repr(exc)[:300]}
    if world > 1:
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(out), flush=True)


# ---------------------------------------------------------------------------
# the oracle on the host cores
# ---------------------------------------------------------------------------
def _pack_one(u):
    from block_scaled_fp4_softmax_gb300 import synth
    from oracle import oracle as O
    g, up, d = synth.expert_weights(H, I, synth.expert_seed(WORKLOAD_ID, 0, int(u)))
    return O.pack_expert(g.numpy(), up.numpy(), d.numpy(), O.FMT_NVFP4)


def _oracle_sample(budget_s: float, max_layers: int = LAYERS):
    """Run the oracle through the decode stack for one token until the time
    budget is used; returns (expert bytes processed, seconds, layers).  The
    records are inputs: the oracle packs them itself, in spawned worker
    processes, outside the timed part."""
    import concurrent.futures as cf
    import multiprocessing as mp

    import torch

    from block_scaled_fp4_softmax_gb300 import synth
    from oracle import oracle as O

    def bits(t):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)

    rec_bytes = O.record_bytes(H, I, O.FMT_NVFP4)
    x = bits(synth.activations(1, H, synth.seed_of(WORKLOAD_ID, 100, synth.T_X)))
    done_bytes, busy, layers = 0, 0.0, 0
    with cf.ProcessPoolExecutor(max_workers=min(K_TOP, os.cpu_count() or 2),
                                mp_context=mp.get_context("spawn")) as ex:
        for L in range(max_layers):
            wr = bits(synth.router_weights(E, H, synth.seed_of(WORKLOAD_ID, L, synth.T_ROUTER)))
            rng = np.random.default_rng(synth.seed_of(WORKLOAD_ID, L, synth.T_PERM))
            choice = rng.permutation(UNIQUE_EXPERTS)[:E]
            t0 = time.perf_counter()
            idx, w = O.topk_softmax(O.router_logits(x, wr), K_TOP)
            busy += time.perf_counter() - t0
            sel = [int(e) for e in idx.ravel()]
            recs = dict(zip(sel, ex.map(_pack_one, [int(choice[e]) for e in sel])))
            t0 = time.perf_counter()
            y = O.moe_layer_decode(x, idx, w, recs, H, I, O.FMT_NVFP4)
            x = O.rmsnorm_bf16(y, 1e-6)
            busy += time.perf_counter() - t0
            done_bytes += K_TOP * rec_bytes
            layers += 1
            if busy >= budget_s:
                break
    return done_bytes, busy, layers


def _cores():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        n = max((i.get("num_threads", 1) for i in info), default=1)
        return int(n)
    except Exception:
        return os.cpu_count() or 1


def _spawn_pool(n):
    import concurrent.futures as cf
    import multiprocessing as mp
    return cf.ProcessPoolExecutor(max_workers=min(n, os.cpu_count() or 2), mp_context=mp.get_context("spawn"))


def _pack_seeded(args):
    """Oracle packing of one seeded expert (spawned worker; untimed)."""
    h, i, fmt, seed = args
    from block_scaled_fp4_softmax_gb300 import synth
    from oracle import oracle as O
    g, up, d = synth.expert_weights(h, i, seed)
    return O.pack_expert(g.numpy(), up.numpy(), d.numpy(), fmt)


def _bits_np(t):
    import torch
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def cpu_baseline_config0(budget_s: float):
    """The oracle on the one-layer workload: router over 64 experts + 10
    experts for one token, per call; records packed outside the timed part."""
    from block_scaled_fp4_softmax_gb300 import synth
    from oracle import oracle as O
    wr = _bits_np(synth.router_weights(64, H, synth.seed_of(0, 0, synth.T_ROUTER)))
    busy, calls, recs = 0.0, 0, {}
    with _spawn_pool(K_TOP) as ex:
        while busy < budget_s and calls < 64:
            x = _bits_np(synth.activations(1, H, synth.seed_of(0, 100 + calls, synth.T_X)))
            t0 = time.perf_counter()
            idx, w = O.topk_softmax(O.router_logits(x, wr), K_TOP)
            busy += time.perf_counter() - t0
            need = [int(e) for e in idx.ravel() if int(e) not in recs]
            for e, r in zip(need, ex.map(_pack_seeded, [(H, I, O.FMT_NVFP4, synth.expert_seed(0, 0, e)) for e in need])):
                recs[e] = r
            t0 = time.perf_counter()
            O.moe_layer_decode(x, idx, w, recs, H, I, O.FMT_NVFP4)
            busy += time.perf_counter() - t0
            calls += 1
    rb = O.record_bytes(H, I, O.FMT_NVFP4)
    return {"value": round(calls * K_TOP * rb / busy / 1e9, 4), "unit": "GB/s", "cores": _cores(), "kind": "oracle",
            "sample": f"{calls} one-token layer calls (router over 64 experts + 10 experts), float64 numpy; "
                      "record packing untimed", "seconds": round(busy, 2)}


def cpu_baseline_config3(budget_s: float):
    """The oracle on the DeepSeek-shaped calls: router over 384 experts + 6
    MXFP4 experts per call; records packed outside the timed part."""
    from block_scaled_fp4_softmax_gb300 import synth
    from oracle import oracle as O
    HD, ID, NE, KD = 4096, 2880, 384, 6
    busy, calls = 0.0, 0
    with _spawn_pool(KD) as ex:
        while busy < budget_s and calls < 40:
            wr = _bits_np(synth.router_weights(NE, HD, synth.seed_of(3, calls, synth.T_ROUTER)))
            x = _bits_np(synth.activations(1, HD, synth.seed_of(3, calls, synth.T_X)))
            t0 = time.perf_counter()
            idx, w = O.topk_softmax(O.router_logits(x, wr), KD)
            busy += time.perf_counter() - t0
            sel = [int(e) for e in idx.ravel()]
            recs = dict(zip(sel, ex.map(_pack_seeded, [(HD, ID, O.FMT_MXFP4, synth.expert_seed(3, 0, e)) for e in sel])))
            t0 = time.perf_counter()
            O.moe_layer_decode(x, idx, w, recs, HD, ID, O.FMT_MXFP4)
            busy += time.perf_counter() - t0
            calls += 1
    rb = O.record_bytes(HD, ID, O.FMT_MXFP4)
    return {"value": round(calls * KD * rb / busy / 1e9, 4), "unit": "GB/s", "cores": _cores(), "kind": "oracle",
            "sample": f"{calls} of the 40 DeepSeek-shaped calls (router over 384 + 6 MXFP4 experts), float64 numpy; "
                      "record packing untimed", "seconds": round(busy, 2)}


def cpu_baseline_config4(budget_s: float):
    """The oracle on the batched stack: tokens of layer 0 of a 32-token batch,
    one at a time (router + 10 experts each), until the budget is used; the
    unit is tokens per second through one layer, divided by the 48 layers."""
    from block_scaled_fp4_softmax_gb300 import synth
    from oracle import oracle as O
    wr = _bits_np(synth.router_weights(E, H, synth.seed_of(WORKLOAD_ID, 0, synth.T_ROUTER)))
    rng = np.random.default_rng(synth.seed_of(WORKLOAD_ID, 0, synth.T_PERM))
    choice = rng.permutation(UNIQUE_EXPERTS)[:E]
    xs = _bits_np(synth.activations(32, H, synth.seed_of(4, 100, synth.T_X)))
    busy, done = 0.0, 0
    with _spawn_pool(K_TOP) as ex:
        while busy < budget_s and done < 32:
            x = xs[done:done + 1]
            t0 = time.perf_counter()
            idx, w = O.topk_softmax(O.router_logits(x, wr), K_TOP)
            busy += time.perf_counter() - t0
            sel = [int(e) for e in idx.ravel()]
            recs = dict(zip(sel, ex.map(_pack_seeded, [(H, I, O.FMT_NVFP4, synth.expert_seed(WORKLOAD_ID, 0, int(choice[e])))
                                                       for e in sel])))
            t0 = time.perf_counter()
            O.moe_layer_decode(x, idx, w, recs, H, I, O.FMT_NVFP4)
            busy += time.perf_counter() - t0
            done += 1
    return {"value": round(done / busy / LAYERS, 5), "unit": "tokens/s", "cores": _cores(), "kind": "oracle",
            "sample": f"{done} tokens of one layer of the 32-token batch (router + 10 experts each), float64 numpy, "
                      "rate divided by 48 layers; record packing untimed", "seconds": round(busy, 2)}


def cpu_baseline_prompt(budget_s: float):
    """The oracle on the prompt layer: its expert-by-expert form on a sample
    of the hit experts (each with all of its tokens), scaled to all hit
    experts, plus the router logits of a token sample scaled to 2451 tokens."""
    import torch
    from block_scaled_fp4_softmax_gb300 import synth
    from oracle import oracle as O
    T = PromptLayer.T
    x = _bits_np(synth.activations(T, H, synth.seed_of(2, 0, synth.T_X)))
    wr = _bits_np(synth.router_weights(E, H, synth.seed_of(2, 0, synth.T_ROUTER)))
    bias = synth.zipf_bias(E, synth.seed_of(2, 0, synth.T_BIAS)).numpy()
    # routing of all tokens (untimed; the logits are timed on a sample below)
    lg = (O.bf16_bits_to_f32(x).astype(np.float64) @ O.bf16_bits_to_f32(wr).astype(np.float64).T) + bias
    idx = np.argsort(-lg, axis=1, kind="stable")[:, :K_TOP].astype(np.int32)
    w = np.full(idx.shape, 1.0 / K_TOP)
    hit = np.unique(idx)
    rng = np.random.default_rng(5)
    t0 = time.perf_counter()
    O.router_logits(x[:64], wr, bias)
    t_router = (time.perf_counter() - t0) * T / 64
    busy, n = 0.0, 0
    order = rng.permutation(hit)
    with _spawn_pool(8) as ex:
        while busy < budget_s and n < len(order):
            batch = [int(e) for e in order[n:n + 4]]
            recs = dict(zip(batch, ex.map(_pack_seeded, [(H, I, O.FMT_NVFP4, synth.expert_seed(2, 0, e)) for e in batch])))
            for e in batch:
                toks = np.nonzero((idx == e).any(axis=1))[0]
                idx_e = np.full((len(toks), 1), e, dtype=np.int32)
                w_e = np.full((len(toks), 1), 1.0 / K_TOP)
                t0 = time.perf_counter()
                O.moe_layer_grouped_by_expert(x[toks], idx_e, w_e, recs, H, I, O.FMT_NVFP4)
                busy += time.perf_counter() - t0
                n += 1
    est = t_router + busy * len(hit) / n
    return {"value": round(T / est, 2), "unit": "tokens/s", "cores": _cores(), "kind": "oracle",
            "sample": f"{n} of {len(hit)} hit experts (each with all its tokens) through the oracle's "
                      "expert-by-expert form, scaled to all hit experts, plus router logits of 64 tokens "
                      "scaled to 2451; float64 numpy; record packing untimed",
            "seconds": round(busy, 2)}


def _oracle_sample_one_thread(budget_s: float):
    """The same bounded sample with the oracle's BLAS limited to one thread
    (a fresh interpreter, so the limit is in place before numpy loads)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json, sys; sys.path.insert(0, %r); import bench; "
            "print(json.dumps(bench._oracle_sample(%r)))" % (ROOT, float(budget_s)))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
    nbytes, secs, layers = json.loads(r.stdout.strip().splitlines()[-1])
    return nbytes, secs, layers


def cpu_baseline(budget_s: float):
    nbytes, secs, layers = _oracle_sample(budget_s)
    out = {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": _cores(),
           "kind": "oracle",
           "sample": f"{layers} layers of the decode stack for 1 token (router + 10 experts + "
                     f"RMS chaining per layer), float64 numpy; record packing untimed",
           "seconds": round(secs, 2)}
    try:
        n1, s1, l1 = _oracle_sample_one_thread(budget_s / 2)
        out["one_thread"] = {"value": round(n1 / s1 / 1e9, 4), "cores": 1, "layers": l1, "seconds": round(s1, 2)}
    except Exception as exc:  # report, do not hide
        out["one_thread"] = {"error": repr(exc)[:200]}
    return out


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    steps, warm = args.steps, args.warmup
    per_step_budget = max(0.5, args.cpu_seconds / max(1, steps))
    for _ in range(min(warm, 1)):
        _oracle_sample(0.0, max_layers=1)
    t_bytes, t_secs, t_layers = 0, 0.0, 0
    for _ in range(steps):
        b, s, l = _oracle_sample(per_step_budget, max_layers=2)
        t_bytes += b
        t_secs += s
        t_layers += l
    value = t_bytes / t_secs / 1e9
    cores = _cores()
    sample = (f"{t_layers} layers over {steps} steps of the decode stack for 1 token, "
              f"float64 numpy oracle")
    out = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
           "steps": steps, "warmup": warm, "ms_per_step": round(t_secs / steps * 1e3, 2),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "impl": "reference",
           "config": {"workload": "qwen_decode_stack (bounded sample on host cores)"},
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "kind": "oracle",
                            "cores": cores, "sample": sample},
           "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_profile_case(args):
    """A small case of one kernel family for ncu: one decode layer (a 512-expert
    router over a 64-record pool, 177 MB of records, larger than L2), one
    DeepSeek-shaped call, one 32-token batched-decode call over a 64-record
    pool, FP8 GEMVs on distinct matrices, or the prompt layer."""
    import torch

    from block_scaled_fp4_softmax_gb300 import build, moe, synth

    build.build()
    dev = torch.device("cuda", 0)
    if args.profile_case == "decode_layer":
        s = moe.shape(H, I, moe.FMT_NVFP4)
        nE = 64
        pool = torch.empty(nE, moe.moe_expert_record_bytes(s), dtype=torch.uint8, device=dev)
        for e in range(nE):
            g, up, d = synth.expert_weights(H, I, synth.expert_seed(0, 0, e), device=dev)
            moe.fp4_pack_expert(g, up, d, s, record=pool[e])
        # a 512-expert router over the 64 records (expert e -> record e % 64)
        ptrs = moe.pointer_table([pool[e % nE] for e in range(E)])
        wr = synth.router_weights(E, H, synth.seed_of(0, 0, synth.T_ROUTER), device=dev)
        ws = torch.zeros(moe.moe_experts_decode_workspace(1, K_TOP, s), dtype=torch.uint8, device=dev)
        y = torch.empty(1, H, dtype=torch.float32, device=dev)
        for i in range(args.warmup + args.steps):
            x = synth.activations(1, H, synth.seed_of(0, 50 + i, synth.T_X), device=dev)
            moe.moe_decode_layer(wr, None, K_TOP, ptrs, s, x=x, y=y, workspace=ws)
        torch.cuda.synchronize()
    elif args.profile_case == "deepseek_call":
        # the DeepSeek-shaped call (router over 384 MXFP4 experts, top-6, then
        # the ring kernel's expert pass) over 16 distinct records (301 MB):
        # expert e uses record e % 16
        D = DeepSeekCalls
        s = moe.shape(D.HD, D.ID, moe.FMT_MXFP4)
        nE = 16
        pool = torch.empty(nE, moe.moe_expert_record_bytes(s), dtype=torch.uint8, device=dev)
        for e in range(nE):
            g, up, d = synth.expert_weights(D.HD, D.ID, synth.expert_seed(D.WORKLOAD, 0, e), device=dev)
            moe.fp4_pack_expert(g, up, d, s, record=pool[e])
        ptrs = moe.pointer_table([pool[e % nE] for e in range(D.NE)])
        ws = torch.zeros(moe.moe_experts_decode_workspace(1, D.KD, s), dtype=torch.uint8, device=dev)
        for i in range(args.warmup + args.steps):
            wr = synth.router_weights(D.NE, D.HD, synth.seed_of(D.WORKLOAD, i, synth.T_ROUTER), device=dev)
            x = synth.activations(1, D.HD, synth.seed_of(D.WORKLOAD, i, synth.T_X), device=dev)
            idx, w, _ = moe.moe_router_topk(x, wr, None, D.KD)
            moe.moe_experts_decode(x, idx, w, ptrs, s, workspace=ws)
        torch.cuda.synchronize()
    elif args.profile_case == "batched_call":
        # one layer of the batched decode: 32 tokens routed by a 512-expert
        # router over 64 distinct records (177 MB, larger than L2; expert e
        # uses record e % 64), then the ring kernel's expert pass
        s = moe.shape(H, I, moe.FMT_NVFP4)
        nE, T = 64, 32
        pool = torch.empty(nE, moe.moe_expert_record_bytes(s), dtype=torch.uint8, device=dev)
        for e in range(nE):
            g, up, d = synth.expert_weights(H, I, synth.expert_seed(0, 0, e), device=dev)
            moe.fp4_pack_expert(g, up, d, s, record=pool[e])
        ptrs = moe.pointer_table([pool[e % nE] for e in range(E)])
        wr = synth.router_weights(E, H, synth.seed_of(0, 0, synth.T_ROUTER), device=dev)
        ws = torch.zeros(moe.moe_experts_decode_workspace(T, K_TOP, s), dtype=torch.uint8, device=dev)
        y = torch.empty(T, H, dtype=torch.float32, device=dev)
        for i in range(args.warmup + args.steps):
            x = synth.activations(T, H, synth.seed_of(0, 70 + i, synth.T_X), device=dev)
            idx, w, _ = moe.moe_router_topk(x, wr, None, K_TOP)
            moe.moe_experts_decode(x, idx, w, ptrs, s, y, workspace=ws)
        torch.cuda.synchronize()
    elif args.profile_case == "fp8_gemv":
        # 8192 x 2560 E4M3 GEMVs on 8 distinct matrices (168 MB, larger than L2)
        M, K, n = 8192, 2560, 8
        ws_ = [synth.expert_matrix((M, K), seed=M + K + i, device=dev).to(torch.float8_e4m3fn).view(torch.uint8)
               for i in range(n)]
        sc = synth.uniform((M,), seed=M, lo=0.5, hi=2.0, device=dev)
        x = synth.activations(1, K, seed=K, device=dev)[0]
        y = torch.empty(M, dtype=torch.float32, device=dev)
        for i in range(args.warmup + args.steps):
            moe.fp8_rowscale_gemv(ws_[i % n], sc, x, y)
        torch.cuda.synchronize()
    else:
        pl = PromptLayer(torch, moe, synth, dev)
        for _ in range(args.warmup + args.steps):
            pl.step()
        torch.cuda.synchronize()
    print("profile case done", file=sys.stderr)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prompt", action="store_true")
    ap.add_argument("--no-others", action="store_true", help="skip the one-layer, DeepSeek-shaped and batched workloads")
    ap.add_argument("--cpu-seconds-other", type=float, default=6.0)
    ap.add_argument("--profile-case", choices=("none", "decode_layer", "prompt_layer", "deepseek_call", "batched_call",
                                               "fp8_gemv"), default="none",
                    help="small fixed case for ncu captures (no JSON line)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.profile_case != "none":
        run_profile_case(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
