#!/usr/bin/env python
"""Benchmark of the routed-MoE FFN with block-scaled FP4 experts on GB300.

Default workload: the Qwen-shaped decode stack -- 48 layers, each with 512
NVFP4 experts (H=2560, I=640, 2,764,800-byte records, ~68 GB resident in
HBM), top-10 routing, one token per step; each layer's input is the previous
layer's output, RMS-normalised.  A step runs router -> experts -> RMS chaining
for all 48 layers.  The metric is expert GB/s: the bytes of the records the
step selects divided by the step time, and its fraction of the HBM roofline.

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
            torch.sum(self.flush, 0, out=self.flush_out)  # L2 flush (read sweep)
            a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
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
        return {"tokens_per_s": round(self.T / (ms / 1e3), 1), "ms_per_layer": round(ms, 4),
                "expert_pass_ms": round(ms_exp, 4),
                "expert_tflops": round(flops / (ms_exp / 1e3) / 1e12, 2),
                "expert_weight_gbs": round(hit * self.pool.shape[1] / (ms_exp / 1e3) / 1e9, 1),
                "experts_hit": hit, "max_tokens_per_expert": int(counts.max().item()),
                "tokens": self.T, "dev_status": int(self.st.item()),
                "l2": "flushed between steps by reading a 512 MB buffer"}


def measure_fp8_gemv(torch, moe, synth, device, reps: int = 20):
    """FP8 row-scaled GEMV on the two proposed shapes; GB/s of W + x + y per
    call, L2 flushed between calls."""
    out = {}
    flush = torch.ones(512 << 18, dtype=torch.int32, device=device)   # read sweep evicts the L2
    flush_out = torch.zeros((), dtype=torch.int64, device=device)
    for M, K in ((8192, 2560), (2560, 4096)):
        # enough distinct matrices that consecutive calls never share L2 lines
        n = max(2, (256 << 20) // (M * K) + 1)
        ws = [synth.expert_matrix((M, K), seed=M + K + i, device=device).to(torch.float8_e4m3fn)
              .view(torch.uint8) for i in range(n)]
        s = synth.uniform((M,), seed=M, lo=0.5, hi=2.0, device=device)
        x = synth.activations(1, K, seed=K, device=device)[0]
        y = torch.empty(M, dtype=torch.float32, device=device)
        for i in range(3):
            moe.fp8_rowscale_gemv(ws[i % n], s, x, y)
        tot = 0.0
        for i in range(reps):
            torch.sum(flush, 0, out=flush_out)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            moe.fp8_rowscale_gemv(ws[i % n], s, x, y)
            b.record()
            torch.cuda.synchronize()
            tot += a.elapsed_time(b)
        us = tot / reps * 1e3
        nbytes = M * K + M * 4 + K * 2 + M * 4
        out[f"{M}x{K}"] = {"us": round(us, 2), "gbs": round(nbytes / (us * 1e-6) / 1e9, 1)}
    return out


def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """The largest value over all ranks (the slowest rank's time)."""
    import torch
    if dist is None or not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _hash_sources():
    h = hashlib.sha256()
    d = os.path.join(ROOT, "block_scaled_fp4_softmax_gb300", "csrc")
    for n in sorted(os.listdir(d)):
        with open(os.path.join(d, n), "rb") as f:
            h.update(n.encode() + f.read())
    return h.hexdigest()[:16]


def _traffic_from_profiles(kernel_key: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources."""
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
    time.sleep(0.3)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    t_start.record(stream)
    for s in range(steps):
        one_step(warm + s)
    t_end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = t_start.elapsed_time(t_end) / steps
    if world > 1:
        ms = max_over_ranks(ms, dist, dev)
        dist.barrier()
    st = int(wl.st.item())

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

    # end to end through the C ABI with host buffers: H2D of the token, all
    # 48 layers as separate library calls, D2H of the output
    e2e = None
    if not args.no_e2e:
        x_host = wl.x0.cpu().pin_memory()
        y_host = torch.empty(1, H, dtype=torch.float32).pin_memory()
        e_steps = max(3, min(steps, 20))
        for s in range(2):
            wl.x.copy_(x_host[s:s + 1], non_blocking=True)
            wl.run_layers()
            y_host.copy_(wl.y, non_blocking=True)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        a.record()
        for s in range(e_steps):
            wl.x.copy_(x_host[s % x_host.shape[0]:s % x_host.shape[0] + 1], non_blocking=True)
            wl.run_layers()
            y_host.copy_(wl.y, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        wall = (time.perf_counter() - t0) / e_steps
        e2e = {"value": round(wl.expert_bytes_per_step() / wall / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": H * 2, "d2h_bytes_per_step": H * 4,
               "ms_per_step": round(wall * 1e3, 4), "api": "eager C-ABI calls, 48 per token (moe_decode_layer)"}

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
        "dev_status": st,
        "setup_s": round(wl.setup_s, 1),
    }
    if rank == 0 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
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


def cpu_baseline(budget_s: float):
    nbytes, secs, layers = _oracle_sample(budget_s)
    return {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": _cores(),
            "kind": "oracle",
            "sample": f"{layers} layers of the decode stack for 1 token (router + 10 experts + "
                      f"RMS chaining per layer), float64 numpy; record packing untimed",
            "seconds": round(secs, 2)}


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
    router over a 64-record pool, 177 MB of records, larger than L2), or the
    prompt layer."""
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
    else:
        pl = PromptLayer(torch, moe, synth, dev)
        for _ in range(args.warmup + args.steps):
            pl.step()
        torch.cuda.synchronize()
    print("profile case done", file=sys.stderr)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prompt", action="store_true")
    ap.add_argument("--profile-case", choices=("none", "decode_layer", "prompt_layer"), default="none",
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
