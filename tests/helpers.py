"""Test helpers: seeded pools on the device and their host copies for the
oracle.  Only inputs travel from the device to the oracle (FP32 weights drawn
by torch's generator, BF16 activations); nothing the library computes does."""
import os

import numpy as np
import torch

from block_scaled_fp4_softmax_gb300 import moe, synth
from oracle import oracle as O


def bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


class Pool:
    """E experts packed on the device by fp4_pack_expert, each from FP32
    weights drawn on the device with a per-expert seed."""

    def __init__(self, E, H, I, fmt, workload, layer=0, std=0.02, device="cuda"):
        self.E, self.H, self.I, self.fmt = E, H, I, fmt
        self.workload, self.layer, self.std = workload, layer, std
        self.shape = moe.shape(H, I, fmt)
        nbytes = moe.moe_expert_record_bytes(self.shape)
        self.stride = (nbytes + 4095) // 4096 * 4096
        self.buf = torch.empty(E * self.stride, dtype=torch.uint8, device=device)
        for e in range(E):
            g, u, d = self.weights(e, device)
            moe.fp4_pack_expert(g, u, d, self.shape, record=self.record(e))
        self.ptrs = moe.pointer_table([self.record(e) for e in range(E)])
        self._oracle_records = {}

    def seed(self, e):
        return synth.expert_seed(self.workload, self.layer, e)

    def weights(self, e, device="cuda"):
        return synth.expert_weights(self.H, self.I, self.seed(e), device=device, std=self.std)

    def record(self, e):
        n = moe.moe_expert_record_bytes(self.shape)
        return self.buf[e * self.stride: e * self.stride + n]

    def oracle_record(self, e):
        """The oracle's own packing of expert e (from the same FP32 inputs)."""
        if e not in self._oracle_records:
            g, u, d = (w.cpu().numpy() for w in self.weights(e))
            self._oracle_records[e] = O.pack_expert(g, u, d, self.fmt)
        return self._oracle_records[e]

    def oracle_records(self, experts):
        return {int(e): self.oracle_record(int(e)) for e in set(int(v) for v in experts)}


def _pack_worker(args):
    g, u, d, fmt = args
    return O.pack_expert(g, u, d, fmt)


_POOL = None


def oracle_pack_many(pool: "Pool", experts):
    """The oracle's records for many experts, packed in parallel worker
    processes (spawned, never forked, so no CUDA state is inherited)."""
    import concurrent.futures as cf
    import multiprocessing as mp
    global _POOL
    want = [int(e) for e in sorted(set(int(v) for v in experts)) if int(e) not in pool._oracle_records]
    if want:
        if _POOL is None:
            _POOL = cf.ProcessPoolExecutor(max_workers=min(16, os.cpu_count() or 4),
                                           mp_context=mp.get_context("spawn"))
        jobs = []
        for e in want:
            g, u, d = (w.cpu().numpy() for w in pool.weights(e))
            jobs.append(_POOL.submit(_pack_worker, (g, u, d, pool.fmt)))
        for e, j in zip(want, jobs):
            pool._oracle_records[e] = j.result()
    return {int(e): pool._oracle_records[int(e)] for e in experts}


def _split_worker(args):
    fn_name, x, idx, w, recs, H, I, fmt, subset = args
    fn = getattr(O, fn_name)
    return fn(x, idx, w, recs, H, I, fmt, experts=subset)


def oracle_layer_split(fn_name, xb, idx, w, records, H, I, fmt, parts=16):
    """The oracle's layer function (moe_layer_decode or
    moe_layer_grouped_by_expert) with its experts split over worker processes:
    each worker sums the pairs of its experts, and the parts are added in
    float64.  Each pair's arithmetic is the oracle's own; only the order in
    which whole expert contributions are added differs (float64, far below the
    tolerances)."""
    import concurrent.futures as cf
    import multiprocessing as mp
    global _POOL
    if _POOL is None:
        _POOL = cf.ProcessPoolExecutor(max_workers=min(16, os.cpu_count() or 4),
                                       mp_context=mp.get_context("spawn"))
    experts = sorted({int(e) for e in np.asarray(idx).ravel()})
    groups = [experts[i::parts] for i in range(parts) if experts[i::parts]]
    jobs = [_POOL.submit(_split_worker, (fn_name, xb, idx, w, {e: records[e] for e in g}, H, I, fmt, g))
            for g in groups]
    y = np.zeros((np.asarray(xb).shape[0], H), dtype=np.float64)
    for j in jobs:
        y += j.result().astype(np.float64)
    return y.astype(np.float32)
