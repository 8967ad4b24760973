"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module draws random numbers and nothing else: it holds none of the
method's arithmetic (no quantisation, routing or FFN math).  Every tensor is a
pure function of (shape, seed, device):

* activations ``x``: BF16 ~ N(0, 1);
* router weights ``W_r``: BF16 ~ N(0, 0.02);
* expert weights (gate, up, down): FP32 ~ N(0, 0.02), later packed by the
  caller into block-scaled FP4 records;
* a Zipf popularity bias over experts for the skewed prompt workload.

CPU generation (``device="cpu"``) is used for the small parity cases; the big
resident expert pools are drawn on the GPU with a per-expert CUDA generator so
that any single expert can be re-drawn later (and copied to the host) by seed.
"""

from __future__ import annotations

import math

import numpy as np
import torch

# tensor ids inside a seed; a seed is 1000*workload + 10*layer + tensor_id for
# per-layer tensors, and a separate space for per-expert weights.
T_X, T_ROUTER, T_BIAS, T_PERM = 0, 1, 2, 3


def seed_of(workload: int, layer: int, tensor_id: int) -> int:
    return 1000 * int(workload) + 10 * int(layer) + int(tensor_id)


def expert_seed(workload: int, layer: int, expert: int) -> int:
    # disjoint from seed_of's range for any realistic workload/layer count
    return 10_000_000 + 1_000_000 * int(workload) + 1000 * int(layer) + int(expert)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def activations(T: int, H: int, seed: int, device="cpu") -> torch.Tensor:
    """x: BF16 [T, H] ~ N(0, 1)."""
    g = _gen(seed, device)
    return torch.randn(T, H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def router_weights(E: int, H: int, seed: int, device="cpu") -> torch.Tensor:
    """W_r: BF16 [E, H] ~ N(0, 0.02)."""
    g = _gen(seed, device)
    w = torch.randn(E, H, generator=g, device=device, dtype=torch.float32) * 0.02
    return w.to(torch.bfloat16)


def expert_weights(H: int, I: int, seed: int, device="cpu", std: float = 0.02):
    """One expert's FP32 (gate [I,H], up [I,H], down [H,I]) ~ N(0, std)."""
    g = _gen(seed, device)
    flat = torch.randn(3 * I * H, generator=g, device=device, dtype=torch.float32) * std
    gate = flat[: I * H].view(I, H)
    up = flat[I * H: 2 * I * H].view(I, H)
    down = flat[2 * I * H:].view(H, I)
    return gate, up, down


def zipf_bias(E: int, seed: int, s: float = 1.1, tau: float = 0.5) -> torch.Tensor:
    """FP32 [E] router bias from a Zipf(s) popularity profile.

    Expert e gets rank r(e) = perm(e) + 1 from a seeded permutation;
    bias[e] = tau * ln(p_r), p_r = r^-s / sum_r' r'^-s.  The bias is an input of
    the router (it shifts the logits), it is not part of the method.
    """
    rng = np.random.default_rng(int(seed))
    perm = rng.permutation(E)
    ranks = perm.astype(np.float64) + 1.0
    norm = math.fsum((np.arange(1, E + 1, dtype=np.float64) ** (-s)).tolist())
    p = ranks ** (-s) / norm
    return torch.from_numpy((tau * np.log(p)).astype(np.float32))


def expert_matrix(shape, seed: int, device="cpu", std: float = 0.02) -> torch.Tensor:
    """A plain FP32 matrix ~ N(0, std) (used for FP8 row-scaled GEMV weights)."""
    g = _gen(seed, device)
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * std


def uniform(shape, seed: int, lo: float, hi: float, device="cpu") -> torch.Tensor:
    g = _gen(seed, device)
    return torch.rand(*shape, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo


def random_bytes(n: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(int(seed))
    return rng.integers(0, 256, size=n, dtype=np.uint8)
