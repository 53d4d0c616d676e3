"""Seeded synthetic MoE workloads (inputs only; none of the method's arithmetic).

Shared by the tests, the oracle checks and ``bench.py``.  The pages measure on
no public dataset, so these five recipes stand in for the workloads they
describe: BF16 tokens of an MoE layer (activations for the dispatch forward,
gradients for the combine backward) plus top-k routing ids.

Recipe: numpy ``default_rng`` (PCG64); the token values are drawn from the
stream seeded ``[seed, 0]`` and the routing from the stream seeded
``[seed, 1]``.  Values are drawn in float32 and rounded to BF16 with
round-to-nearest-even (torch's float32 -> bfloat16 conversion).  Every config
can be scaled down (``T``/``H`` overrides) for parity tests that the oracle
finishes in seconds; the recipe is otherwise unchanged.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

ALIGNMENT = 128          # per-expert slot alignment of the grouped operands
SIGN_MASK = 0xA53C       # RHT sign vector: bit i set -> sigma_i = -1
SR_SEED = 1234           # Philox seed of the stochastic-rounding workload


@dataclass
class Workload:
    name: str
    description: str
    tokens: np.ndarray          # uint16 [T, H], BF16 bit patterns
    topk: np.ndarray            # int32 [T, k], expert ids (-1 = dropped slot)
    E: int
    A: int = ALIGNMENT
    rounding: int = 0           # 0 = RNE, 1 = stochastic rounding
    seed: int = 0               # Philox seed for stochastic rounding
    sign_mask: int = SIGN_MASK
    ops: tuple = ("pack", "direct_receive")
    extra: dict = field(default_factory=dict)

    @property
    def T(self) -> int:
        return int(self.tokens.shape[0])

    @property
    def H(self) -> int:
        return int(self.tokens.shape[1])

    @property
    def k(self) -> int:
        return int(self.topk.shape[1])


def to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """float32 -> BF16 bit patterns (uint16), round to nearest even."""
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32)


def _topk_uniform(rng, T, E, k, excluded=()):
    keys = rng.random((T, E))
    if len(excluded):
        keys[:, list(excluded)] = np.inf
    return np.argsort(keys, axis=1, kind="stable")[:, :k].astype(np.int32)


def _topk_weighted(rng, T, p, k):
    # Gumbel-top-k: k draws without replacement, each proportional to p
    g = rng.gumbel(size=(T, p.shape[0]))
    keys = np.log(p)[None, :] + g
    return np.argsort(-keys, axis=1, kind="stable")[:, :k].astype(np.int32)


def _shape(T, H, T0, H0):
    return (T0 if T is None else int(T)), (H0 if H is None else int(H))


def config1(T=None, H=None, seed=0) -> Workload:
    """Tiny pack / unpack / direct receive: rows N(0,1) * lognormal(0,1)."""
    T, H = _shape(T, H, 256, 1024)
    rd, rr = np.random.default_rng([seed, 0]), np.random.default_rng([seed, 1])
    x = rd.standard_normal((T, H), dtype=np.float32)
    x *= np.exp(rd.standard_normal((T, 1), dtype=np.float32))
    topk = _topk_uniform(rr, T, 8, 2)
    return Workload("cfg1", f"{T}x{H} bf16 N(0,1)*lognormal(0,1) per row; 8 experts top-2 uniform; RNE",
                    to_bf16_bits(x), topk, E=8, ops=("pack", "unpack", "direct_receive"))


def config2(T=None, H=None, seed=2) -> Workload:
    """Dispatch forward: N(0,1) with 0.1% of the entries x50; softmax top-2 of
    16 experts, experts 14 and 15 forced empty."""
    T, H = _shape(T, H, 4096, 4096)
    rd, rr = np.random.default_rng([seed, 0]), np.random.default_rng([seed, 1])
    x = rd.standard_normal((T, H), dtype=np.float32)
    n_out = int(round(0.001 * T * H))
    idx = rd.choice(T * H, size=n_out, replace=False)
    x.reshape(-1)[idx] *= 50.0
    logits = rr.standard_normal((T, 16))
    logits[:, 14:] = -np.inf
    p = np.exp(logits - logits.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    # larger probability first, the lower expert id on a tie (stable sort)
    topk = np.argsort(-p, axis=1, kind="stable")[:, :2].astype(np.int32)
    return Workload("cfg2", f"{T}x{H} bf16 N(0,1), 0.1% entries x50; 16 experts softmax top-2, experts 14,15 empty",
                    to_bf16_bits(x), topk, E=16)


def config3(T=None, H=None, seed=3) -> Workload:
    """Imbalanced MoE: tokens N(0,1) * lognormal(0,0.5); 8 experts top-2 with
    loads Zipf(s=1.2); also unpacked to BF16."""
    T, H = _shape(T, H, 8192, 4096)
    rd, rr = np.random.default_rng([seed, 0]), np.random.default_rng([seed, 1])
    x = rd.standard_normal((T, H), dtype=np.float32)
    x *= np.exp(0.5 * rd.standard_normal((T, 1), dtype=np.float32))
    p = (np.arange(1, 9, dtype=np.float64)) ** -1.2
    p /= p.sum()
    topk = _topk_weighted(rr, T, p, 2)
    return Workload("cfg3", f"{T}x{H} bf16 N(0,1)*lognormal(0,0.5); 8 experts top-2 Zipf(1.2)",
                    to_bf16_bits(x), topk, E=8, ops=("pack", "direct_receive", "unpack"))


def config4(T=None, H=None, seed=4, E=256, k=8) -> Workload:
    """Combine-backward gradients: 1e-3 * N(0,1) * lognormal(0,1) per token;
    256 experts top-8, 10% of the experts empty; stochastic rounding."""
    T, H = _shape(T, H, 16384, 7168)
    rd, rr = np.random.default_rng([seed, 0]), np.random.default_rng([seed, 1])
    x = rd.standard_normal((T, H), dtype=np.float32)
    x *= np.float32(1e-3) * np.exp(rd.standard_normal((T, 1), dtype=np.float32))
    n_empty = int(np.ceil(0.1 * E))
    empty = rr.permutation(E)[:n_empty]
    topk = _topk_uniform(rr, T, E, k, excluded=empty)
    return Workload("cfg4", f"{T}x{H} bf16 1e-3*N(0,1)*lognormal(0,1); {E} experts top-{k}, {n_empty} empty; SR seed {SR_SEED}",
                    to_bf16_bits(x), topk, E=E, rounding=1, seed=SR_SEED,
                    extra={"empty_experts": np.sort(empty).tolist()})


def config5(T=None, H=None, seed=5) -> Workload:
    """MXFP8 vs NVFP4 dispatch: StudentT(df=4); 64 experts top-6 uniform."""
    T, H = _shape(T, H, 16384, 7168)
    rd, rr = np.random.default_rng([seed, 0]), np.random.default_rng([seed, 1])
    x = rd.standard_t(4, size=(T, H)).astype(np.float32)
    topk = _topk_uniform(rr, T, 64, 6)
    return Workload("cfg5", f"{T}x{H} bf16 StudentT(4); 64 experts top-6 uniform; MXFP8 and NVFP4",
                    to_bf16_bits(x), topk, E=64, ops=("mxfp8_pack", "pack", "direct_receive"))


CONFIGS = {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}


def make(cfg: int, **kw) -> Workload:
    return CONFIGS[int(cfg)](**kw)
