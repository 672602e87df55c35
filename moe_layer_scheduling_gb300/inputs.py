"""Seeded synthetic workloads for the MoE layer, the split-K row sum and the chain.

This module only draws random numbers and casts them; it holds none of the
method's arithmetic.  Both the CUDA path and the fp64 oracle are fed from here,
so that the two sides see bit-identical inputs.

Random numbers come from numpy's PCG64 generator (``numpy.random.default_rng``),
whose streams are fixed by the seed on every platform; fp32 draws are rounded to
bf16 with round-to-nearest-even through torch's dtype cast.

Workload shapes follow the MoE layer the Event Tensor pages benchmark
("Event Tensor: A Unified Abstraction for Compiling Dynamic Megakernel",
Figure 13 and the podcast transcript's scoreboard cue: Qwen3-30B-A3B, 128
experts, top-k 8) and the split-K example of Figure 3.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

# Qwen3-30B-A3B MoE layer shape (hidden, experts, top-k, expert intermediate).
QWEN_H, QWEN_E, QWEN_K, QWEN_I = 2048, 128, 8, 768
# Tiny layer used for exhaustive parity.
TINY_H, TINY_E, TINY_K, TINY_I = 256, 8, 2, 512
WEIGHT_STD = 0.02


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a CPU bf16 tensor as a uint16 numpy array (no copy of values)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


@dataclass
class MoEWeights:
    hidden: int
    n_experts: int
    top_k: int
    inter: int
    gate_w: torch.Tensor        # bf16 [H, E]   router weight, row-major
    w_gate_up: torch.Tensor     # bf16 [E, 2I, H]  rows 0..I-1 gate, I..2I-1 up
    w_down: torch.Tensor        # bf16 [E, H, I]
    router_bias: torch.Tensor | None = None  # fp32 [E] or None
    norm_w: torch.Tensor | None = None       # bf16 [H] RMSNorm gain (chain blocks)


def moe_weights(hidden: int, n_experts: int, top_k: int, inter: int, seed: int,
                std: float = WEIGHT_STD) -> MoEWeights:
    """Router and expert weights ~ N(0, std^2), cast to bf16."""
    rng = np.random.default_rng(seed)
    gate_w = _bf16(rng.standard_normal((hidden, n_experts), dtype=np.float32) * std)
    wgu = np.empty((n_experts, 2 * inter, hidden), dtype=np.float32)
    wd = np.empty((n_experts, hidden, inter), dtype=np.float32)
    for e in range(n_experts):  # per expert keeps peak host memory low
        wgu[e] = rng.standard_normal((2 * inter, hidden), dtype=np.float32) * std
        wd[e] = rng.standard_normal((hidden, inter), dtype=np.float32) * std
    return MoEWeights(hidden, n_experts, top_k, inter, gate_w, _bf16(wgu), _bf16(wd))


def tokens(T: int, hidden: int, seed: int) -> torch.Tensor:
    """Activations x ~ N(0, 1), bf16 [T, H]."""
    rng = np.random.default_rng(seed)
    return _bf16(rng.standard_normal((T, hidden), dtype=np.float32))


def zipf_bias(n_experts: int, s: float = 1.2, seed: int = 0) -> torch.Tensor:
    """Per-expert router bias -s*ln(rank), ranks 1..E in a seeded random order.

    exp(bias) is then proportional to rank^-s: a Zipf(s) preference over experts
    that skews routing so that some experts receive no tokens.
    """
    rng = np.random.default_rng(seed)
    rank = 1 + rng.permutation(n_experts)
    return torch.from_numpy((-s * np.log(rank.astype(np.float64))).astype(np.float32))


def splitk_matrix(n_rows: int, n_cols: int, seed: int = 0) -> torch.Tensor:
    """A ~ U(-1, 1), fp32 [n_rows, n_cols]."""
    rng = np.random.default_rng(seed)
    return torch.from_numpy(rng.uniform(-1.0, 1.0, size=(n_rows, n_cols)).astype(np.float32))


def chain_t_sequence(n: int = 200, lo: int = 1, hi: int = 512, seed: int = 7) -> list[int]:
    """Per-call token counts for the dynamic-shape chain, uniform in [lo, hi]."""
    rng = np.random.default_rng(seed)
    return [int(v) for v in rng.integers(lo, hi + 1, size=n)]


# ----------------------------------------------------------------------------
# Named workloads
# ----------------------------------------------------------------------------

@dataclass
class MoEWorkload:
    name: str
    T: int
    weights: MoEWeights
    x: torch.Tensor
    meta: dict = field(default_factory=dict)


def tiny_layer(seed: int = 0) -> MoEWorkload:
    """T=4, hidden 256, 8 experts, top-2, intermediate 512."""
    w = moe_weights(TINY_H, TINY_E, TINY_K, TINY_I, seed)
    x = tokens(4, TINY_H, seed + 1)
    return MoEWorkload("tiny_T4_H256_E8_k2_I512", 4, w, x)


def qwen_weights(seed: int = 0) -> MoEWeights:
    return moe_weights(QWEN_H, QWEN_E, QWEN_K, QWEN_I, seed)


def decode_layer(T: int, weights: MoEWeights | None = None) -> MoEWorkload:
    """Qwen3-30B-A3B-shaped decode batch, near-uniform routing from random gate weights."""
    w = weights if weights is not None else qwen_weights(0)
    return MoEWorkload(f"qwen3_30b_a3b_moe_decode_T{T}", T, w, tokens(T, QWEN_H, 1000 + T))


def prefill_skew_layer(T: int = 4096, weights: MoEWeights | None = None) -> MoEWorkload:
    """Same shape, T=4096, router logits skewed by a Zipf(1.2) per-expert bias."""
    w = weights if weights is not None else qwen_weights(0)
    w = MoEWeights(w.hidden, w.n_experts, w.top_k, w.inter, w.gate_w, w.w_gate_up,
                   w.w_down, router_bias=zipf_bias(w.n_experts, 1.2, 0))
    return MoEWorkload(f"qwen3_30b_a3b_moe_prefill_T{T}_zipf1.2", T, w, tokens(T, QWEN_H, 2000 + T))


def chain_blocks(n_blocks: int = 4, hidden: int = QWEN_H, n_experts: int = QWEN_E,
                 top_k: int = QWEN_K, inter: int = QWEN_I) -> list[MoEWeights]:
    """Independent weight sets for the RMSNorm -> MoE -> residual chain (seeds 100+b), unit norm gains."""
    blocks = []
    for b in range(n_blocks):
        w = moe_weights(hidden, n_experts, top_k, inter, 100 + b)
        w.norm_w = torch.ones(hidden, dtype=torch.bfloat16)
        blocks.append(w)
    return blocks


# ----------------------------------------------------------------------------
# Dense MLP (the appendix's Table 4: sequence length S, hidden H, intermediate I)
# ----------------------------------------------------------------------------

MLP_SHAPES = {
    "MLP-1": (8192, 4096, 12288),   # Qwen3-8B
    "MLP-2": (8192, 4096, 14336),   # LLaMA-3.1-8B
    "MLP-3": (8192, 3584, 14336),   # Gemma-2-9B
    "MLP-4": (8192, 4608, 36864),   # Gemma-2-27B
    "MLP-5": (8192, 5120, 25600),   # Qwen3-32B
}


@dataclass
class MLPWeights:
    hidden: int
    inter: int
    w_gate_up: torch.Tensor     # bf16 [2I, H]  rows 0..I-1 gate, I..2I-1 up
    w_down: torch.Tensor        # bf16 [H, I]


def mlp_weights(hidden: int, inter: int, seed: int, std: float = WEIGHT_STD) -> MLPWeights:
    """Dense MLP weights ~ N(0, std^2), cast to bf16, drawn in row slabs (low host memory)."""
    rng = np.random.default_rng(seed)
    slab = max(1, (1 << 24) // hidden)
    wgu = torch.empty(2 * inter, hidden, dtype=torch.bfloat16)
    for r in range(0, 2 * inter, slab):
        n = min(slab, 2 * inter - r)
        wgu[r:r + n] = _bf16(rng.standard_normal((n, hidden), dtype=np.float32) * std)
    wd = torch.empty(hidden, inter, dtype=torch.bfloat16)
    slab = max(1, (1 << 24) // inter)
    for r in range(0, hidden, slab):
        n = min(slab, hidden - r)
        wd[r:r + n] = _bf16(rng.standard_normal((n, inter), dtype=np.float32) * std)
    return MLPWeights(hidden, inter, wgu, wd)


def mlp_layer(name: str = "MLP-1", T: int | None = None, seed: int = 300):
    """(weights, x) of a Table 4 MLP shape; x ~ N(0, 1) with T rows (S by default)."""
    S, H, I = MLP_SHAPES[name]
    return mlp_weights(H, I, seed), tokens(S if T is None else T, H, seed + 1)


def expected_touched_experts(T: int, n_experts: int = QWEN_E, top_k: int = QWEN_K) -> float:
    """E * (1 - ((E-k)/E)^T): expected number of experts hit under uniform routing."""
    return n_experts * (1.0 - math.pow((n_experts - top_k) / n_experts, T))
