"""Seeded synthetic inputs for the block-scaled FP8 linear layer.

This module only draws random tensors; it holds none of the quantisation or
GEMM arithmetic, so both the CUDA path and the CPU oracle can take their
inputs from it.  Every tensor comes from its own numpy PCG64 stream, seeded
with ``seed * 1000 + tensor_id``, drawn in float32 and rounded to bf16
(round-to-nearest-even, through torch) -- the layer's inputs are bf16.

Workloads (shapes and value distributions follow the layer shapes of the
models the pages measure on: Llama 3.1 8B, Qwen3-8B, Qwen3-30B-A3B MoE):

* ``tiny``      A [256, 512] ~ N(0,1) with 4 outlier columns x20,
                W [384, 512] ~ N(0, 0.02).
* ``llama8b``   M = 4096 tokens ~ N(0,1) with round(0.01 K) outlier channels
                x30; layers QKV (K 4096, N 6144), gate+up (4096, 28672),
                down (14336, 4096); W ~ N(0, 0.02).
* ``qwen_prefill`` M = 16384, Student-t (nu = 4) activations; gate+up
                (4096, 24576), down (12288, 4096), o-proj (4096, 4096).
* ``decode``    M in {1, 8, 64, 256}; (K, N) in {(4096, 6144), (14336, 4096)}.
* ``moe``       8192 tokens, hidden 2048, 128 experts, top-8 routing with
                Zipf(1.1) expert popularity; gate+up (2048 -> 1536) and down
                (768 -> 2048) per expert.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

__all__ = [
    "stream", "to_bf16", "normal_bf16", "student_t_bf16", "with_outlier_columns",
    "LinearCase", "tiny", "llama8b_layers", "qwen_prefill_layers", "decode_case",
    "MoECase", "moe_case", "LLAMA8B_LAYERS", "QWEN_PREFILL_LAYERS", "DECODE_SHAPES",
]

LLAMA8B_LAYERS = {"qkv": (4096, 6144), "gate_up": (4096, 28672), "down": (14336, 4096)}
QWEN_PREFILL_LAYERS = {"gate_up": (4096, 24576), "down": (12288, 4096), "o_proj": (4096, 4096)}
DECODE_SHAPES = [(4096, 6144), (14336, 4096)]
DECODE_TOKENS = [1, 8, 64, 256]


def stream(seed: int, tensor_id: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed * 1000 + tensor_id))


def to_bf16(x: np.ndarray) -> torch.Tensor:
    """float32 numpy array -> bf16 torch CPU tensor (round to nearest even)."""
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def normal_bf16(g: np.random.Generator, shape, std: float = 1.0) -> torch.Tensor:
    x = g.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return to_bf16(x)


def student_t_bf16(g: np.random.Generator, shape, nu: float = 4.0) -> torch.Tensor:
    return to_bf16(g.standard_t(nu, shape).astype(np.float32))


def with_outlier_columns(x: torch.Tensor, g: np.random.Generator, count: int, factor: float):
    """Multiply `count` columns (chosen by a seeded permutation) by `factor`."""
    cols = torch.from_numpy(g.permutation(x.shape[1])[:count].copy())
    x = x.clone()
    x[:, cols] = (x[:, cols].float() * factor).to(torch.bfloat16)
    return x, cols


@dataclass
class LinearCase:
    name: str
    a: torch.Tensor            # bf16 [M, K], CPU
    w: torch.Tensor            # bf16 [N, K], CPU
    info: dict = field(default_factory=dict)

    @property
    def shape(self):
        return self.a.shape[0], self.w.shape[0], self.a.shape[1]   # M, N, K


def tiny(seed: int = 0) -> LinearCase:
    a = normal_bf16(stream(seed, 1), (256, 512))
    a, cols = with_outlier_columns(a, stream(seed, 2), 4, 20.0)
    w = normal_bf16(stream(seed, 3), (384, 512), std=0.02)
    return LinearCase("tiny", a, w, {"outlier_cols": cols.tolist()})


def llama8b_layers(seed: int = 0, M: int = 4096, layers=None) -> list[LinearCase]:
    out = []
    for i, (name, (K, N)) in enumerate(LLAMA8B_LAYERS.items()):
        if layers is not None and name not in layers:
            continue
        a = normal_bf16(stream(seed, 10 + 3 * i), (M, K))
        a, cols = with_outlier_columns(a, stream(seed, 11 + 3 * i), round(0.01 * K), 30.0)
        w = normal_bf16(stream(seed, 12 + 3 * i), (N, K), std=0.02)
        out.append(LinearCase(f"llama8b.{name}", a, w, {"outlier_cols": len(cols)}))
    return out


def qwen_prefill_layers(seed: int = 0, M: int = 16384, layers=None) -> list[LinearCase]:
    out = []
    for i, (name, (K, N)) in enumerate(QWEN_PREFILL_LAYERS.items()):
        if layers is not None and name not in layers:
            continue
        a = student_t_bf16(stream(seed, 40 + 2 * i), (M, K))
        w = normal_bf16(stream(seed, 41 + 2 * i), (N, K), std=0.02)
        out.append(LinearCase(f"qwen_prefill.{name}", a, w))
    return out


def decode_case(M: int, K: int, N: int, seed: int = 0) -> LinearCase:
    a = normal_bf16(stream(seed, 60 + M), (M, K))
    w = normal_bf16(stream(seed, 70 + (K // 128) % 100), (N, K), std=0.02)
    return LinearCase(f"decode.M{M}.K{K}.N{N}", a, w)


@dataclass
class MoECase:
    x: torch.Tensor             # bf16 [tokens, hidden]
    row_token: np.ndarray       # int64 [sum M_e]: token feeding each expert-sorted row
    offsets: np.ndarray         # int32 [G+1]: rows of expert g are offsets[g]..offsets[g+1]-1
    a_gate_up: torch.Tensor     # bf16 [sum M_e, hidden] = x[row_token]
    w_gate_up: torch.Tensor     # bf16 [G, 1536, hidden]
    a_down: torch.Tensor        # bf16 [sum M_e, 768]
    w_down: torch.Tensor        # bf16 [G, hidden, 768]


def zipf_routing(g: np.random.Generator, tokens: int, experts: int, top_k: int, s: float):
    """Each token draws `top_k` distinct experts with probabilities
    proportional to (rank+1)**-s (Gumbel-top-k sampling without replacement);
    ranks are assigned to expert ids by a seeded permutation.  Returns the
    expert-sorted row -> token map and the group offsets."""
    p = (np.arange(experts) + 1.0) ** -s
    p = p[g.permutation(experts)]
    logits = np.log(p / p.sum())
    gumbel = -np.log(-np.log(g.uniform(1e-12, 1.0, (tokens, experts))))
    choice = np.argsort(-(logits[None, :] + gumbel), axis=1)[:, :top_k]   # [T, k]
    expert = choice.reshape(-1)
    token = np.repeat(np.arange(tokens), top_k)
    order = np.argsort(expert, kind="stable")
    counts = np.bincount(expert, minlength=experts)
    offsets = np.zeros(experts + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    return token[order], offsets


def moe_case(seed: int = 0, tokens: int = 8192, hidden: int = 2048, experts: int = 128,
             top_k: int = 8, inter: int = 768, gate_up: int = 1536, zipf_s: float = 1.1,
             with_weights: bool = True) -> MoECase:
    x = normal_bf16(stream(seed, 80), (tokens, hidden))
    row_token, offsets = zipf_routing(stream(seed, 81), tokens, experts, top_k, zipf_s)
    a_gu = x[torch.from_numpy(row_token)]
    a_dn = normal_bf16(stream(seed, 84), (len(row_token), inter))
    if with_weights:
        w_gu = normal_bf16(stream(seed, 82), (experts, gate_up, hidden), std=0.02)
        w_dn = normal_bf16(stream(seed, 83), (experts, hidden, inter), std=0.02)
    else:
        w_gu = w_dn = None
    return MoECase(x, row_token, offsets, a_gu, w_gu, a_dn, w_dn)
