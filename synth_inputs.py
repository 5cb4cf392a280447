"""Seeded synthetic inputs shared by the oracle side and the GPU side.

This module holds no arithmetic of the method: it only draws random numbers
in the distributions and shapes of the workloads and rounds them to the
dtype the GPU path computes in.  Matrices are produced in their global
(unsharded) form; each side shards them with its own layout code.

Draws use ``torch.Generator`` on the CPU in float32, then round to nearest
even into bfloat16 where the workload is bf16.  The seed of workload n is
20260 + n unless a test passes its own.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

SEED_BASE = 20260


def gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal(shape, std: float, seed: int, dtype=torch.bfloat16, mean: float = 0.0) -> torch.Tensor:
    """N(mean, std^2) in float32, rounded to ``dtype``."""
    t = torch.randn(*shape, generator=gen(seed), dtype=torch.float32) * std + mean
    return t.to(dtype)


def uniform_ints(shape, lo: int, hi: int, seed: int, dtype=torch.bfloat16) -> torch.Tensor:
    """Integers uniform in [lo, hi], exact in bf16 while |x| <= 256."""
    t = torch.randint(lo, hi + 1, tuple(shape), generator=gen(seed), dtype=torch.int32)
    return t.to(dtype)


def random_bits16(shape, seed: int) -> torch.Tensor:
    """Uniform 16-bit patterns (as int16), for bit-transparency checks."""
    return torch.randint(-32768, 32768, tuple(shape), generator=gen(seed), dtype=torch.int32).to(torch.int16)


def bf16_bits(t: torch.Tensor):
    """A bf16 tensor's bit patterns as a numpy uint16 array (no arithmetic)."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def as_f64(t: torch.Tensor):
    """Widen exactly to float64 numpy (bf16 and fp32 values are exact in fp64)."""
    return t.to(torch.float64).numpy()


@dataclass(frozen=True)
class Workload:
    name: str
    q: int
    sizes: dict
    dtype: str


# The five workloads, by what they are and their sizes.
LINEAR_F32_Q2 = Workload("linear q=2 M=N=K=64 fp32", 2, dict(M=64, N=64, K=64), "f32")
MLP_Q2 = Workload("MLP q=2 tokens 2048 hidden 1024 ffn 4096 bf16", 2, dict(M=2048, h=1024, f=4096), "bf16")
LAYER_Q2 = Workload("GPT layer fwd+bwd q=2 b4 s1024 h2048 16 heads ffn 8192 bf16", 2,
                    dict(batch=4, seq=1024, hidden=2048, heads=16, ffn=8192), "bf16")
MLP_Q4 = Workload("MLP q=4 tokens 8192 hidden 4096 ffn 16384 bf16", 4, dict(M=8192, h=4096, f=16384), "bf16")
RESHARD_8K = Workload("reshard 8192x8192 bf16 among ROW4 COL4 BLK2x2 CUBE_A(q=2) REP4", 2,
                      dict(R=8192, C=8192), "bf16")


def mlp_inputs(M, h, f, seed, bias_std: float = 0.0):
    """X ~ N(0,1); W1, W2 ~ N(0, 0.02); biases N(0, bias_std) (0 = zero bias)."""
    X = normal((M, h), 1.0, seed)
    W1 = normal((h, f), 0.02, seed + 1)
    W2 = normal((f, h), 0.02, seed + 2)
    if bias_std > 0:
        b1 = normal((f,), bias_std, seed + 3)
        b2 = normal((h,), bias_std, seed + 4)
    else:
        b1 = torch.zeros(f, dtype=torch.bfloat16)
        b2 = torch.zeros(h, dtype=torch.bfloat16)
    return dict(X=X, W1=W1, b1=b1, W2=W2, b2=b2)


def layer_inputs(batch, seq, hidden, heads, ffn, seed, perturb: bool = False):
    """GPT layer: X ~ N(0,1), weights N(0, 0.02), dY ~ N(0,1); biases 0,
    gamma 1, beta 0 unless ``perturb`` (then biases, beta ~ N(0, 0.02) and
    gamma ~ 1 + N(0, 0.02)), all rounded to bf16."""
    M, h, f = batch * seq, hidden, ffn
    out = dict(X=normal((M, h), 1.0, seed), dY=normal((M, h), 1.0, seed + 1),
               w_qkv=normal((h, 3 * h), 0.02, seed + 2), w_o=normal((h, h), 0.02, seed + 3),
               w_1=normal((h, f), 0.02, seed + 4), w_2=normal((f, h), 0.02, seed + 5))
    vec = {"b_qkv": 3 * h, "b_o": h, "b_1": f, "b_2": h, "ln1_b": h, "ln2_b": h}
    for i, (k, n) in enumerate(vec.items()):
        out[k] = normal((n,), 0.02, seed + 10 + i) if perturb else torch.zeros(n, dtype=torch.bfloat16)
    for i, k in enumerate(("ln1_g", "ln2_g")):
        out[k] = normal((h,), 0.02, seed + 20 + i, mean=1.0) if perturb else torch.ones(h, dtype=torch.bfloat16)
    return out
