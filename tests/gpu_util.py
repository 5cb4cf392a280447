"""Helpers of the GPU parity tests: move seeded inputs, sharded by the
oracle's layout maps, onto the GPU, and bring results back."""
import numpy as np
import pytest
import torch

import synth_inputs as S
from oracle import layouts as L


def device():
    if not torch.cuda.is_available():
        pytest.fail("a GPU test ran without a GPU")
    return torch.device("cuda:0")


def to_dev_bf16(G_bf16: torch.Tensor, lay) -> torch.Tensor:
    """Global bf16 matrix -> sharded flat bf16 device buffer (oracle layout map)."""
    bits = L.to_sharded(S.bf16_bits(G_bf16).reshape(G_bf16.shape), lay)
    return torch.from_numpy(bits.view(np.int16).copy()).to(device()).view(torch.bfloat16)


def to_dev_f32(G: torch.Tensor, lay) -> torch.Tensor:
    buf = L.to_sharded(G.to(torch.float32).numpy(), lay)
    return torch.from_numpy(np.ascontiguousarray(buf)).to(device())


def sharded_f64(G: torch.Tensor, lay):
    return L.to_sharded(S.as_f64(G), lay)


def bits_u16(t: torch.Tensor):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def as_np64(t: torch.Tensor):
    return t.float().cpu().numpy().astype(np.float64)
