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


GUARD_BYTES = 64 * 1024
SENTINEL = 0xFF


def guarded(n: int, dtype) -> tuple:
    """An output buffer of n elements between two 64 KiB guard bands, every
    byte 0xFF (the interior too: NaN in bf16 and fp32, so an element never
    written shows as well).  Returns (whole buffer, interior view); the
    interior starts 64 KiB in, so it keeps the allocation's alignment."""
    esz = torch.empty(0, dtype=dtype).element_size()
    whole = torch.full((2 * GUARD_BYTES + n * esz,), SENTINEL, dtype=torch.uint8, device=device())
    return whole, whole[GUARD_BYTES:GUARD_BYTES + n * esz].view(dtype)


def assert_guards_intact(whole: torch.Tensor, what="") -> None:
    """Both guard bands still hold the sentinel: nothing was stored outside the output."""
    head = whole[:GUARD_BYTES]
    tail = whole[whole.numel() - GUARD_BYTES:]
    assert bool((head == SENTINEL).all()) and bool((tail == SENTINEL).all()), f"store outside the output {what}"
