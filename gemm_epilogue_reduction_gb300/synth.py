"""Seeded synthetic inputs for the LM-head projection.

This module is shared by the CUDA path's tests and benchmark and by the oracle's tests. It
holds none of the method's arithmetic: it only draws the inputs and converts bf16 tensors to
the raw bit patterns the oracle reads.

Recipe (the shapes are the five workloads of the test suite; the distributions are chosen so
the logits are on an N(0, 1) scale, like a trained output head's):
  * H ~ N(0, 1), drawn in fp32 and rounded to bf16 (round-to-nearest-even);
  * W ~ N(0, 1/d), drawn in fp32, scaled by d**-0.5, rounded to bf16;
  * H is drawn first, then W in chunks of ``_CHUNK`` rows, from one torch.Generator seeded
    with ``seed`` on ``device`` (CPU and CUDA generators give different numbers; each test
    draws on one device and copies the bits to the other);
  * scoring targets: uniform int32 in [0, V) from a second generator seeded with
    ``target_seed``.
"""
from __future__ import annotations

import numpy as np
import torch

_CHUNK = 8192


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a bf16 tensor as a host uint16 array."""
    assert t.dtype == torch.bfloat16
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bits_to_bf16(bits: np.ndarray, device="cpu") -> torch.Tensor:
    """Inverse of :func:`bf16_bits`."""
    a = np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)
    return torch.from_numpy(a.copy()).view(torch.bfloat16).to(device)


def make_hw(M: int, d: int, V: int, seed: int = 0, device="cpu"):
    """(H [M, d], W [V, d]) bf16 on ``device`` per the recipe above."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    H = torch.randn(M, d, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)
    W = torch.empty(V, d, device=device, dtype=torch.bfloat16)
    scale = float(d) ** -0.5
    for r0 in range(0, V, _CHUNK):
        r1 = min(V, r0 + _CHUNK)
        blk = torch.randn(r1 - r0, d, generator=g, device=device, dtype=torch.float32)
        W[r0:r1] = (blk * scale).to(torch.bfloat16)
    return H, W


def make_targets(M: int, V: int, seed: int = 1, device="cpu") -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return torch.randint(0, V, (M,), generator=g, device=device, dtype=torch.int32)


def duplicate_rows(W: torch.Tensor, pairs) -> torch.Tensor:
    """Copy of W with W[dst] := W[src] for each (src, dst): crafted exact logit ties."""
    W = W.clone()
    for src, dst in pairs:
        W[dst] = W[src]
    return W
