"""Seeded synthetic inputs shared by the oracle side and the CUDA side.

This module draws numbers; it holds none of the MoE layer's arithmetic.
Every value comes from one counter-based generator written with integer
torch ops only, so the same (seed, stream, index) gives the same bits on
the CPU and on a GPU.  That lets the large configurations (tens of GB of
expert weights) be drawn on the device, while the oracle redraws exactly
the slices it checks on the host.

Generator definition
--------------------
``mix32`` is the 32-bit integer finaliser
    x ^= x >> 16; x *= 0x45D9F3B (mod 2^32); x ^= x >> 16;
    x *= 0x45D9F3B (mod 2^32); x ^= x >> 16
(a bijection on 32-bit words).  A stream key is
``key = mix32(mix32(seed) ^ stream)``.  Element ``n`` of the stream uses the
two words ``mix32(key + 2n)`` and ``mix32(key + 2n + 1)`` (mod 2^32), split
into four 16-bit uniforms ``u0..u3``.  The approximately normal draw is the
Irwin-Hall sum ``c = u0 + u1 + u2 + u3 - 2*65535`` (an integer, exact in
fp32) times the fp32 constant ``sigma * sqrt(3) / 65536``, one IEEE multiply,
then rounded to bf16 (round to nearest even).  Its standard deviation is
``sigma`` to within 0.01 %, and it is bounded by about ``3.46 * sigma``.

All int64 intermediates stay below 2^60, so no step relies on overflow.
"""
from __future__ import annotations

import math

import numpy as np
import torch

M32 = 0xFFFFFFFF
_MUL = 0x45D9F3B


def mix32(x: torch.Tensor) -> torch.Tensor:
    """32-bit finaliser on an int64 tensor holding values in [0, 2^32)."""
    x = x ^ (x >> 16)
    x = (x * _MUL) & M32
    x = x ^ (x >> 16)
    x = (x * _MUL) & M32
    x = x ^ (x >> 16)
    return x


def _key(seed: int, stream: int) -> int:
    s = mix32(torch.tensor([seed & M32], dtype=torch.int64))
    return int(mix32(s ^ (stream & M32))[0])


def uniform_words(seed: int, stream: int, n: int, device="cpu", start: int = 0) -> torch.Tensor:
    """``n`` 32-bit hash words (int64 tensor) of one stream, from index ``start``."""
    key = _key(seed, stream)
    idx = torch.arange(start, start + n, dtype=torch.int64, device=device)
    return mix32((idx + key) & M32)


def normal_f32(seed: int, stream: int, n: int, sigma: float, device="cpu", start: int = 0) -> torch.Tensor:
    """Irwin-Hall(4) approximately-normal fp32 draws (before any bf16 rounding)."""
    key = _key(seed, stream)
    idx = torch.arange(start, start + n, dtype=torch.int64, device=device)
    w0 = mix32((2 * idx + key) & M32)
    w1 = mix32((2 * idx + 1 + key) & M32)
    c = (w0 & 0xFFFF) + (w0 >> 16) + (w1 & 0xFFFF) + (w1 >> 16) - 2 * 65535
    scale = torch.tensor(sigma * math.sqrt(3.0) / 65536.0, dtype=torch.float32, device=device)
    return c.to(torch.float32) * scale


def normal_bf16(seed: int, stream: int, n: int, sigma: float, device="cpu", start: int = 0) -> torch.Tensor:
    return normal_f32(seed, stream, n, sigma, device, start).to(torch.bfloat16)


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    """A seeded permutation of 0..n-1 (argsort of distinct hash words)."""
    w = uniform_words(seed, stream, n).numpy()
    return np.argsort(w, kind="stable").astype(np.int64)


# Stream ids.  One stream per tensor; expert slabs get one stream each.
def stream_id(kind: int, layer: int = 0, index: int = 0) -> int:
    return ((kind & 0xFF) << 24) | ((layer & 0xFF) << 16) | (index & 0xFFFF)


KIND_X = 1
KIND_ROUTER = 2
KIND_EXPERT = 3
KIND_OFFSET = 4
KIND_RESIDENCY = 5
KIND_BRIGHT = 6
KIND_STEPX = 7
