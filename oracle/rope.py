"""Rotary position embedding of the decoupled RoPE key (TEST INFRASTRUCTURE
ONLY: tests, the smoke check and the benchmark's CPU leg).

The cached row keeps a 64-dim RoPE key beside the 512-dim latent; RoPE is
applied to it at the token's position before it is cached (GLM-4.7-Flash
record, phantomic12 inference-research, configuration clause:
qk_rope_head_dim 64, rope_theta 1000000).  The pages do not say how the 64
values pair up; the reading taken here is the interleaved pairing of the MLA
family's RoPE key: pair i = (x[2i], x[2i+1]), i = 0..31, turned by the angle
pos * theta^(-2i/64):

    y[2i]   = x[2i] cos(a_i) - x[2i+1] sin(a_i)
    y[2i+1] = x[2i] sin(a_i) + x[2i+1] cos(a_i),     a_i = pos * theta^(-2i/d)

Plain float64 numpy; nothing here is shared with the CUDA path.
"""
from __future__ import annotations

import numpy as np

ROPE_DIM = 64
ROPE_THETA = 1.0e6


def inverse_frequencies(dim: int = ROPE_DIM, theta: float = ROPE_THETA) -> np.ndarray:
    """theta^(-2i/dim) for pair i = 0 .. dim/2 - 1."""
    i = np.arange(dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / dim)


def rope_rotate(x: np.ndarray, pos: int, theta: float = ROPE_THETA) -> np.ndarray:
    """Rotate one RoPE key x (float64 [dim], dim even) to position pos."""
    x = np.asarray(x, dtype=np.float64)
    dim = x.shape[-1]
    ang = float(pos) * inverse_frequencies(dim, theta)
    c, s = np.cos(ang), np.sin(ang)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    y = np.empty_like(x)
    y[..., 0::2] = x0 * c - x1 * s
    y[..., 1::2] = x0 * s + x1 * c
    return y
