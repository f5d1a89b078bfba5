"""FP8 latent-cache encoding for the CPU oracle (TEST INFRASTRUCTURE ONLY).

Layout (GLM-4.7-Flash record, phantomic12 inference-research, engine-kernel
constraint (2) on FlashMLA: an FP8 latent with per-token inlined scales,
float8_e4m3 values with one float8_e8m0 scale per 32 e4m3 values, the RoPE
dims quantised too).  This build stores all 576 dims of a cached row:

    token row = 576 e4m3 bytes || 18 e8m0 bytes   (594 bytes)

and a page of P tokens is P contiguous rows (P * 594 bytes).  Group g covers
dims [32 g, 32 g + 32); scale byte g of the row belongs to group g.

Value decoding follows the OCP 8-bit floating point definitions:
  e4m3 (fn): sign bit, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0
  is subnormal (m/8 * 2**-6); S.1111.111 is NaN; no infinities.
  e8m0: unsigned 8-bit exponent, value 2**(byte - 127); 0xFF is NaN.

Quantiser (data generation, not on the decode path).  Reading of "scales from
per-group absmax": e = clamp(ceil(log2(amax / 448)), -127, 127), scale byte
e + 127, values round-to-nearest-even of x / 2**e into e4m3, saturating at
+-448; an all-zero group gets scale byte 0 and zero values.
"""
from __future__ import annotations

import numpy as np

D_QK = 576
GROUP = 32
N_GROUPS = D_QK // GROUP
ROW_BYTES = D_QK + N_GROUPS
E4M3_MAX = 448.0


def e4m3_to_f64(code: np.ndarray) -> np.ndarray:
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = c & 0x7
    val = np.where(exp == 0,
                   np.ldexp(man / 8.0, -6),
                   np.ldexp(1.0 + man / 8.0, exp - 7))
    val = sign * val
    return np.where((exp == 0xF) & (man == 0x7), np.nan, val)


def e8m0_to_f64(code: np.ndarray) -> np.ndarray:
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    val = np.ldexp(1.0, c - 127)
    return np.where(c == 0xFF, np.nan, val)


def dequant_rows(rows: np.ndarray) -> np.ndarray:
    """rows: uint8 [..., 594] -> float64 [..., 576] = e4m3 * 2**(s - 127)."""
    rows = np.asarray(rows, dtype=np.uint8)
    vals = e4m3_to_f64(rows[..., :D_QK])
    scales = e8m0_to_f64(rows[..., D_QK:])
    return vals * np.repeat(scales, GROUP, axis=-1)


def _f64_to_e4m3_code(v: np.ndarray) -> np.ndarray:
    """Encode values already rounded to e4m3-representable magnitudes."""
    v = np.asarray(v, dtype=np.float64)
    sign = (np.signbit(v)).astype(np.uint8) << 7
    a = np.abs(v)
    m, e = np.frexp(a)                    # a = m * 2**e, m in [0.5, 1)
    normal = a >= 2.0 ** -6
    exp_field = np.where(normal, e - 1 + 7, 0)
    man_normal = np.round((m * 2.0 - 1.0) * 8.0)
    man_sub = np.round(a / 2.0 ** -9)
    man = np.where(normal, man_normal, man_sub)
    code = (exp_field.astype(np.int64) << 3) | man.astype(np.int64)
    code = np.where(a == 0, 0, code)
    return sign | code.astype(np.uint8)


def _round_to_e4m3(v: np.ndarray) -> np.ndarray:
    """Round to the nearest e4m3 value (ties to even), saturating at +-448."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, e = np.frexp(a)
    # spacing: normal binade [2**(e-1), 2**e) has 3 fraction bits; subnormal 2**-9
    q = np.ldexp(1.0, np.maximum(e - 1, -6) - 3)
    r = np.round(a / q) * q
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, v)


def quantize_rows(x: np.ndarray) -> np.ndarray:
    """x: float [..., 576] -> uint8 [..., 594] (values then scales)."""
    x = np.asarray(x, dtype=np.float64)
    lead = x.shape[:-1]
    g = x.reshape(*lead, N_GROUPS, GROUP)
    amax = np.abs(g).max(axis=-1)
    mant, ex = np.frexp(amax / E4M3_MAX)   # amax/448 = mant * 2**ex
    # ceil(log2(y)) exactly: ex if mant > 0.5 else ex - 1
    e = np.where(mant > 0.5, ex, ex - 1)
    e = np.clip(e, -127, 127)
    zero = amax == 0
    e = np.where(zero, -127, e)
    scaled = g / np.ldexp(1.0, e)[..., None]
    vals = _round_to_e4m3(scaled)
    vals = np.where(zero[..., None], 0.0, vals)
    codes = _f64_to_e4m3_code(vals).reshape(*lead, D_QK)
    scale_bytes = (e + 127).astype(np.uint8)
    return np.concatenate([codes, scale_bytes], axis=-1)


def quantize_pages(latent_f32: np.ndarray, slot_valid: np.ndarray, rng_seed: int = 0,
                   garbage: str = "finite", chunk_pages: int = 2048) -> np.ndarray:
    """Quantise a float cache [num_pages, P, 576] into the paged FP8 layout
    uint8 [num_pages, P * 594].  Slots without a live token get garbage bytes:
    random finite codes ("finite") or e4m3 NaN with scale 0x7F ("nan")."""
    num_pages, P, _ = latent_f32.shape
    out = np.empty((num_pages, P, ROW_BYTES), dtype=np.uint8)
    for s in range(0, num_pages, chunk_pages):
        e = min(num_pages, s + chunk_pages)
        x = np.where(slot_valid[s:e, :, None], latent_f32[s:e], 0.0)
        out[s:e] = quantize_rows(x)
    inv = ~slot_valid
    if inv.any():
        n = int(inv.sum())
        if garbage == "nan":
            fill = np.full((n, ROW_BYTES), 0x7F, dtype=np.uint8)
        else:
            rng = np.random.default_rng(rng_seed + 7919)
            fill = rng.integers(0, 0x7F, size=(n, ROW_BYTES), dtype=np.uint8)
            fill[:, :D_QK] |= (rng.integers(0, 2, size=(n, D_QK), dtype=np.uint8) << 7)
            fill[:, D_QK:] = rng.integers(120, 134, size=(n, N_GROUPS), dtype=np.uint8)
        out[inv] = fill
    return out.reshape(num_pages, P * ROW_BYTES)
