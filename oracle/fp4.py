"""FP4 latent-cache encoding for the CPU oracle (TEST INFRASTRUCTURE ONLY).

Source (GLM-4.7-Flash record, phantomic12 inference-research, engine-kernel
constraint (2) on FlashMLA): next to the FP8 latent with per-token inlined
e8m0 scales, the decode kernel takes an FP4 latent at 288 bytes per token for
a 512-value row.  The record gives only that byte count.  Reading: 512 FP4
values take 256 bytes, so 32 bytes remain for scales, i.e. one scale byte per
16 values, and the scales are the FP8 variant's float8_e8m0, inlined after
the values of the same token.  For this build's 576-value rows (512 latent +
64 RoPE, all quantised like the FP8 variant):

    token row = 288 bytes of packed e2m1 codes || 36 e8m0 bytes   (324 bytes)

Value 2i of the row sits in the low nibble of code byte i and value 2i+1 in
its high nibble (the packing order of the OCP microscaling formats).  Group g
covers values [16 g, 16 g + 16); scale byte g belongs to group g.  A page of
P tokens is P contiguous rows (P * 324 bytes).

Value decoding, OCP 4-bit float e2m1: a sign bit, 2 exponent bits (bias 1)
and 1 mantissa bit; exponent 0 is subnormal (m/2); there is no infinity and
no NaN, so the magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4 and 6.  e8m0 as for the
FP8 variant: value 2**(byte - 127), 0xFF is NaN.  A cached value is
e2m1(code) * 2**(scale - 127).

Quantiser (data generation and the cache-append oracle, not on the decode
path), read like the FP8 one: e = clamp(ceil(log2(amax / 6)), -127, 127),
scale byte e + 127; values x / 2**e rounded to the nearest e2m1 value with
ties to the even code, saturating at +-6; an all-zero group gets scale byte
0 and zero codes.  The sign of a value that rounds to zero is kept (code 8
for negative inputs).
"""
from __future__ import annotations

import numpy as np

D_QK = 576
GROUP = 16
N_GROUPS = D_QK // GROUP          # 36
CODE_BYTES = D_QK // 2            # 288
ROW_BYTES = CODE_BYTES + N_GROUPS  # 324
E2M1_MAX = 6.0


def e2m1_to_f64(code: np.ndarray) -> np.ndarray:
    """4-bit codes (0..15, any integer dtype) -> float64 values."""
    c = np.asarray(code).astype(np.int64) & 0xF
    sign = np.where(c & 0x8, -1.0, 1.0)
    exp = (c >> 1) & 0x3
    man = c & 0x1
    val = np.where(exp == 0, man * 0.5, np.ldexp(1.0 + man / 2.0, exp - 1))
    return sign * val


def e8m0_to_f64(code: np.ndarray) -> np.ndarray:
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    return np.where(c == 0xFF, np.nan, np.ldexp(1.0, c - 127))


def unpack_codes(code_bytes: np.ndarray) -> np.ndarray:
    """uint8 [..., n] packed bytes -> uint8 [..., 2n] codes, low nibble first."""
    b = np.asarray(code_bytes, dtype=np.uint8)
    out = np.empty(b.shape[:-1] + (2 * b.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = b & 0xF
    out[..., 1::2] = b >> 4
    return out


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """uint8 [..., 2n] codes (0..15) -> uint8 [..., n], value 2i in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def dequant_rows(rows: np.ndarray) -> np.ndarray:
    """rows: uint8 [..., 324] -> float64 [..., 576] = e2m1 * 2**(s - 127)."""
    rows = np.asarray(rows, dtype=np.uint8)
    vals = e2m1_to_f64(unpack_codes(rows[..., :CODE_BYTES]))
    scales = e8m0_to_f64(rows[..., CODE_BYTES:])
    return vals * np.repeat(scales, GROUP, axis=-1)


def _round_to_e2m1(v: np.ndarray) -> np.ndarray:
    """Nearest e2m1 value (ties to the even code), saturating at +-6.

    The e2m1 grid has spacing 0.5 below 2, 1 in [2, 4) and 2 in [4, 8), and
    consecutive codes alternate between even and odd mantissa, so rounding
    |v| / spacing half-to-even is rounding to the even code."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    q = np.where(a < 2.0, 0.5, np.where(a < 4.0, 1.0, 2.0))
    r = np.minimum(np.round(a / q) * q, E2M1_MAX)
    return np.copysign(r, v)


def _f64_to_e2m1_code(v: np.ndarray) -> np.ndarray:
    """Codes of values already on the e2m1 grid (sign taken from the sign bit)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    mag = np.searchsorted(grid, a).astype(np.uint8)
    assert np.all(grid[np.minimum(mag, 7)] == a), "value not on the e2m1 grid"
    return mag | (np.signbit(v).astype(np.uint8) << 3)


def quantize_rows(x: np.ndarray) -> np.ndarray:
    """x: float [..., 576] -> uint8 [..., 324] (packed codes then scales)."""
    x = np.asarray(x, dtype=np.float64)
    lead = x.shape[:-1]
    g = x.reshape(*lead, N_GROUPS, GROUP)
    amax = np.abs(g).max(axis=-1)
    mant, ex = np.frexp(amax / E2M1_MAX)   # amax / 6 = mant * 2**ex, mant in [0.5, 1)
    e = np.where(mant > 0.5, ex, ex - 1)   # ceil(log2(amax / 6)), exactly
    e = np.clip(e, -127, 127)
    zero = amax == 0
    e = np.where(zero, -127, e)
    vals = _round_to_e2m1(g / np.ldexp(1.0, e)[..., None])
    codes = _f64_to_e2m1_code(vals)
    codes = np.where(zero[..., None], 0, codes).astype(np.uint8).reshape(*lead, D_QK)
    return np.concatenate([pack_codes(codes), (e + 127).astype(np.uint8)], axis=-1)


def quantize_pages(latent_f32: np.ndarray, slot_valid: np.ndarray, rng_seed: int = 0,
                   garbage: str = "finite", chunk_pages: int = 2048) -> np.ndarray:
    """Quantise a float cache [num_pages, P, 576] into the paged FP4 layout
    uint8 [num_pages, P * 324].  Slots without a live token get garbage bytes:
    random codes with scales up to 2**7 ("finite") or the e8m0 NaN scale
    byte 0xFF ("nan")."""
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
            fill = np.full((n, ROW_BYTES), 0xFF, dtype=np.uint8)
        else:
            rng = np.random.default_rng(rng_seed + 7919)
            fill = rng.integers(0, 256, size=(n, ROW_BYTES), dtype=np.uint8)
            fill[:, CODE_BYTES:] = rng.integers(120, 135, size=(n, N_GROUPS), dtype=np.uint8)
        out[inv] = fill
    return out.reshape(num_pages, P * ROW_BYTES)
