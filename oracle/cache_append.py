"""Oracle for appending a decode step's new token to the paged latent cache
(TEST INFRASTRUCTURE ONLY: tests, the smoke check and the benchmark's CPU leg).

Each request's newest token brings one cached row: its 512-dim latent c_kv
and its 64-dim RoPE key (the pages' cache holds the shared latent plus the
decoupled RoPE key: GLM-4.7-Flash record, phantomic12 inference-research,
the MLA configuration clause; the cache-writing step with an on-GPU FP8
quantiser is named among the engine-kernel constraints of the same record).
The row goes to logical position pos of its request, i.e. physical page
block_table[b, pos // P], slot pos % P.

With rope_theta > 0 the RoPE key is first rotated to position pos
(oracle.rope.rope_rotate, float64, rope_theta 1000000 in the same record's
configuration clause) and rounded to bf16, the type of the row it came in;
with rope_theta = 0 it is taken as already rotated.

  * bf16 cache: the row's 576 bf16 values are stored as they are.
  * FP8 cache (576 e4m3 || 18 e8m0 per token): every 32-value group is
    quantised with the oracle's quantiser (oracle.fp8.quantize_rows: scale
    2^e with e = ceil(log2(amax / 448)) clamped to [-127, 127], values
    rounded to nearest-even e4m3 of x / 2^e, saturating at 448; an all-zero
    group gets scale byte 0 and zero codes).
  * FP4 cache (288 bytes of packed e2m1 || 36 e8m0 per token): every
    16-value group is quantised with oracle.fp4.quantize_rows (e =
    ceil(log2(amax / 6)) clamped to [-127, 127], values rounded to the nearest
    e2m1 value with ties to the even code).

A position of -1 appends nothing for that request.  A position outside the
request's pages or a page id outside the pool appends nothing either (the
CUDA path reports it in its status word).
"""
from __future__ import annotations

import numpy as np

from . import fp4 as _fp4
from . import fp8 as _fp8
from . import rope as _rope
from .mla_oracle import bf16_to_f64, round_to_bf16

D_QK = 576


def _f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Nearest bf16 (ties to even) of float64 values, as bit patterns."""
    r = round_to_bf16(x).astype(np.float32)       # exact: r has 8 significant bits
    return (r.view(np.uint32) >> 16).astype(np.uint16)


def rotate_row(row_bf16: np.ndarray, pos: int, rope_theta: float) -> np.ndarray:
    """The cached form of one new row (bf16 bits [576]): its last 64 values
    rotated to position pos and rounded to bf16 when rope_theta > 0."""
    row = np.array(row_bf16, dtype=np.uint16, copy=True)
    if rope_theta > 0:
        k = bf16_to_f64(row[D_QK - _rope.ROPE_DIM:])
        row[D_QK - _rope.ROPE_DIM:] = _f64_to_bf16_bits(_rope.rope_rotate(k, pos, rope_theta))
    return row


def append_rows(cache: np.ndarray, rows_bf16: np.ndarray, positions: np.ndarray,
                block_table: np.ndarray, page_size: int, kv_dtype: str,
                rope_theta: float = 0.0) -> np.ndarray:
    """Return a copy of `cache` with row b of `rows_bf16` (uint16 bf16 bits,
    [B, 576]) written at logical position positions[b] of request b.

    cache: bf16 bits uint16 [num_pages, P, 576], FP8 bytes uint8
    [num_pages, P * 594] or FP4 bytes uint8 [num_pages, P * 324]."""
    out = np.array(cache, copy=True)
    num_pages = out.shape[0]
    max_pages = block_table.shape[1]
    for b, pos in enumerate(np.asarray(positions, dtype=np.int64)):
        if pos < 0 or pos >= max_pages * page_size:
            continue
        page = int(block_table[b, pos // page_size])
        if page < 0 or page >= num_pages:
            continue
        slot = int(pos % page_size)
        row = rotate_row(rows_bf16[b], int(pos), rope_theta)
        if kv_dtype == "bf16":
            out[page, slot, :] = row
        else:
            x = (row.astype(np.uint32) << 16).view(np.float32)
            enc = _fp4 if kv_dtype == "fp4" else _fp8
            row = enc.quantize_rows(x.astype(np.float64)[None, :])[0]
            out[page, slot * enc.ROW_BYTES:(slot + 1) * enc.ROW_BYTES] = row
    return out
