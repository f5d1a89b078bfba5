"""Oracle for appending a decode step's new token to the paged latent cache
(TEST INFRASTRUCTURE ONLY: tests, the smoke check and the benchmark's CPU leg).

Each request's newest token brings one cached row: its 512-dim latent c_kv
and its 64-dim RoPE key, already rotated (the pages' cache holds the shared
latent plus the decoupled RoPE key: GLM-4.7-Flash record, phantomic12
inference-research, the MLA configuration clause; the cache-writing step
with an on-GPU FP8 quantiser is named among the engine-kernel constraints of
the same record).  The row goes to logical position pos of its request,
i.e. physical page block_table[b, pos // P], slot pos % P.

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

D_QK = 576


def append_rows(cache: np.ndarray, rows_bf16: np.ndarray, positions: np.ndarray,
                block_table: np.ndarray, page_size: int, kv_dtype: str) -> np.ndarray:
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
        if kv_dtype == "bf16":
            out[page, slot, :] = rows_bf16[b]
        else:
            x = (np.asarray(rows_bf16[b], dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
            enc = _fp4 if kv_dtype == "fp4" else _fp8
            row = enc.quantize_rows(x.astype(np.float64)[None, :])[0]
            out[page, slot * enc.ROW_BYTES:(slot + 1) * enc.ROW_BYTES] = row
    return out
