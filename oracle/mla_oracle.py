"""CPU oracle for paged MLA latent-cache decode.

TEST INFRASTRUCTURE ONLY.  Plain, slow, float64 numpy.  Only the test suite,
the smoke check and the benchmark's CPU-baseline leg may import this module;
the product path (the CUDA library and its Python binding) never does, and
this module imports nothing from the product path.

What it computes (per request b, query token j, head h) is the plain,
NON-absorbed definition of MLA decode attention:

  1. Each visible cached token t holds a shared latent c_kv[t] (512) and a
     decoupled, already-rotated RoPE key k_rope[t] (64); the cache is the
     shared low-rank latent plus the RoPE key, not per-head K/V
     (GLM-4.7-Flash record, phantomic12 inference-research: the
     "serviceability join" paragraph on the MLA family and the MLA
     configuration clause: kv_lora_rank 512, qk_rope_head_dim 64,
     qk_nope_head_dim 192, v_head_dim 256).
  2. Decompress per head with the kv_b_proj up-projections (same record,
     "kv_a_proj_with_mqa and kv_b_proj"): k_nope[t] = W_UK[h]^T c_kv[t] (192),
     v[t] = W_UV[h]^T c_kv[t] (256).
  3. Query q = [q_nope (192) || q_rope (64)]; key k[t] = [k_nope[t] || k_rope[t]]
     (the 256-wide query head is 192 + 64, same record, head_dim paragraph),
     score s_t = sm_scale * q . k[t] with sm_scale = 1/sqrt(256).
  4. lse = ln sum_t exp(s_t);  o = sum_t exp(s_t - lse) v[t];  the latent-space
     output is o_lat = sum_t exp(s_t - lse) c_kv[t], so that o = W_UV[h]^T o_lat.

The visible set of tokens (readings of the pages, stated where they apply):
  * dense, one query token: positions 0 .. T_b - 1;
  * dense or sparse with q_len Q draft tokens, causal: draft j (0-based) sees
    positions 0 .. T_b - Q + j (the context length includes the drafts);
  * sparse: the positions listed in that query token's top-k row, one list per
    query token shared by all heads, with -1 slots masked (vllm API docs,
    vllm.models.glm5next.common.model, Glm5NextModel.__init__: the top-k
    buffer is padded to 128-column tiles and padded slots stay masked).
    Entries outside the visible window are masked too.
  * an empty visible set gives o = 0, o_lat = 0, lse = -inf.

Logical position t of request b lives at physical page block_table[b, t // P],
slot t % P, where P is the page size (64 or 128: fix: Add glm4_moe_lite to MLA
detection, the note on CUTLASS_MLA enforcing block_size=128; GLM-4.7-Flash
record: the decode kernels are built per KV-cache page-block size and a
planner fixes 64).

An independent ABSORBED form (q_lat = W_UK[h] q_nope, scores against the
576-wide cached row, output accumulated in latent space and up-projected by
W_UV) is provided as a cross-check; the two agree by associativity.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence

import numpy as np

from . import fp4 as _fp4
from . import fp8 as _fp8

D_C, D_R, D_NOPE, D_V = 512, 64, 192, 256
D_QK = D_C + D_R
N_LAYERS = 47
BYTES_BF16 = 2
SPARSE_TILE_COLUMNS = 128


# ----------------------------------------------------------------------------
# closed forms
# ----------------------------------------------------------------------------
def kv_cache_bytes_per_token(n_layers: int = N_LAYERS, kv_lora_rank: int = D_C,
                             rope_dim: int = D_R, bytes_per_elem: int = BYTES_BF16) -> int:
    """GLM-4.7-Flash record, KV-cache clause: layers x (kv_lora_rank +
    qk_rope_head_dim) x bytes per element."""
    return n_layers * (kv_lora_rank + rope_dim) * bytes_per_elem


def topk_buffer_width(topk: int, kpool: int = 1) -> int:
    """Width of the per-token top-k index buffer (vllm API docs,
    vllm.models.glm5next.common.model, Glm5NextModel.__init__): room for the
    incomplete pool tail when kpool > 1, rounded up to 128-column tiles."""
    width = topk + (kpool - 1 if kpool > 1 else 0)
    return ((width + SPARSE_TILE_COLUMNS - 1) // SPARSE_TILE_COLUMNS) * SPARSE_TILE_COLUMNS


# ----------------------------------------------------------------------------
# dtype decoding (own implementations; no shared code with the CUDA path)
# ----------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even), returned
    as float64.  Used where the compared output is stored as bf16."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                     # x = m * 2**e, 0.5 <= |m| < 1
    # bf16 keeps 8 significant bits; normal range down to 2**-126
    e_eff = np.maximum(e, -125)
    q = np.ldexp(1.0, e_eff - 8)
    with np.errstate(invalid="ignore"):
        return np.where(np.isfinite(x) & (x != 0), np.round(x / q) * q, x)


# ----------------------------------------------------------------------------
# paged addressing (bit-exact integer work)
# ----------------------------------------------------------------------------
def physical_rows(block_table_row: np.ndarray, positions: np.ndarray,
                  page_size: int) -> tuple[np.ndarray, np.ndarray]:
    """Map logical positions of one request to (physical page, slot)."""
    positions = np.asarray(positions, dtype=np.int64)
    pages = np.asarray(block_table_row, dtype=np.int64)[positions // page_size]
    slots = positions % page_size
    return pages, slots


def visible_positions(seq_len: int, q_len: int, j: int, causal: bool = True,
                      topk_row: Optional[np.ndarray] = None) -> np.ndarray:
    """Logical positions query token j of a request attends to, in the order
    they are summed (dense: ascending; sparse: the row's order)."""
    hi = seq_len - q_len + j + 1 if causal else seq_len   # exclusive bound
    hi = max(0, min(hi, seq_len))
    if topk_row is None:
        return np.arange(hi, dtype=np.int64)
    row = np.asarray(topk_row, dtype=np.int64)
    keep = (row >= 0) & (row < hi)
    return row[keep]


def gather_rows(batch_cache: np.ndarray, pages: np.ndarray, slots: np.ndarray) -> np.ndarray:
    return batch_cache[pages, slots]


# ----------------------------------------------------------------------------
# attention over one (request, query token): non-absorbed and absorbed forms
# ----------------------------------------------------------------------------
def attend_non_absorbed(q_nope: np.ndarray, q_rope: np.ndarray, w_uk: np.ndarray,
                        w_uv: np.ndarray, c_kv: np.ndarray, k_rope: np.ndarray,
                        sm_scale: float):
    """q_nope [H, Dn], q_rope [H, Dr], w_uk [H, Dc, Dn], w_uv [H, Dc, Dv],
    c_kv [n, Dc], k_rope [n, Dr]  ->  o [H, Dv], lse [H], o_lat [H, Dc]."""
    H = q_nope.shape[0]
    n = c_kv.shape[0]
    Dc, Dv = w_uv.shape[1], w_uv.shape[2]
    o = np.zeros((H, Dv))
    o_lat = np.zeros((H, Dc))
    lse = np.full(H, -np.inf)
    if n == 0:
        return o, lse, o_lat
    for h in range(H):
        k_nope = c_kv @ w_uk[h]                       # [n, Dn] = (W_UK^T c)^T
        v = c_kv @ w_uv[h]                            # [n, Dv]
        s = (k_nope @ q_nope[h] + k_rope @ q_rope[h]) * sm_scale
        m = s.max()
        lse[h] = m + math.log(np.exp(s - m).sum())
        p = np.exp(s - lse[h])
        o[h] = p @ v
        o_lat[h] = p @ c_kv
    return o, lse, o_lat


def absorb_query(q_nope: np.ndarray, w_uk: np.ndarray) -> np.ndarray:
    """q_lat[h] = W_UK[h] q_nope[h]  (latent-space query, [H, Dc])."""
    return np.einsum("hcn,hn->hc", w_uk, q_nope)


def attend_absorbed(q_lat: np.ndarray, q_rope: np.ndarray, w_uv: np.ndarray,
                    c_kv: np.ndarray, k_rope: np.ndarray, sm_scale: float):
    """Absorbed form: scores against [c_kv || k_rope] with [q_lat || q_rope],
    accumulate in latent space, then up-project with W_UV."""
    H = q_lat.shape[0]
    n = c_kv.shape[0]
    Dc, Dv = w_uv.shape[1], w_uv.shape[2]
    if n == 0:
        return np.zeros((H, Dv)), np.full(H, -np.inf), np.zeros((H, Dc))
    row = np.concatenate([c_kv, k_rope], axis=1)           # [n, Dc + Dr]
    q_hat = np.concatenate([q_lat, q_rope], axis=1)        # [H, Dc + Dr]
    s = (q_hat @ row.T) * sm_scale                          # [H, n]
    m = s.max(axis=1, keepdims=True)
    lse = (m + np.log(np.exp(s - m).sum(axis=1, keepdims=True)))[:, 0]
    p = np.exp(s - lse[:, None])
    o_lat = p @ c_kv
    o = np.einsum("hc,hcv->hv", o_lat, w_uv)
    return o, lse, o_lat


def combine_partials(o_parts: Sequence[np.ndarray], lse_parts: Sequence[np.ndarray]):
    """Merge attention results over disjoint token subsets: lse = ln sum_i
    exp(lse_i); o = sum_i exp(lse_i - lse) o_i (subsets with lse_i = -inf
    contribute nothing)."""
    lse_parts = [np.asarray(l, dtype=np.float64) for l in lse_parts]
    stack = np.stack(lse_parts)
    m = np.max(stack, axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.exp(stack - m_safe)                 # exp(-inf) = 0
    tot = w.sum(axis=0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, tot, 1.0)), -np.inf)
    o = np.zeros_like(np.asarray(o_parts[0], dtype=np.float64))
    for oi, li in zip(o_parts, lse_parts):
        wi = np.where(finite, np.exp(li - np.where(finite, lse, 0.0)), 0.0)
        o = o + wi[..., None] * oi
    return o, lse


# ----------------------------------------------------------------------------
# whole-batch driver
# ----------------------------------------------------------------------------
def cache_rows_f64(batch, pages: np.ndarray, slots: np.ndarray) -> np.ndarray:
    """Cached rows [n, 576] in float64 for the given physical locations:
    bf16 decoded, or FP8 / FP4 dequantised from the exact bytes the GPU reads
    (``batch.extra['cache_fp8']``, uint8 [num_pages, P * 594];
    ``batch.extra['cache_fp4']``, uint8 [num_pages, P * 324])."""
    w = batch.workload
    if w.kv_dtype == "bf16":
        return bf16_to_f64(batch.cache_bf16[pages, slots])
    if w.kv_dtype == "fp4":
        raw = batch.extra["cache_fp4"]
        rows = raw.reshape(raw.shape[0], w.page_size, _fp4.ROW_BYTES)[pages, slots]
        return _fp4.dequant_rows(rows)
    raw = batch.extra["cache_fp8"]
    rows = raw.reshape(raw.shape[0], w.page_size, _fp8.ROW_BYTES)[pages, slots]
    return _fp8.dequant_rows(rows)


def decode(batch, requests: Optional[Iterable[int]] = None,
           heads: Optional[Sequence[int]] = None, form: str = "non_absorbed",
           q_hat: Optional[np.ndarray] = None):
    """Run the oracle over (a subset of) a batch.

    form "non_absorbed" (the definition) or "absorbed" (the cross-check).
    q_hat: optional float64 [B, Q, H, 576] absorbed query to attend with
    directly (absorbed form), e.g. one already rounded to bf16.

    Returns dict (b, j) -> (o [h, 256], lse [h], o_lat [h, 512]) for the
    requested heads (default all)."""
    w = batch.workload
    P = w.page_size
    H = w.heads
    heads = list(range(H)) if heads is None else list(heads)
    w_uk = bf16_to_f64(batch.w_uk)[heads]
    w_uv = bf16_to_f64(batch.w_uv)[heads]
    out = {}
    reqs = range(w.batch) if requests is None else requests
    for b in reqs:
        T = int(batch.seq_lens[b])
        for j in range(w.q_len):
            topk_row = None if not w.topk else batch.topk_idx[b * w.q_len + j]
            pos = visible_positions(T, w.q_len, j, causal=w.causal, topk_row=topk_row)
            pages, slots = physical_rows(batch.block_table[b], pos, P)
            rows = cache_rows_f64(batch, pages, slots)
            c_kv, k_rope = rows[:, :D_C], rows[:, D_C:]
            qn = bf16_to_f64(batch.q_nope[b, j])[heads]
            qr = bf16_to_f64(batch.q_rope[b, j])[heads]
            if q_hat is not None:
                qh = np.asarray(q_hat[b, j], dtype=np.float64)[heads]
                res = attend_absorbed(qh[:, :D_C], qh[:, D_C:], w_uv, c_kv, k_rope, w.sm_scale)
            elif form == "non_absorbed":
                res = attend_non_absorbed(qn, qr, w_uk, w_uv, c_kv, k_rope, w.sm_scale)
            else:
                res = attend_absorbed(absorb_query(qn, w_uk), qr, w_uv, c_kv, k_rope,
                                      w.sm_scale)
            out[(b, j)] = res
    return out
