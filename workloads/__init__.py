"""Seeded synthetic inputs for paged MLA latent-cache decode.

This module only draws random tensors with the shapes, sizes and value
distributions of the decode workloads.  It holds none of the attention
arithmetic (no query absorption, no scores, no softmax, no quantisation):
both the CUDA path (through the tests and the benchmark) and the CPU oracle
consume what it returns.

Geometry (GLM-4.7-Flash record, phantomic12 inference-research, the MLA
configuration clause): each cached token of one layer holds a 512-dim shared
latent c_kv (kv_lora_rank) and a 64-dim decoupled RoPE key; queries are split
into a 192-dim no-RoPE part and a 64-dim RoPE part; the value head is 256.

bf16 tensors are returned as uint16 bit patterns (numpy has no bfloat16).

FP8 caches (576 e4m3 codes then 18 e8m0 scale bytes per cached row) are drawn
directly as bytes: the decode's input is the byte layout, so no quantiser is
involved.  Live rows: ~99% of codes have a random sign, an exponent field
distributed as round(N(10, 0.75)) clipped to [0, 12] and a uniform 3-bit
mantissa, the other ~1% are uniform over the codes with exponent field <= 8
(zeros and subnormals included); scale bytes are uniform in [121, 124]
(2**-6 .. 2**-3), so live values have magnitudes around 0.5 and at most 7.5,
like the N(0, 1) bf16 cache.  FP4 caches (288 bytes of e2m1 codes, two per
byte with the even value in the low nibble, then 36 e8m0 scale bytes, one per
16 values) are drawn the same way: each code's magnitude index 0..7 (values
0, 0.5, 1, 1.5, 2, 3, 4, 6) with probabilities 12, 22, 20, 16, 14, 9, 5 and 2
percent and a random sign; scale bytes uniform in [125, 126] (2**-2, 2**-1),
so live values have magnitudes up to 3.  ``fp8_source="float"`` instead
returns a float32 latent for the oracle's quantisers (FP8 and FP4; small
cases only).

Draw order for one workload (one ``numpy.random.default_rng(seed)``):
seq_lens -> block table -> cache -> q_nope -> q_rope -> W_UK -> W_UV ->
sparse indices.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

D_C = 512      # kv_lora_rank: shared latent width
D_R = 64       # qk_rope_head_dim: decoupled RoPE key width
D_QK = D_C + D_R  # 576: one cached row
D_NOPE = 192   # qk_nope_head_dim
D_V = 256      # v_head_dim
N_LAYERS = 47  # GLM-4.7-Flash decoder layers
FP8_GROUP = 32                      # values per e8m0 scale
FP8_ROW_BYTES = D_QK + D_QK // FP8_GROUP  # 576 e4m3 + 18 e8m0 = 594
FP4_GROUP = 16                      # values per e8m0 scale (FP4 reading)
FP4_ROW_BYTES = D_QK // 2 + D_QK // FP4_GROUP  # 288 packed e2m1 + 36 e8m0 = 324

BF16_NAN = np.uint16(0x7FC0)


# ----------------------------------------------------------------------------
# bf16 bit-pattern conversion (a dtype cast, not part of the method)
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    out = (rounded >> np.uint32(16)).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = BF16_NAN
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# ----------------------------------------------------------------------------
# workloads
# ----------------------------------------------------------------------------
@dataclass(frozen=True)
class Workload:
    """One decode batch of one layer.

    seq_lens: explicit tuple, or drawn uniformly from [seq_lo, seq_hi]
    (integers, both ends inclusive).  For the sparse workload every request
    has the same context length ``seq_lo == seq_hi``.
    """

    name: str
    batch: int
    heads: int
    q_len: int = 1
    seq_lens: Optional[tuple] = None
    seq_lo: int = 0
    seq_hi: int = 0
    page_size: int = 64
    kv_dtype: str = "bf16"          # "bf16" | "fp8" | "fp4"
    topk: int = 0                   # 0 = dense
    topk_pad_slots: int = 0         # extra -1 slots (width = topk + pad)
    causal: bool = True             # draft tokens see their prefix only
    spare_frac: float = 0.10        # spare physical pages in the pool
    seed: int = 0
    sm_scale: float = 1.0 / 16.0    # 1/sqrt(192 + 64)

    @property
    def topk_width(self) -> int:
        return self.topk + self.topk_pad_slots if self.topk else 0

    @property
    def cache_row_bytes(self) -> int:
        return {"bf16": 2 * D_QK, "fp8": FP8_ROW_BYTES, "fp4": FP4_ROW_BYTES}[self.kv_dtype]


WORKLOADS = {
    # batch 2, H=4, seq_lens {37, 130}, page 64, random block table
    "tiny": Workload("tiny", batch=2, heads=4, seq_lens=(37, 130), page_size=64),
    # GLM-4.7-Flash-shaped dense decode: B=64, H=20, T~U[1024, 8192], page 64
    "dense": Workload("dense", batch=64, heads=20, seq_lo=1024, seq_hi=8192, page_size=64),
    # long-context split-KV: B=8, T~U[65536, 131072], page 128
    "long": Workload("long", batch=8, heads=20, seq_lo=65536, seq_hi=131072, page_size=128),
    # FP8 latent (e4m3 + e8m0 per 32): B=128, T~U[2048, 16384], page 64
    "fp8": Workload("fp8", batch=128, heads=20, seq_lo=2048, seq_hi=16384, page_size=64,
                    kv_dtype="fp8"),
    # sparse top-2048, q_len 4 causal drafts, context 65536, page 64
    "sparse": Workload("sparse", batch=32, heads=20, q_len=4, seq_lo=65536, seq_hi=65536,
                       page_size=64, topk=2048),
    # speculative verify: the dense workload with 2 causal draft tokens per
    # request (one MTP draft pair); both drafts share each staged page
    "mtp": Workload("mtp", batch=64, heads=20, q_len=2, seq_lo=1024, seq_hi=8192, page_size=64),
    # FP4 latent (e2m1 + e8m0 per 16), on the FP8 workload's shape
    "fp4": Workload("fp4", batch=128, heads=20, seq_lo=2048, seq_hi=16384, page_size=64,
                    kv_dtype="fp4"),
    # speculative verify over the FP8 cache: the FP8 workload with 2 causal
    # draft tokens per request, both drafts sharing each staged page
    "mtp_fp8": Workload("mtp_fp8", batch=128, heads=20, q_len=2, seq_lo=2048, seq_hi=16384,
                        page_size=64, kv_dtype="fp8"),
}

# Reduced sizes the oracle checks element by element: several tiles and a
# ragged tail per request, both page sizes, a forced split and padded slots.
SMALL_WORKLOADS = {
    "tiny": WORKLOADS["tiny"],
    "dense_small": Workload("dense_small", batch=5, heads=20, seq_lo=65, seq_hi=700,
                            page_size=64, seed=1),
    "long_small": Workload("long_small", batch=3, heads=20, seq_lo=2000, seq_hi=5000,
                           page_size=128, seed=2),
    "fp8_small": Workload("fp8_small", batch=4, heads=20, seq_lo=100, seq_hi=900,
                          page_size=64, kv_dtype="fp8", seed=3),
    "mtp_small": Workload("mtp_small", batch=4, heads=20, q_len=3, seq_lo=70, seq_hi=900,
                          page_size=64, seed=6),
    "fp4_small": Workload("fp4_small", batch=4, heads=20, seq_lo=100, seq_hi=900,
                          page_size=64, kv_dtype="fp4", seed=5),
    "sparse_small": Workload("sparse_small", batch=2, heads=20, q_len=4, seq_lo=1500,
                             seq_hi=1500, page_size=64, topk=256, topk_pad_slots=128,
                             seed=4),
}


def with_overrides(w: Workload, **kw) -> Workload:
    return replace(w, **kw)


def draw_seq_lens(w: Workload, rng: np.random.Generator) -> np.ndarray:
    if w.seq_lens is not None:
        return np.asarray(w.seq_lens, dtype=np.int32)
    return rng.integers(w.seq_lo, w.seq_hi, size=w.batch, endpoint=True).astype(np.int32)


def _normal_bf16(rng: np.random.Generator, shape, scale: float = 1.0,
                 chunk: int = 1 << 24) -> np.ndarray:
    """N(0, scale^2) drawn in float32 and rounded to bf16 bit patterns."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = rng.standard_normal(e - s, dtype=np.float32)
        if scale != 1.0:
            x *= np.float32(scale)
        out[s:e] = f32_to_bf16_bits(x)
    return out.reshape(shape)


def _normal_f32(rng: np.random.Generator, shape, chunk: int = 1 << 24) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = rng.standard_normal(e - s, dtype=np.float32)
    return out.reshape(shape)


@dataclass
class Batch:
    """Arrays of one decode batch (host, numpy)."""

    workload: Workload
    seq_lens: np.ndarray        # int32 [B]
    block_table: np.ndarray     # int32 [B, max_pages]; unused entries -1
    num_pages: int
    slot_valid: np.ndarray      # bool [num_pages, P]: holds a live token
    cache_bf16: Optional[np.ndarray]  # uint16 [num_pages, P, 576] (bf16 workloads)
    latent_f32: Optional[np.ndarray]  # float32 [num_pages, P, 576] (fp8_source="float" only)
    q_nope: np.ndarray          # uint16 bf16 [B, Q, H, 192]
    q_rope: np.ndarray          # uint16 bf16 [B, Q, H, 64]
    w_uk: np.ndarray            # uint16 bf16 [H, 512, 192]
    w_uv: np.ndarray            # uint16 bf16 [H, 512, 256]
    topk_idx: Optional[np.ndarray]  # int32 [B*Q, width]; -1 = masked slot
    extra: dict = field(default_factory=dict)

    @property
    def cache_fp8(self) -> Optional[np.ndarray]:
        """uint8 [num_pages, P * 594] FP8 cache bytes, if drawn."""
        return self.extra.get("cache_fp8")

    @property
    def cache_fp4(self) -> Optional[np.ndarray]:
        """uint8 [num_pages, P * 324] FP4 cache bytes, if drawn."""
        return self.extra.get("cache_fp4")

    @property
    def cache_quant(self) -> Optional[np.ndarray]:
        """The FP8 or FP4 cache bytes of a quantised workload."""
        return self.extra.get("cache_" + self.workload.kv_dtype)

    @property
    def latent_bytes_read(self) -> int:
        """Bytes of cached rows the decode must read (one row per visible token,
        per request for dense; per query token for sparse)."""
        w = self.workload
        if w.topk:
            valid = int((self.topk_idx >= 0).sum())
            return valid * w.cache_row_bytes
        return int(self.seq_lens.astype(np.int64).sum()) * w.cache_row_bytes


def _exponent_table() -> np.ndarray:
    """256-entry table: a uniform random byte -> an e4m3 exponent field with
    the probabilities of round(N(10, 0.75)) clipped to [0, 12]."""
    from math import erf, sqrt
    cdf = [0.5 * (1.0 + erf((e + 0.5 - 10.0) / (0.75 * sqrt(2.0)))) for e in range(12)] + [1.0]
    edges = np.rint(np.asarray(cdf) * 256).astype(np.int64)
    return np.searchsorted(edges, np.arange(256), side="right").clip(0, 12).astype(np.uint8)


_EXP_TABLE = _exponent_table()


def _fp8_rows(rng: np.random.Generator, n: int, chunk: int = 1 << 16) -> np.ndarray:
    """n live FP8 rows (uint8 [n, 594]) drawn as codes, as described above.
    One random 32-bit word per code: bits 0-7 pick the exponent field, 8-10
    the mantissa, 11 the sign; bits 12-19 below 3 (~1.2%) replace the code
    by the small code in bits 20-26 (taken modulo 0x48)."""
    out = np.empty((n, FP8_ROW_BYTES), dtype=np.uint8)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        m = e - s
        r = rng.integers(0, 1 << 32, size=(m, D_QK), dtype=np.uint32)
        exp = _EXP_TABLE[(r & 0xFF).astype(np.uint8)]
        man = ((r >> 8) & 7).astype(np.uint8)
        codes = (exp << 3) | man
        wild = ((r >> 12) & 0xFF) < 3
        small = (((r >> 20) & 0x7F) % 0x48).astype(np.uint8)
        codes = np.where(wild, small, codes)
        codes |= (((r >> 11) & 1).astype(np.uint8) << 7)
        out[s:e, :D_QK] = codes
        out[s:e, D_QK:] = rng.integers(121, 125, size=(m, D_QK // FP8_GROUP), dtype=np.uint8)
    return out


_FP4_MAG_TABLE = np.searchsorted(
    np.rint(np.cumsum([12, 22, 20, 16, 14, 9, 5, 2]) * 2.56).astype(np.int64),
    np.arange(256), side="right").clip(0, 7).astype(np.uint8)


def _fp4_rows(rng: np.random.Generator, n: int, chunk: int = 1 << 16) -> np.ndarray:
    """n live FP4 rows (uint8 [n, 324]) drawn as codes, as described above.
    One random 16-bit word per code: bits 0-7 pick the magnitude index, bit 8
    the sign."""
    out = np.empty((n, FP4_ROW_BYTES), dtype=np.uint8)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        m = e - s
        r = rng.integers(0, 1 << 16, size=(m, D_QK), dtype=np.uint32)
        codes = _FP4_MAG_TABLE[(r & 0xFF).astype(np.uint8)] | (((r >> 8) & 1).astype(np.uint8) << 3)
        out[s:e, :D_QK // 2] = codes[:, 0::2] | (codes[:, 1::2] << 4)
        out[s:e, D_QK // 2:] = rng.integers(125, 127, size=(m, D_QK // FP4_GROUP), dtype=np.uint8)
    return out


def _fp4_garbage(rng: np.random.Generator, n: int, garbage: str) -> np.ndarray:
    if garbage == "nan":     # e8m0 NaN scale bytes make every value NaN
        return np.full((n, FP4_ROW_BYTES), 0xFF, dtype=np.uint8)
    out = rng.integers(0, 256, size=(n, FP4_ROW_BYTES), dtype=np.uint8)
    out[:, D_QK // 2:] = rng.integers(120, 135, size=(n, D_QK // FP4_GROUP), dtype=np.uint8)
    return out


def _fp8_garbage(rng: np.random.Generator, n: int, garbage: str) -> np.ndarray:
    if garbage == "nan":     # e4m3 NaN values, scale byte 0x7F
        return np.full((n, FP8_ROW_BYTES), 0x7F, dtype=np.uint8)
    out = rng.integers(0, 0x7F, size=(n, FP8_ROW_BYTES), dtype=np.uint8)
    out[:, :D_QK] |= rng.integers(0, 2, size=(n, D_QK), dtype=np.uint8) << 7
    out[:, D_QK:] = rng.integers(120, 135, size=(n, D_QK // FP8_GROUP), dtype=np.uint8)
    return out


def generate(w: Workload, garbage: str = "finite", fp8_source: str = "codes") -> Batch:
    """Draw one batch.  ``garbage`` fills slots that hold no live token (tail
    slots of a request's last page and spare pages): "finite" uses bf16 values
    of magnitude up to 1e4 (FP8 and FP4: random finite codes with scales up to
    2**7), "nan" uses NaN.  ``fp8_source`` ("codes" or "float", for FP8 and
    FP4 caches) is described in the module docstring."""
    rng = np.random.default_rng(w.seed)
    B, Q, H, P = w.batch, w.q_len, w.heads, w.page_size
    seq_lens = draw_seq_lens(w, rng)
    pages_per_req = (seq_lens.astype(np.int64) + P - 1) // P
    used = int(pages_per_req.sum())
    num_pages = max(1, int(np.ceil(used * (1.0 + w.spare_frac))))
    max_pages = max(1, int(pages_per_req.max()) if B else 1)
    perm = rng.permutation(num_pages).astype(np.int32)
    block_table = np.full((B, max_pages), -1, dtype=np.int32)
    slot_valid = np.zeros((num_pages, P), dtype=bool)
    cursor = 0
    for b in range(B):
        n = int(pages_per_req[b])
        block_table[b, :n] = perm[cursor:cursor + n]
        cursor += n
        for j in range(n):
            live = min(P, int(seq_lens[b]) - j * P)
            slot_valid[block_table[b, j], :live] = True

    cache_bf16 = latent_f32 = cache_q = None
    if w.kv_dtype == "bf16":
        cache_bf16 = _normal_bf16(rng, (num_pages, P, D_QK))
    elif fp8_source == "codes":
        draw = _fp8_rows if w.kv_dtype == "fp8" else _fp4_rows
        cache_q = draw(rng, num_pages * P).reshape(num_pages, P, w.cache_row_bytes)
    else:
        latent_f32 = _normal_f32(rng, (num_pages, P, D_QK))
    inv = ~slot_valid
    if cache_q is not None and inv.any():
        junk = _fp8_garbage if w.kv_dtype == "fp8" else _fp4_garbage
        cache_q[inv] = junk(rng, int(inv.sum()), garbage)
    elif inv.any():
        n_inv = int(inv.sum())
        if garbage == "nan":
            fill_bits = np.full((n_inv, D_QK), BF16_NAN, dtype=np.uint16)
            fill_f32 = np.full((n_inv, D_QK), np.nan, dtype=np.float32)
        else:
            fill_f32 = rng.uniform(-1e4, 1e4, size=(n_inv, D_QK)).astype(np.float32)
            fill_bits = f32_to_bf16_bits(fill_f32)
        if cache_bf16 is not None:
            cache_bf16[inv] = fill_bits
        else:
            latent_f32[inv] = fill_f32

    q_nope = _normal_bf16(rng, (B, Q, H, D_NOPE))
    q_rope = _normal_bf16(rng, (B, Q, H, D_R))
    w_uk = _normal_bf16(rng, (H, D_C, D_NOPE), scale=1.0 / np.sqrt(D_C))
    w_uv = _normal_bf16(rng, (H, D_C, D_V), scale=1.0 / np.sqrt(D_C))

    topk_idx = None
    if w.topk:
        width = w.topk_width
        topk_idx = np.full((B * Q, width), -1, dtype=np.int32)
        for b in range(B):
            for j in range(Q):
                window = int(seq_lens[b]) - Q + j + 1 if w.causal else int(seq_lens[b])
                k = min(w.topk, window)
                picks = rng.choice(window, size=k, replace=False).astype(np.int32)
                row = np.full(width, -1, dtype=np.int32)
                if w.topk_pad_slots:
                    slots = np.sort(rng.choice(width, size=k, replace=False))
                    row[slots] = picks
                else:
                    row[:k] = picks
                topk_idx[b * Q + j] = row

    batch = Batch(w, seq_lens, block_table, num_pages, slot_valid, cache_bf16, latent_f32,
                  q_nope, q_rope, w_uk, w_uv, topk_idx)
    if cache_q is not None:
        batch.extra["cache_" + w.kv_dtype] = cache_q.reshape(num_pages, P * w.cache_row_bytes)
    return batch
