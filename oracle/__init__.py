"""CPU oracle for paged MLA latent-cache decode (TEST INFRASTRUCTURE ONLY).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU
baseline leg may import this package.  It shares no code with the CUDA path.
"""
from . import cache_append, fp4, fp8, rope
from .mla_oracle import (
    D_C, D_R, D_NOPE, D_V, D_QK, N_LAYERS,
    absorb_query, attend_absorbed, attend_non_absorbed, bf16_to_f64,
    combine_partials, decode, kv_cache_bytes_per_token, physical_rows,
    round_to_bf16, topk_buffer_width, visible_positions,
)
