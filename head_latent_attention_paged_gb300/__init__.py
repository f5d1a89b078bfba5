"""Python binding of libmla_gb300.so (paged MLA latent-cache decode, sm_103a).

Argument marshalling only: every step of the decode runs in the library's
CUDA kernels.  Functions mirror the C ABI in include/mla_decode.h and take
device addresses as ints (or any object with ``data_ptr()``, e.g. a torch
tensor) and CUDA streams as ints (``torch.cuda.current_stream().cuda_stream``)
or None for the default stream.  There is no fallback: if the library cannot
be loaded every call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmla_gb300.so")

MLA_OK = 0
MLA_ERR_INVALID_ARGUMENT = -1
MLA_ERR_UNSUPPORTED = -2
MLA_ERR_MISALIGNED = -3
MLA_ERR_WORKSPACE_TOO_SMALL = -4
MLA_ERR_CUDA = -5

MLA_KV_BF16 = 0
MLA_KV_FP8_E4M3_E8M0 = 1
MLA_KV_FP4_E2M1_E8M0 = 2

MLA_STATUS_BAD_PAGE = 0x1
MLA_STATUS_BAD_INDEX = 0x2
MLA_STATUS_TIMEOUT = 0x4

MLA_TILE_TOKENS = 64

EXPORTED = (
    "mla_decode_plan", "mla_q_absorb", "mla_decode_run", "mla_combine", "mla_uv_proj",
    "mla_get_status", "mla_clear_status", "mla_strerror", "mla_version",
    "mla_decode_run_static", "mla_cache_append", "mla_selftest_bounded_wait", "mla_decode_step",
)


class MlaProblem(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("q_len", ctypes.c_int32), ("num_heads", ctypes.c_int32),
        ("kv_lora_rank", ctypes.c_int32), ("rope_dim", ctypes.c_int32),
        ("nope_dim", ctypes.c_int32), ("v_head_dim", ctypes.c_int32),
        ("page_size", ctypes.c_int32), ("num_pages", ctypes.c_int32),
        ("max_pages_per_seq", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
        ("topk_width", ctypes.c_int32), ("causal", ctypes.c_int32), ("sm_scale", ctypes.c_float),
    ]


class MlaPlan(ctypes.Structure):
    _fields_ = [
        ("problem", MlaProblem), ("num_streams", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
        ("num_slots", ctypes.c_int32), ("smem_bytes", ctypes.c_int32),
        ("ws_partial_o", ctypes.c_int64), ("ws_partial_lse", ctypes.c_int64),
        ("ws_prefix", ctypes.c_int64), ("ws_status", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_int64),
        ("planned_tiles", ctypes.c_int64), ("ws_q_hat", ctypes.c_int64),
        ("split_tokens", ctypes.c_int32), ("sm_count", ctypes.c_int32),
        ("prefix_pass", ctypes.c_int32), ("reserved", ctypes.c_int32 * 3),
    ]


class MlaError(RuntimeError):
    def __init__(self, fn: str, code: int):
        self.code = code
        super().__init__(f"{fn} failed: {code} ({strerror(code)})")


_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the shared library (once).  Raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    vp, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    P = ctypes.POINTER
    sz = ctypes.c_size_t
    lib.mla_decode_plan.argtypes = [P(MlaProblem), P(ctypes.c_int32), i32, i32, P(MlaPlan), P(sz)]
    lib.mla_q_absorb.argtypes = [P(MlaPlan), vp, vp, vp, vp]
    lib.mla_decode_run.argtypes = [P(MlaPlan), vp, vp, vp, vp, vp, vp, vp, sz, vp, vp, vp]
    lib.mla_combine.argtypes = [P(MlaPlan), vp, vp, sz, vp, vp, vp, vp, vp]
    lib.mla_decode_step.argtypes = [P(MlaPlan), vp, vp, vp, vp, vp, vp, vp, sz, vp, vp, vp, vp, vp]
    lib.mla_decode_run_static.argtypes = [P(MlaPlan), vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.mla_uv_proj.argtypes = [vp, vp, vp, i32, i32, vp]
    lib.mla_cache_append.argtypes = [P(MlaProblem), vp, vp, vp, ctypes.c_float, vp, vp, vp]
    lib.mla_selftest_bounded_wait.argtypes = [vp, i64, vp, vp]
    lib.mla_get_status.argtypes = [P(MlaPlan), vp, P(ctypes.c_uint32), vp]
    lib.mla_clear_status.argtypes = [P(MlaPlan), vp, vp]
    lib.mla_strerror.argtypes = [ctypes.c_int]
    lib.mla_strerror.restype = ctypes.c_char_p
    lib.mla_version.argtypes = []
    for name in EXPORTED:
        if name not in ("mla_strerror",):
            getattr(lib, name).restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    return int(x)


def _stream(s) -> Optional[int]:
    if s is None:
        return None
    if hasattr(s, "cuda_stream"):
        return int(s.cuda_stream)
    return int(s)


def _check(fn: str, rc: int) -> None:
    if rc != MLA_OK:
        raise MlaError(fn, rc)


def strerror(code: int) -> str:
    return load().mla_strerror(code).decode()


def version() -> int:
    return load().mla_version()


def make_problem(batch, q_len, num_heads, page_size, num_pages, max_pages_per_seq,
                 kv_dtype=MLA_KV_BF16, topk_width=0, causal=1, sm_scale=1.0 / 16.0,
                 kv_lora_rank=512, rope_dim=64, nope_dim=192, v_head_dim=256) -> MlaProblem:
    return MlaProblem(batch, q_len, num_heads, kv_lora_rank, rope_dim, nope_dim, v_head_dim,
                      page_size, num_pages, max_pages_per_seq, kv_dtype, topk_width, causal,
                      sm_scale)


def _nbytes(buf, given, plan) -> int:
    """Byte size of a device buffer: as given, else a tensor's size, else the
    plan's workspace size (a bare address carries no size)."""
    if given is not None:
        return int(given)
    if hasattr(buf, "numel") and hasattr(buf, "element_size"):
        return int(buf.numel()) * int(buf.element_size())
    return int(plan.workspace_bytes)


def mla_decode_plan(problem: MlaProblem, seq_lens_host=None, sm_count: int = 152,
                    split_tokens: int = 0) -> MlaPlan:
    plan = MlaPlan()
    ws = ctypes.c_size_t(0)
    arr = None
    if seq_lens_host is not None:
        arr = np.ascontiguousarray(seq_lens_host, dtype=np.int32)
        ptr = arr.ctypes.data_as(ctypes.POINTER(ctypes.c_int32))
    else:
        ptr = None
    _check("mla_decode_plan", load().mla_decode_plan(ctypes.byref(problem), ptr, int(sm_count),
                                                     int(split_tokens), ctypes.byref(plan),
                                                     ctypes.byref(ws)))
    assert ws.value == plan.workspace_bytes
    return plan


def mla_q_absorb(plan: MlaPlan, q, w_uk, q_hat, stream=None) -> None:
    """q_hat = [W_UK[h] q[..., :192] || q[..., 192:]] (q bf16 [B*Q][H][256])."""
    _check("mla_q_absorb", load().mla_q_absorb(ctypes.byref(plan), _ptr(q), _ptr(w_uk),
                                               _ptr(q_hat), _stream(stream)))


def mla_decode_run(plan: MlaPlan, q, w_uk, kv_cache, block_table, seq_lens, topk_idx, workspace,
                   o_lat, lse, stream=None, workspace_bytes=None) -> None:
    """The attention pass.  q is the absorbed q_hat (w_uk None) or the
    un-absorbed [q_nope || q_rope] with w_uk.  Split row sets are completed
    by mla_combine."""
    _check("mla_decode_run", load().mla_decode_run(
        ctypes.byref(plan), _ptr(q), _ptr(w_uk), _ptr(kv_cache), _ptr(block_table),
        _ptr(seq_lens), _ptr(topk_idx), _ptr(workspace), _nbytes(workspace, workspace_bytes, plan),
        _ptr(o_lat), _ptr(lse), _stream(stream)))


def mla_decode_run_static(plan: MlaPlan, q_hat, kv_cache, block_table, seq_lens, topk_idx,
                          o_lat, lse, status=None, stream=None) -> None:
    """mla_decode_run and the merge without a caller workspace: the scratch is
    the library's fixed 16 MiB device array (for callers that cannot
    allocate)."""
    _check("mla_decode_run_static", load().mla_decode_run_static(
        ctypes.byref(plan), _ptr(q_hat), _ptr(kv_cache), _ptr(block_table), _ptr(seq_lens),
        _ptr(topk_idx), _ptr(o_lat), _ptr(lse), _ptr(status), _stream(stream)))


def mla_combine(plan: MlaPlan, seq_lens, workspace, o_lat, lse, w_uv=None, out=None,
                stream=None, workspace_bytes=None) -> None:
    """Merge split row sets into o_lat / lse; with w_uv also out = W_UV^T o_lat
    (bf16 [B*Q][H][256]) in the same kernel."""
    _check("mla_combine", load().mla_combine(
        ctypes.byref(plan), _ptr(seq_lens), _ptr(workspace),
        _nbytes(workspace, workspace_bytes, plan), _ptr(w_uv), _ptr(o_lat), _ptr(lse), _ptr(out),
        _stream(stream)))


def mla_decode_step(plan: MlaPlan, q, w_uk, kv_cache, block_table, seq_lens, topk_idx, workspace,
                    w_uv, o_lat, lse, out, stream=None, workspace_bytes=None) -> None:
    """A whole decode step, mla_decode_run then mla_combine with W_UV: two
    kernels, the attention pass and then the merge of split row sets inside
    the W_UV projection (a programmatic dependent of the first)."""
    _check("mla_decode_step", load().mla_decode_step(
        ctypes.byref(plan), _ptr(q), _ptr(w_uk), _ptr(kv_cache), _ptr(block_table),
        _ptr(seq_lens), _ptr(topk_idx), _ptr(workspace), _nbytes(workspace, workspace_bytes, plan),
        _ptr(w_uv), _ptr(o_lat), _ptr(lse), _ptr(out), _stream(stream)))


def mla_cache_append(problem: MlaProblem, new_rows, positions, block_table, kv_cache,
                     status=None, stream=None, rope_theta: float = 0.0) -> None:
    """Write row b of new_rows (bf16 [batch][576]) at logical position
    positions[b] of request b (bf16 copy or on-GPU FP8 / FP4 quantisation);
    with rope_theta > 0 its RoPE key is rotated to that position first."""
    _check("mla_cache_append", load().mla_cache_append(
        ctypes.byref(problem), _ptr(new_rows), _ptr(positions), _ptr(block_table),
        float(rope_theta), _ptr(kv_cache), _ptr(status), _stream(stream)))


def mla_selftest_bounded_wait(status, limit_ns: int, waited_ns=None, stream=None) -> None:
    """Launch the bounded-wait self-test: a wait that nothing completes gives
    up after limit_ns and ORs MLA_STATUS_TIMEOUT into the device word status."""
    _check("mla_selftest_bounded_wait", load().mla_selftest_bounded_wait(
        _ptr(status), int(limit_ns), _ptr(waited_ns), _stream(stream)))


def mla_uv_proj(o_lat, w_uv, out, rows: int, num_heads: int, stream=None) -> None:
    _check("mla_uv_proj", load().mla_uv_proj(_ptr(o_lat), _ptr(w_uv), _ptr(out), int(rows),
                                             int(num_heads), _stream(stream)))


def mla_get_status(plan: MlaPlan, workspace, stream=None) -> int:
    bits = ctypes.c_uint32(0)
    _check("mla_get_status", load().mla_get_status(ctypes.byref(plan), _ptr(workspace),
                                                   ctypes.byref(bits), _stream(stream)))
    return int(bits.value)


def mla_clear_status(plan: MlaPlan, workspace, stream=None) -> None:
    _check("mla_clear_status", load().mla_clear_status(ctypes.byref(plan), _ptr(workspace),
                                                       _stream(stream)))
