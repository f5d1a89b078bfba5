"""Device buffers for one decode step, allocated with torch, and the C-ABI
calls in order (torch is plumbing here: memory and streams only)."""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import (MLA_KV_BF16, MLA_KV_FP4_E2M1_E8M0, MLA_KV_FP8_E4M3_E8M0, make_problem, mla_clear_status, mla_combine,
               mla_decode_plan, mla_decode_run, mla_get_status, mla_q_absorb, mla_uv_proj)


def to_device_bf16(bits: np.ndarray, device) -> torch.Tensor:
    """uint16 bf16 bit patterns -> torch.bfloat16 tensor on `device`."""
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(torch.bfloat16)


def to_device(arr: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)


class DecodeStep:
    """One layer's decode step over a paged latent cache.

    Inputs (numpy, host): q_nope/q_rope bf16 bits [B, Q, H, 192/64],
    w_uk [H, 512, 192] and w_uv [H, 512, 256] bf16 bits, the cache (bf16 bits
    [num_pages, P, 576], FP8 bytes [num_pages, P*594] or FP4 bytes
    [num_pages, P*324]), block_table int32
    [B, max_pages], seq_lens int32 [B], optional topk_idx int32 [B*Q, width].
    """

    def __init__(self, *, q_nope, q_rope, w_uk, w_uv, cache, block_table, seq_lens,
                 page_size: int, kv_dtype: int = MLA_KV_BF16, topk_idx=None, causal: bool = True,
                 sm_scale: float = 1.0 / 16.0, sm_count: Optional[int] = None, device="cuda:0",
                 absorb_on_device: bool = True):
        self.device = torch.device(device)
        B, Q, H, _ = q_nope.shape
        self.B, self.Q, self.H = B, Q, H
        self.rows = B * Q
        if sm_count is None:
            sm_count = torch.cuda.get_device_properties(self.device).multi_processor_count
        num_pages = cache.shape[0]
        width = 0 if topk_idx is None else int(topk_idx.shape[1])
        self.problem = make_problem(B, Q, H, page_size, num_pages, int(block_table.shape[1]),
                                    kv_dtype=kv_dtype, topk_width=width, causal=int(causal),
                                    sm_scale=sm_scale)
        self.plan = mla_decode_plan(self.problem, seq_lens, sm_count)
        dev = self.device
        self.q_nope = to_device_bf16(q_nope, dev)
        self.q_rope = to_device_bf16(q_rope, dev)
        self.w_uk = to_device_bf16(w_uk, dev)
        self.w_uv = to_device_bf16(w_uv, dev)
        if kv_dtype in (MLA_KV_FP8_E4M3_E8M0, MLA_KV_FP4_E2M1_E8M0):
            self.cache = to_device(cache.astype(np.uint8, copy=False), dev)
        else:
            self.cache = to_device_bf16(cache, dev)
        self.block_table = to_device(block_table.astype(np.int32, copy=False), dev)
        self.seq_lens = to_device(np.asarray(seq_lens, dtype=np.int32), dev)
        self.topk_idx = None if topk_idx is None else to_device(topk_idx.astype(np.int32, copy=False), dev)
        self.workspace = torch.zeros(int(self.plan.workspace_bytes), dtype=torch.uint8, device=dev)
        self.q_hat = torch.empty((self.rows, H, 576), dtype=torch.bfloat16, device=dev)
        self.o_lat = torch.empty((self.rows, H, 512), dtype=torch.float32, device=dev)
        self.lse = torch.empty((self.rows, H), dtype=torch.float32, device=dev)
        self.out = torch.empty((self.rows, H, 256), dtype=torch.bfloat16, device=dev)
        if absorb_on_device:
            self.absorb()

    @property
    def stream(self):
        return torch.cuda.current_stream(self.device)

    def absorb(self):
        mla_q_absorb(self.plan, self.q_nope, self.q_rope, self.w_uk, self.q_hat, self.stream)

    def run(self):
        """Attention pass and the split merge (two kernels, the second a
        programmatic dependent of the first): writes o_lat and lse."""
        mla_decode_run(self.plan, self.q_hat, self.cache, self.block_table, self.seq_lens,
                       self.topk_idx, self.workspace, self.o_lat, self.lse, self.stream)

    def combine(self):
        """Re-run the split merge from the partials left in the workspace."""
        mla_combine(self.plan, self.seq_lens, self.workspace, self.o_lat, self.lse, self.stream)

    def uv(self):
        mla_uv_proj(self.o_lat, self.w_uv, self.out, self.rows, self.H, self.stream)

    def step(self):
        """Attention pass, split merge and W_UV projection; the absorbed
        query is an input."""
        self.run()
        self.uv()

    def status(self) -> int:
        return mla_get_status(self.plan, self.workspace, self.stream)

    def clear_status(self):
        mla_clear_status(self.plan, self.workspace, self.stream)

    KERNELS_PER_STEP = 3
