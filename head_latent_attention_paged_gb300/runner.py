"""Device buffers for one decode step, allocated with torch, and the C-ABI
calls in order (torch is plumbing here: memory and streams only)."""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

from . import (MLA_KV_BF16, MLA_KV_FP4_E2M1_E8M0, MLA_KV_FP8_E4M3_E8M0, make_problem,
               mla_clear_status, mla_combine, mla_decode_plan, mla_decode_run, mla_decode_step,
               mla_get_status, mla_q_absorb, mla_uv_proj)


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
    [num_pages, P*324], or such a cache already on the device as a torch
    tensor), block_table int32
    [B, max_pages], seq_lens int32 [B], optional topk_idx int32 [B*Q, width].
    """

    def __init__(self, *, q_nope, q_rope, w_uk, w_uv, cache, block_table, seq_lens,
                 page_size: int, kv_dtype: int = MLA_KV_BF16, topk_idx=None, causal: bool = True,
                 sm_scale: float = 1.0 / 16.0, sm_count: Optional[int] = None, device="cuda:0",
                 absorb_on_device: bool = True, split_tokens: int = 0,
                 plan_with_host_lengths: bool = True):
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
        # the plan sizes its grid from the host lengths when given them (else
        # it fills every SM; the kernels derive the split from the device
        # lengths either way)
        self.plan = mla_decode_plan(self.problem, seq_lens if plan_with_host_lengths else None,
                                    sm_count, split_tokens)
        dev = self.device
        # the un-absorbed query, one [q_nope (192) || q_rope (64)] per head
        self.q = to_device_bf16(np.concatenate([q_nope, q_rope], axis=-1).reshape(B * Q, H, 256), dev)
        self.w_uk = to_device_bf16(w_uk, dev)
        self.w_uv = to_device_bf16(w_uv, dev)
        if isinstance(cache, torch.Tensor):          # already on the device
            self.cache = cache
        elif kv_dtype in (MLA_KV_FP8_E4M3_E8M0, MLA_KV_FP4_E2M1_E8M0):
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
        mla_q_absorb(self.plan, self.q, self.w_uk, self.q_hat, self.stream)

    def attend(self, w_uk=False):
        """The attention pass alone (mla_decode_run): rows of row sets held by
        one CTA are final, split ones wait in the workspace for combine().
        w_uk=True hands the library the un-absorbed query and W_UK instead of
        q_hat (it absorbs into the workspace first)."""
        if w_uk:
            mla_decode_run(self.plan, self.q, self.w_uk, self.cache, self.block_table,
                           self.seq_lens, self.topk_idx, self.workspace, self.o_lat, self.lse,
                           self.stream)
        else:
            mla_decode_run(self.plan, self.q_hat, None, self.cache, self.block_table,
                           self.seq_lens, self.topk_idx, self.workspace, self.o_lat, self.lse,
                           self.stream)

    def combine(self, uv: bool = False):
        """Merge split row sets (mla_combine); uv=True then also writes out =
        W_UV^T o_lat."""
        mla_combine(self.plan, self.seq_lens, self.workspace, self.o_lat, self.lse,
                    self.w_uv if uv else None, self.out if uv else None, self.stream)

    def run(self):
        """Attention pass and merge: o_lat and lse complete (two kernels, the
        second a programmatic dependent of the first)."""
        self.attend()
        self.combine()

    def uv(self):
        """W_UV as a pass of its own over o_lat (mla_uv_proj)."""
        mla_uv_proj(self.o_lat, self.w_uv, self.out, self.rows, self.H, self.stream)

    def step(self):
        """One decode step (mla_decode_step): the attention pass, then the
        merge of split row sets inside the W_UV projection (two kernels, the
        second a programmatic dependent of the first, behind a one-block
        prefix pre-pass when the row sets are many); the absorbed query is an
        input."""
        mla_decode_step(self.plan, self.q_hat, None, self.cache, self.block_table, self.seq_lens,
                        self.topk_idx, self.workspace, self.w_uv, self.o_lat, self.lse, self.out,
                        self.stream)

    def step_two_calls(self):
        """The same step as mla_decode_run then mla_combine with W_UV."""
        self.attend()
        self.combine(uv=True)

    def status(self) -> int:
        return mla_get_status(self.plan, self.workspace, self.stream)

    def clear_status(self):
        mla_clear_status(self.plan, self.workspace, self.stream)

    @property
    def kernels_per_step(self) -> int:
        """Kernels one step() launches: the decode, then the merge with W_UV,
        behind the prefix pre-pass when the plan has one."""
        return 2 + int(self.plan.prefix_pass)


class HostPipeline:
    """Host <-> device pipeline for a sequence of decode steps.

    Every step's inputs (the absorbed queries, the block table, the context
    lengths, the top-k lists, each request's newest token row and its
    position) live in one pinned host arena and go to the device in one copy;
    the step's outputs (o and lse) come back in one copy.  `depth` sets of
    arenas rotate, and the copies run on their own streams: the inputs of
    step k + 1 and the outputs of step k - 1 move while step k computes.
    Each step appends its newest token rows to the cache (mla_cache_append,
    RoPE applied to their keys when rope_theta > 0) and runs the whole decode
    step (mla_decode_step) on the compute stream.

    The caller refills host arena `k % depth` for step k only after
    `input_copied(k - depth)` has been synchronised (the static inputs of a
    benchmark need no refill).  `caches` optionally lists identical copies of
    the latent cache that consecutive steps take in turn (a benchmark uses
    two so that no step finds the previous one's cache lines in L2).  Each
    submitted step re-points the DecodeStep's input and output tensors (and
    its cache) at that step's arena views.
    """

    ALIGN = 256

    def __init__(self, step: DecodeStep, *, q_hat_bits, block_table, seq_lens, new_rows,
                 positions, topk_idx=None, depth: int = 2, caches=None, rope_theta: float = 0.0):
        self.step = step
        self.rope_theta = rope_theta
        self.depth = depth
        self.caches = list(caches) if caches else [step.cache]
        dev = step.device
        parts = [("q_hat", np.ascontiguousarray(q_hat_bits).view(np.int16)),
                 ("block_table", np.ascontiguousarray(block_table, dtype=np.int32)),
                 ("seq_lens", np.ascontiguousarray(seq_lens, dtype=np.int32)),
                 ("new_rows", np.ascontiguousarray(new_rows).view(np.int16)),
                 ("positions", np.ascontiguousarray(positions, dtype=np.int32))]
        if topk_idx is not None:
            parts.append(("topk_idx", np.ascontiguousarray(topk_idx, dtype=np.int32)))
        self.layout, off = {}, 0
        for name, arr in parts:
            self.layout[name] = (off, arr.dtype, arr.shape)
            off += (arr.nbytes + self.ALIGN - 1) // self.ALIGN * self.ALIGN
        self.in_bytes = off
        self.h2d_bytes = sum(arr.nbytes for _, arr in parts)
        out_shape, lse_shape = tuple(step.out.shape), tuple(step.lse.shape)
        out_nb = int(np.prod(out_shape)) * 2
        self.out_off = (0, (out_nb + self.ALIGN - 1) // self.ALIGN * self.ALIGN)
        self.out_bytes = self.out_off[1] + int(np.prod(lse_shape)) * 4
        self.d2h_bytes = out_nb + int(np.prod(lse_shape)) * 4
        self.host_in, self.dev_in, self.host_out, self.dev_out, self.views = [], [], [], [], []
        for _ in range(depth):
            h = torch.empty(self.in_bytes, dtype=torch.uint8).pin_memory()
            hn = h.numpy()
            for name, arr in parts:
                o, _, _ = self.layout[name]
                hn[o:o + arr.nbytes] = arr.reshape(-1).view(np.uint8)
            d = torch.empty(self.in_bytes, dtype=torch.uint8, device=dev)
            ho = torch.empty(self.out_bytes, dtype=torch.uint8).pin_memory()
            do = torch.empty(self.out_bytes, dtype=torch.uint8, device=dev)
            v = {name: self._view(d, name) for name, _ in parts}
            v["out"] = do[:out_nb].view(torch.bfloat16).view(out_shape)
            v["lse"] = do[self.out_off[1]:].view(torch.float32).view(lse_shape)
            self.host_in.append(h)
            self.dev_in.append(d)
            self.host_out.append(ho)
            self.dev_out.append(do)
            self.views.append(v)
        self.h2d_stream = torch.cuda.Stream(dev)
        self.d2h_stream = torch.cuda.Stream(dev)
        self.h2d_done = [torch.cuda.Event() for _ in range(depth)]
        self.computed = [torch.cuda.Event() for _ in range(depth)]
        self.d2h_done = [torch.cuda.Event() for _ in range(depth)]
        self.used = [False] * depth

    def _view(self, dev_arena, name):
        off, dtype, shape = self.layout[name]
        nb = int(np.prod(shape)) * np.dtype(dtype).itemsize
        t = dev_arena[off:off + nb]
        tdt = {np.dtype(np.int16): torch.int16, np.dtype(np.int32): torch.int32}[np.dtype(dtype)]
        return t.view(tdt).view(shape)

    def input_copied(self, k: int) -> torch.cuda.Event:
        return self.h2d_done[k % self.depth]

    def output_ready(self, k: int) -> torch.cuda.Event:
        """Recorded once step k's outputs are in host arena k % depth."""
        return self.d2h_done[k % self.depth]

    def host_outputs(self, k: int):
        """(o bf16 bits [rows][H][256], lse f32 [rows][H]) of step k (valid
        after output_ready(k))."""
        i = k % self.depth
        hn = self.host_out[i].numpy()
        nb = self.out_off[1]
        o = hn[:int(np.prod(self.step.out.shape)) * 2].view(np.uint16).reshape(tuple(self.step.out.shape))
        lse = hn[nb:].view(np.float32).reshape(tuple(self.step.lse.shape))
        return o, lse

    def submit(self, k: int, compute_stream=None):
        """Enqueue step k: input copy, append + decode + merge/W_UV, output copy."""
        from . import mla_cache_append
        i = k % self.depth
        st = self.step
        cs = compute_stream if compute_stream is not None else torch.cuda.current_stream(st.device)
        if self.used[i]:
            self.h2d_stream.wait_event(self.computed[i])   # the compute of step k - depth read set i
        with torch.cuda.stream(self.h2d_stream):
            self.dev_in[i].copy_(self.host_in[i], non_blocking=True)
            self.h2d_done[i].record(self.h2d_stream)
        cs.wait_event(self.h2d_done[i])
        if self.used[i]:
            cs.wait_event(self.d2h_done[i])                 # outputs of step k - depth copied out
        v = self.views[i]
        st.q_hat = v["q_hat"].view(torch.bfloat16)
        st.block_table, st.seq_lens = v["block_table"], v["seq_lens"]
        st.topk_idx = v.get("topk_idx")
        st.out, st.lse = v["out"], v["lse"]
        st.cache = self.caches[k % len(self.caches)]
        with torch.cuda.stream(cs):
            mla_cache_append(st.problem, v["new_rows"], v["positions"], st.block_table, st.cache,
                             stream=cs, rope_theta=self.rope_theta)
            st.step()
            self.computed[i].record(cs)
        self.d2h_stream.wait_event(self.computed[i])
        with torch.cuda.stream(self.d2h_stream):
            self.host_out[i].copy_(self.dev_out[i], non_blocking=True)
            self.d2h_done[i].record(self.d2h_stream)
        self.used[i] = True

    def capture(self, k0: int, n: int):
        """Capture steps k0 .. k0 + n - 1 (copies, append, decode, merge,
        W_UV and their cross-stream dependencies) in one CUDA graph, so a
        replay issues the whole pipelined sequence with one launch (on any
        stream).  The caller synchronises before capturing."""
        g = torch.cuda.CUDAGraph()
        compute_stream = torch.cuda.Stream(self.step.device)   # capture needs a side stream
        self.used = [False] * self.depth     # work recorded before the capture is complete
        with torch.cuda.graph(g, stream=compute_stream, capture_error_mode="relaxed"):
            fork = torch.cuda.Event()
            fork.record(compute_stream)
            self.h2d_stream.wait_event(fork)
            self.d2h_stream.wait_event(fork)
            for k in range(k0, k0 + n):
                self.submit(k, compute_stream)
            for i in range(self.depth):      # join every copy back into the capture stream
                if self.used[i]:
                    compute_stream.wait_event(self.h2d_done[i])
                    compute_stream.wait_event(self.d2h_done[i])
        self.used = [False] * self.depth
        return g

    def drain(self, k_last: int, compute_stream=None):
        """Make the compute stream wait for step k_last's outputs on the host."""
        cs = compute_stream if compute_stream is not None else torch.cuda.current_stream(self.step.device)
        cs.wait_event(self.d2h_done[k_last % self.depth])


def quantise_cache_on_device(latent_f32: np.ndarray, kv_dtype: int, device,
                             chunk_rows: int = 1 << 18) -> torch.Tensor:
    """An FP8 or FP4 paged cache made on the GPU from a float latent
    [num_pages, P, 576]: every slot's row, rounded to bf16, is quantised by
    mla_cache_append (scales from each group's absolute maximum).  Returns the
    cache bytes [num_pages, P * row_bytes] on `device`."""
    from . import mla_cache_append
    num_pages, P, D = latent_f32.shape
    row_bytes = 594 if kv_dtype == MLA_KV_FP8_E4M3_E8M0 else 324
    cache = torch.empty((num_pages, P * row_bytes), dtype=torch.uint8, device=device)
    flat = latent_f32.reshape(-1, D)
    n = flat.shape[0]
    for s in range(0, n, chunk_rows):
        e = min(n, s + chunk_rows)
        rows = torch.from_numpy(np.ascontiguousarray(flat[s:e])).to(device).to(torch.bfloat16)
        idx = torch.arange(s, e, dtype=torch.int64, device=device)
        # row r of the chunk is slot r % P of page r // P: a one-page block
        # table per row and its slot as the position
        bt = (idx // P).to(torch.int32).view(-1, 1)
        pos = (idx % P).to(torch.int32)
        prob = make_problem(e - s, 1, 1, P, num_pages, 1, kv_dtype=kv_dtype)
        mla_cache_append(prob, rows, pos, bt, cache)
    return cache
