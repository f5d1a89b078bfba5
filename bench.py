#!/usr/bin/env python3
"""Benchmark of one paged MLA decode step (one layer) on GB300.

A step is the whole hot path over one synthetic decode batch, one call of
mla_decode_step: the attention pass over the paged latent cache, the LSE
merge of split partials inside the W_UV up-projection (two kernels, the
second launched as a programmatic dependent of the first; the absorbed query
is an input, precomputed once).  The
default workload is the GLM-4.7-Flash-shaped dense decode: batch 64, 20
heads, q_len 1, seq_lens ~ U[1024, 8192], page 64, bf16 latent cache.

Metric: latent-cache GB/s (bytes of cached rows the step must read, over the
step time) and decode tokens/s per layer.  Prints one JSON line; besides the
headline workload it carries, under per_workload, the decode kernel and the
whole step of the long-context, FP8, sparse, FP4 and multi-token workloads,
each timed launch by launch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle as the reference arm

Under torchrun each rank runs an independent replica of the workload on its
own GPU (the path shards by request and has no exchange step); rank 0 prints
the line with the bytes of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MLA decode latent-cache GB/s (% of HBM peak) and decode tokens/s per layer"
L2_FLUSH_BYTES = 512 * 1024 * 1024
L2_BYTES = 129 * 1000 * 1000     # GB300 L2
DECODE_SOURCES = ["csrc/mla_decode.cu", "csrc/sm103_ptx.cuh", "csrc/mla_internal.h"]


def overhead_bytes(w, batch) -> dict:
    """Bytes a step moves besides the cached rows: the absorbed queries, the
    page tables, the top-k lists, W_UV, and the split partials (an upper
    bound: every slot of the plan written once and read once)."""
    import numpy as np
    rows = w.batch * w.q_len
    g = min(w.q_len, 48 // w.heads) if (w.kv_dtype == "bf16" and not w.topk and w.q_len >= 2) else 1
    g = g if g >= 2 else 1
    row_sets = w.batch * -(-w.q_len // g)
    slots = row_sets + 152 - 1
    d = {"q_hat": rows * w.heads * 576 * 2, "block_table": int(batch.block_table.nbytes),
         "seq_lens": int(batch.seq_lens.nbytes), "w_uv": w.heads * 512 * 256 * 2,
         "partials_max": slots * g * w.heads * (512 + 1) * 4 * 2}
    if w.topk:
        d["topk_idx"] = int(batch.topk_idx.nbytes)
        # rows the drafts of a request share: each read once per request
        uniq = 0
        for b in range(w.batch):
            idx = batch.topk_idx[b * w.q_len:(b + 1) * w.q_len]
            uniq += int(np.unique(idx[idx >= 0]).size)
        d["latent_bytes_union_of_drafts"] = uniq * w.cache_row_bytes
    return d


def workload_description(w, batch, rotate: bool = False) -> dict:
    seq = batch.seq_lens
    d = {
        "workload": f"{w.name}: MLA decode, 1 layer, B={w.batch}, H={w.heads}, q_len={w.q_len}, "
                    f"page {w.page_size}, {w.kv_dtype} latent (512 + 64 rope)"
                    + (f", top-{w.topk} sparse (width {w.topk_width})" if w.topk else "")
                    + (f", seq_lens U[{w.seq_lo},{w.seq_hi}]" if w.seq_lens is None
                       else f", seq_lens {list(w.seq_lens)}"),
        "batch": w.batch, "heads": w.heads, "q_len": w.q_len, "page_size": w.page_size,
        "kv_dtype": w.kv_dtype, "topk": w.topk, "seed": w.seed,
        "total_context_tokens": int(seq.sum()),
        "latent_bytes_per_step": int(batch.latent_bytes_read),
        "overhead_bytes_per_step": overhead_bytes(w, batch),
        "bytes_per_token_row": w.cache_row_bytes,
        "l2": ("no flush: consecutive timed steps read two copies of the cache in turn "
               "(each larger than the 129 MB L2)") if rotate else
              (f"flushed before every timed step by writing {L2_FLUSH_BYTES >> 20} MiB "
               "(step time from CUDA events excludes the flush)"),
    }
    return d


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f)
    return {}


def decode_source_hash() -> str:
    h = hashlib.sha256()
    for rel in DECODE_SOURCES:
        with open(os.path.join(ROOT, "head_latent_attention_paged_gb300", rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on this workload with the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    entry = rec.get(workload)
    if not entry or entry.get("source_hash") != decode_source_hash():
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.samples = []
        self._stop = threading.Event()
        self._thread = threading.Thread(target=self._run, daemon=True)

    def _run(self):
        while not self._stop.is_set():
            try:
                out = subprocess.run(
                    ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                     "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=5)
                if out.returncode == 0 and out.stdout.strip():
                    self.samples.append([x.strip() for x in out.stdout.strip().split(",")])
            except Exception:
                pass
            self._stop.wait(0.05)

    def __enter__(self):
        self._thread.start()
        return self

    def __exit__(self, *exc):
        self._stop.set()
        self._thread.join(timeout=10)

    def summary(self) -> dict:
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"],
                    "samples": 0}
        sm = [float(s[0]) for s in self.samples if s[0].replace(".", "").isdigit()]
        smax = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for s in self.samples:
            for name, val in zip(names, s[4:8]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        power = [float(s[2]) for s in self.samples if s[2].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(self.samples),
                "power_w_max": max(power) if power else None}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(value_bytes: float, seconds: float, world: int, device=None):
    """Sum of bytes over ranks and the slowest rank's time (replicas)."""
    if world == 1:
        return value_bytes, seconds
    import torch
    import torch.distributed as dist
    t = torch.tensor([value_bytes, seconds], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    b = t[0:1].clone()
    s = t[1:2].clone()
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    dist.all_reduce(s, op=dist.ReduceOp.MAX)
    return float(b.item()), float(s.item())


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline leg and reference arm)
# ---------------------------------------------------------------------------
def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        if info:
            return max(int(i.get("num_threads", 1)) for i in info)
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count() or 1


def oracle_sample(batch, budget_s: float, max_tokens: int = None, form: str = "non_absorbed",
                  max_requests: int = None):
    """Time the float64 oracle (the non-absorbed definition, or its absorbed
    form) on a bounded sample: whole requests in order until `budget_s` is
    spent (or `max_requests` are done), or a prefix of the first request of at
    most `max_tokens` tokens.  Returns (bytes, seconds, what)."""
    import numpy as np
    import oracle as O
    w = batch.workload
    if max_tokens is not None:
        sub = _prefix_batch(batch, max_tokens)
        t0 = time.perf_counter()
        O.decode(sub, requests=[0], form=form)
        dt = time.perf_counter() - t0
        return sub.latent_bytes_read_req(0), dt, f"first {int(sub.seq_lens[0])} tokens of request 0, all {w.heads} heads"
    done_bytes, t0, n = 0, time.perf_counter(), 0
    for b in range(w.batch if max_requests is None else min(w.batch, max_requests)):
        O.decode(batch, requests=[b], form=form)
        n += 1
        done_bytes += _request_bytes(batch, b)
        if time.perf_counter() - t0 >= budget_s:
            break
    return done_bytes, time.perf_counter() - t0, f"{n} whole request(s) of {w.batch}, all {w.heads} heads"


def one_thread_sample(workload: str):
    """The non-absorbed oracle on one BLAS thread (a child process started
    with the thread-count variables at 1), on the first 1024 tokens of
    request 0: GB/s, or None if the child fails."""
    env = dict(os.environ)
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = "1"
    code = ("import sys, json; sys.path.insert(0, %r); import bench, workloads as W; "
            "b = W.generate(W.WORKLOADS[%r]); by, dt, what = bench.oracle_sample(b, 0, max_tokens=1024); "
            "print(json.dumps([by, dt, what]))") % (ROOT, workload)
    try:
        out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                             timeout=300)
        by, dt, what = json.loads(out.stdout.strip().splitlines()[-1])
        return {"value": by / dt / 1e9, "unit": "GB/s", "threads": 1,
                "sample": f"{what}: non-absorbed float64 numpy oracle, {dt:.2f} s"}
    except Exception:
        return None


def _request_bytes(batch, b):
    w = batch.workload
    if w.topk:
        return int((batch.topk_idx[b * w.q_len:(b + 1) * w.q_len] >= 0).sum()) * w.cache_row_bytes
    return int(batch.seq_lens[b]) * w.cache_row_bytes


def _prefix_batch(batch, tokens):
    import copy
    import numpy as np
    sub = copy.copy(batch)
    seq = batch.seq_lens.copy()
    seq[0] = min(int(seq[0]), tokens)
    sub.seq_lens = seq
    sub.latent_bytes_read_req = lambda b: _request_bytes(sub, b)
    return sub


def cache_bytes(batch) -> int:
    """Bytes of one copy of the workload's latent cache."""
    for c in (batch.cache_bf16, batch.cache_quant):
        if c is not None:
            return int(c.nbytes)
    return 0


def run_reference(args, world, rank):
    import numpy as np
    import workloads as W
    if rank != 0:
        return 0
    w = W.WORKLOADS[args.workload]
    batch = W.generate(w)
    # calibrate: tokens per step so the whole run stays within ~2 minutes
    b_cal, t_cal, _ = oracle_sample(batch, 0, max_tokens=256)
    rate = b_cal / max(t_cal, 1e-9) / w.cache_row_bytes        # tokens per second
    per_step_s = min(2.0, 120.0 / max(1, args.steps + args.warmup))
    tokens = int(max(64, min(int(batch.seq_lens[0]), rate * per_step_s)))
    for _ in range(args.warmup):
        oracle_sample(batch, 0, max_tokens=tokens)
    times, byts = [], 0
    what = ""
    for _ in range(args.steps):
        bb, dt, what = oracle_sample(batch, 0, max_tokens=tokens)
        times.append(dt)
        byts += bb
    total = sum(times)
    value = byts / total / 1e9
    cores = blas_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": workload_description(w, batch, cache_bytes(batch) > L2_BYTES),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": f"each step: {what} (non-absorbed float64 numpy oracle)"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
PER_WORKLOADS = ["long", "fp8", "sparse", "fp4", "mtp", "mtp_fp8"]


def kernel_label(w) -> str:
    if w.kv_dtype in ("fp8", "fp4"):
        return "mla_decode_kernel<dense %s%s>" % (w.kv_dtype, " multi-token" if w.q_len > 1 else "")
    if w.topk:
        return "mla_decode_kernel<sparse bf16>"
    return "mla_decode_kernel<dense bf16%s>" % (" multi-token" if w.q_len > 1 else "")


def prepare(w, device):
    """The workload's batch and a DecodeStep on `device`.  FP8 and FP4 caches
    are quantised on the GPU (mla_cache_append, scales from each group's
    absolute maximum) from the workload's N(0, 1) latent rounded to bf16."""
    import workloads as W
    from head_latent_attention_paged_gb300 import (MLA_KV_BF16, MLA_KV_FP4_E2M1_E8M0,
                                                   MLA_KV_FP8_E4M3_E8M0)
    from head_latent_attention_paged_gb300.runner import DecodeStep, quantise_cache_on_device
    kv = {"bf16": MLA_KV_BF16, "fp8": MLA_KV_FP8_E4M3_E8M0, "fp4": MLA_KV_FP4_E2M1_E8M0}[w.kv_dtype]
    quant = w.kv_dtype in ("fp8", "fp4")
    batch = W.generate(w, fp8_source="float" if quant else "codes")
    cache = quantise_cache_on_device(batch.latent_f32, kv, device) if quant else batch.cache_bf16
    if quant:
        batch.latent_f32 = None     # the float latent is not needed any more
    step = DecodeStep(q_nope=batch.q_nope, q_rope=batch.q_rope, w_uk=batch.w_uk, w_uv=batch.w_uv,
                      cache=cache, block_table=batch.block_table, seq_lens=batch.seq_lens,
                      page_size=w.page_size, kv_dtype=kv, topk_idx=batch.topk_idx,
                      causal=w.causal, sm_scale=w.sm_scale, device=device)
    return batch, step


class Rotation:
    """Between timed launches no launch may find the previous one's cache
    lines in L2: a cache larger than the L2 is read from two copies in turn
    (no flush, which would leave dirty lines for the next launch to write
    back); a smaller one is flushed by writing 512 MiB before each launch."""

    def __init__(self, step, device):
        import torch
        self.step = step
        self.rotate = int(step.cache.numel()) * step.cache.element_size() > L2_BYTES
        self.caches = [step.cache, step.cache.clone()] if self.rotate else [step.cache]
        self.flush = None if self.rotate else torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8,
                                                          device=device)

    def before(self, k):
        if self.rotate:
            self.step.cache = self.caches[k % 2]
        else:
            self.flush.zero_()


def hold_device(n):
    """Queue a spin of about 0.1 ms per launch group ahead of n timed ones, so
    that the host has queued them all before the device reaches the first:
    the events then bracket device work only, not the host's launch calls."""
    import torch
    torch.cuda._sleep(int(min(n, 2000) * 2.0e5))


def timed(step, rot, n, stream, fn):
    """n launches of fn(), each bracketed by CUDA events on `stream`: times
    in ms."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    hold_device(n)
    for k in range(n):
        rot.before(k)
        ev[k][0].record(stream)
        fn()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def measure_workload(name, device, steps, hbm, warmup=3):
    """Device-timed decode kernel alone and whole steps (decode, then merge +
    W_UV) of one workload: medians and means over `steps` launches each."""
    import gc
    import torch
    import workloads as W
    w = W.WORKLOADS[name]
    batch, step = prepare(w, device)
    stream = torch.cuda.current_stream(device)
    rot = Rotation(step, device)
    for k in range(warmup):
        rot.before(k)
        step.step()
    torch.cuda.synchronize()
    if step.status() != 0:
        raise SystemExit(f"{name}: decode reported status {step.status():#x}")
    with ClockSampler(device.index or 0) as clocks:
        dec = timed(step, rot, steps, stream, step.attend)
        full = timed(step, rot, steps, stream, step.step)
    byts = batch.latent_bytes_read
    dm, fm = statistics.median(dec), statistics.median(full)
    out = {
        "workload": workload_description(w, batch, rot.rotate)["workload"],
        "kernel": kernel_label(w),
        "latent_bytes_per_step": int(byts),
        "decode_us_median": 1e3 * dm, "decode_us_mean": 1e3 * statistics.mean(dec),
        "decode_gbs": byts / (dm / 1e3) / 1e9, "decode_frac": byts / (dm / 1e3) / 1e9 / hbm,
        "step_us_median": 1e3 * fm, "step_us_mean": 1e3 * statistics.mean(full),
        "step_gbs": byts / (fm / 1e3) / 1e9, "step_frac": byts / (fm / 1e3) / 1e9 / hbm,
        "tokens_per_s_per_layer": w.batch * w.q_len / (fm / 1e3),
        "timed_launches": steps,
        "traffic": recorded_traffic(name),
        "l2": "two cache copies read in turn" if rot.rotate else "512 MiB flush before each launch",
        "clocks": clocks.summary(),
    }
    if w.kv_dtype in ("fp8", "fp4"):
        out["cache"] = ("N(0, 1) latent rounded to bf16, quantised on the GPU by mla_cache_append "
                        "(one e8m0 scale per group from its absolute maximum)")
    del step, rot, batch
    gc.collect()
    torch.cuda.empty_cache()
    return out


def run_gpu(args, world, rank, local):
    import numpy as np
    import torch
    import workloads as W
    import __graft_entry__ as graft
    from head_latent_attention_paged_gb300.runner import DecodeStep

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    graft.build()
    peaks = measured_peaks()
    hbm = peaks.get("hbm_gbs")
    peak_src = "measured (MEASURED_PEAKS.json hbm_gbs)"
    if not hbm:
        hbm, peak_src = 6800.0, "fallback 6.8 TB/s"
    w = W.WORKLOADS[args.workload]
    batch, step = prepare(w, device)
    stream = torch.cuda.current_stream(device)
    byts = batch.latent_bytes_read
    rot = Rotation(step, device)

    for k in range(args.warmup):
        rot.before(k)
        step.step()
    torch.cuda.synchronize(device)
    if step.status() != 0:
        raise SystemExit(f"decode reported status {step.status():#x}")

    # The K timed steps: each one call of mla_decode_step (the attention pass,
    # then the merge inside the W_UV launch, a programmatic dependent of the
    # first), bracketed by events on the launching stream.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(device)
    with ClockSampler(local) as clocks:
        hold_device(args.steps)
        t_wall = time.perf_counter()
        for k in range(args.steps):
            rot.before(k)
            ev[k][0].record(stream)
            step.step()
            ev[k][1].record(stream)
        torch.cuda.synchronize(device)
        t_wall = time.perf_counter() - t_wall
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(device)
        # The decode kernel alone, timed on every one of its own launches
        # (after the step loop, so the steps keep their launch overlap).
        dec_ms = timed(step, rot, max(args.decode_steps, 20), stream, step.attend)
    per_workload = {}
    if world == 1 and args.per_workload:
        for name in PER_WORKLOADS:
            if name != args.workload:
                per_workload[name] = measure_workload(name, device, args.per_workload_steps, hbm)
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    step_s = sum(step_ms) / 1e3
    tot_bytes, max_s = aggregate(float(byts) * args.steps, step_s, world, device)
    value = tot_bytes / max_s / 1e9
    ms_per_step = 1e3 * max_s / args.steps
    decode_ms = statistics.median(dec_ms)

    # End to end through the public API with host buffers.  The latent cache
    # is device-resident state (as in serving); what a decode step gets from
    # the host is its inputs: the absorbed queries, the block table, the
    # context lengths, the top-k lists (sparse) and each request's newest
    # token row, which mla_cache_append rotates (RoPE, theta 1e6) and writes
    # at its slot.  Every step copies those in from pinned host memory (one
    # copy of one packed arena), appends, runs the step and copies o and lse
    # back (one copy); HostPipeline overlaps step k's copies with the
    # neighbouring steps' kernels on two copy streams.  No L2 flush here (it
    # would sit inside the pipelined region): the benchmark workloads' caches
    # are larger than the 129 MB L2, and consecutive steps read two different
    # copies of them.
    e2e = None
    if args.e2e_steps > 0:
        from head_latent_attention_paged_gb300.runner import HostPipeline
        # the newest token of each request: a synthetic bf16 row [B][576]
        # (N(0, 1) like the cache, seeded), appended by the step at position
        # T_b - 1 with mla_cache_append (FP8 / FP4 caches quantise it on the GPU)
        last_pos = (batch.seq_lens.astype(np.int64) - 1).astype(np.int32)
        rng = np.random.default_rng(w.seed + 1)
        rows_np = W.f32_to_bf16_bits(rng.standard_normal((w.batch, 576)).astype(np.float32))
        pipe = HostPipeline(step, q_hat_bits=step.q_hat.view(torch.int16).cpu().numpy(),
                            block_table=batch.block_table, seq_lens=batch.seq_lens,
                            new_rows=rows_np, positions=last_pos, topk_idx=batch.topk_idx,
                            caches=rot.caches if rot.rotate else None, rope_theta=1.0e6)
        WARM = 3
        for k in range(WARM):
            pipe.submit(k, stream)
        pipe.drain(WARM - 1, stream)
        torch.cuda.synchronize(device)
        if world > 1:
            torch.distributed.barrier()
        # the timed steps are one CUDA graph (captured once, replayed once
        # untimed, then timed): the host issues the whole pipelined sequence
        # with one launch instead of ~10 Python-level calls per step
        last = WARM + args.e2e_steps - 1
        graph = pipe.capture(WARM, args.e2e_steps)
        torch.cuda.synchronize(device)
        graph.replay()
        torch.cuda.synchronize(device)
        e_start = torch.cuda.Event(enable_timing=True)
        e_end = torch.cuda.Event(enable_timing=True)
        e_start.record(stream)
        graph.replay()
        e_end.record(stream)
        torch.cuda.synchronize(device)
        e2e_s = e_start.elapsed_time(e_end) / 1e3
        # the last two steps had the same inputs: their outputs must agree
        o_a, l_a = (x.copy() for x in pipe.host_outputs(last))
        o_b, l_b = pipe.host_outputs(last - 1)
        if not (np.array_equal(o_a, o_b) and np.array_equal(l_a, l_b)):
            raise SystemExit("end-to-end outputs differ between identical steps")
        if step.status() != 0:
            raise SystemExit(f"end-to-end steps reported status {step.status():#x}")
        eb, es = aggregate(float(byts) * args.e2e_steps, e2e_s, world, device)
        e2e = {"value": eb / es / 1e9, "unit": "GB/s", "h2d_bytes_per_step": int(pipe.h2d_bytes),
               "d2h_bytes_per_step": int(pipe.d2h_bytes), "steps": args.e2e_steps,
               "ms_per_step": 1e3 * es / args.e2e_steps,
               "inputs": "q_hat, block table, seq_lens, top-k lists, newest token row and "
                         "position per request, one packed host->device copy per step "
                         "(rows RoPE-rotated and appended with mla_cache_append; cache "
                         "resident); o and lse one device->host copy per step; copies "
                         "pipelined against the neighbouring steps on two copy streams "
                         "(double-buffered), the timed steps replayed as one CUDA graph; no "
                         "L2 flush: consecutive steps read two copies of the cache (each "
                         "larger than L2)"}

    if rank != 0:
        return 0
    achieved = byts / (decode_ms / 1e3) / 1e9
    traffic = recorded_traffic(args.workload)
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {"bf16": "bf16", "fp8": "fp8-e4m3+e8m0 cache, bf16 tensor-core math",
                  "fp4": "fp4-e2m1+e8m0 cache, bf16 tensor-core math"}[w.kv_dtype],
        "data": "synthetic",
        "config": workload_description(w, batch, rot.rotate),
        "tokens_per_s_per_layer": w.batch * w.q_len * world / (max_s / args.steps),
        "hbm_fraction_of_measured": value / hbm,
        "kernel_ms": {"decode": statistics.mean(dec_ms), "decode_median": decode_ms,
                      "decode_timed_launches": len(dec_ms),
                      "step": statistics.mean(step_ms), "step_median": statistics.median(step_ms),
                      "step_timed": len(step_ms)},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": achieved / hbm, "traffic": traffic,
                     "kernel": kernel_label(w),
                     "timing": f"median of {len(dec_ms)} launches of the decode kernel alone, "
                               "each bracketed by CUDA events on its stream",
                     "peak_source": peak_src,
                     "algorithmic_bytes_per_launch": int(byts),
                     "step_frac": byts / (statistics.median(step_ms) / 1e3) / 1e9 / hbm},
        "per_workload": per_workload or None,
        "e2e": e2e,
        "gpu_launches": step.kernels_per_step * args.steps,
        "clocks": clocks.summary(),
        "wall_s_timed_region": t_wall,
        "status": step.status(),
    }
    if world == 1 and not args.no_cpu_baseline and w.kv_dtype != "bf16":
        line["cpu_baseline"] = None   # the quantised cache exists on the GPU only
    elif world == 1 and not args.no_cpu_baseline:
        cb, ct, what = oracle_sample(batch, args.cpu_budget)
        n_req = int(what.split()[0]) if what.split()[0].isdigit() else 1
        ab, at, _ = oracle_sample(batch, 1e9, form="absorbed", max_requests=n_req)
        line["cpu_baseline"] = {"value": cb / ct / 1e9, "unit": "GB/s", "cores": blas_threads(),
                                "kind": "oracle",
                                "sample": f"{what}: non-absorbed float64 numpy oracle, {ct:.1f} s",
                                "cpu_count": os.cpu_count(),
                                "absorbed_value": ab / at / 1e9,
                                "absorbed_sample": f"the same requests, absorbed float64 form, {at:.1f} s",
                                "one_thread": one_thread_sample(args.workload)}
    print(json.dumps(line))
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="dense",
                    choices=["tiny", "dense", "long", "fp8", "sparse", "fp4", "mtp", "mtp_fp8"])
    ap.add_argument("--impl", default="gpu", choices=["gpu", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--decode-steps", type=int, default=1000,
                    help="launches of the decode kernel alone timed one by one")
    ap.add_argument("--per-workload-steps", type=int, default=300,
                    help="launches of the decode kernel alone and of whole steps timed one by "
                         "one for each of the other workloads")
    ap.add_argument("--no-per-workload", dest="per_workload", action="store_false",
                    help="skip the long / fp8 / sparse / fp4 / mtp / mtp_fp8 measurements")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_gpu(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
