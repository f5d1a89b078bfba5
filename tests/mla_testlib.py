"""Shared helpers for the GPU parity tests: run a workload through the C ABI
and compare with the CPU oracle."""
from __future__ import annotations

import numpy as np

import oracle as O
from oracle import fp4 as F4
from oracle import fp8 as F
import workloads as W

# Tolerances for the bf16, FP8 and FP4 paths: max |err| <= 2e-2 and relative L2
# <= 5e-3 on outputs, |lse err| <= 1e-3 (natural log).
ATOL_MAX = 2e-2
REL_L2 = 5e-3
LSE_TOL = 1e-3


def ensure_built():
    from head_latent_attention_paged_gb300 import _build
    _build.build()


def make_step(batch: W.Batch, sm_count=None, absorb=True, device="cuda:0", fp8_bytes=None,
              split_tokens=0, plan_with_host_lengths=True):
    from head_latent_attention_paged_gb300 import (MLA_KV_BF16, MLA_KV_FP4_E2M1_E8M0,
                                                   MLA_KV_FP8_E4M3_E8M0)
    from head_latent_attention_paged_gb300.runner import DecodeStep
    w = batch.workload
    if w.kv_dtype in ("fp8", "fp4"):
        cache = fp8_bytes if fp8_bytes is not None else batch.extra["cache_" + w.kv_dtype]
        kv_dtype = MLA_KV_FP8_E4M3_E8M0 if w.kv_dtype == "fp8" else MLA_KV_FP4_E2M1_E8M0
    else:
        cache = batch.cache_bf16
        kv_dtype = MLA_KV_BF16
    return DecodeStep(q_nope=batch.q_nope, q_rope=batch.q_rope, w_uk=batch.w_uk, w_uv=batch.w_uv,
                      cache=cache, block_table=batch.block_table, seq_lens=batch.seq_lens,
                      page_size=w.page_size, kv_dtype=kv_dtype, topk_idx=batch.topk_idx,
                      causal=w.causal, sm_scale=w.sm_scale, sm_count=sm_count, device=device,
                      absorb_on_device=absorb, split_tokens=split_tokens,
                      plan_with_host_lengths=plan_with_host_lengths)


def gpu_outputs(step):
    import torch
    torch.cuda.synchronize()
    o = step.out.float().cpu().numpy().reshape(step.B, step.Q, step.H, 256)
    o_lat = step.o_lat.cpu().numpy().reshape(step.B, step.Q, step.H, 512)
    lse = step.lse.cpu().numpy().reshape(step.B, step.Q, step.H)
    return o, o_lat, lse


def oracle_q_hat(batch: W.Batch) -> np.ndarray:
    """The absorbed query computed by the oracle in float64 and rounded to
    bf16 (float64 values, shape [B, Q, H, 576])."""
    w = batch.workload
    out = np.empty((w.batch, w.q_len, w.heads, 576))
    w_uk = O.bf16_to_f64(batch.w_uk)
    for b in range(w.batch):
        for j in range(w.q_len):
            out[b, j, :, :512] = O.round_to_bf16(O.absorb_query(O.bf16_to_f64(batch.q_nope[b, j]), w_uk))
            out[b, j, :, 512:] = O.bf16_to_f64(batch.q_rope[b, j])
    return out


def upload_q_hat(step, q_hat_f64):
    import torch
    bits = W.f32_to_bf16_bits(q_hat_f64.astype(np.float32).reshape(step.rows, step.H, 576))
    step.q_hat.copy_(torch.from_numpy(bits.view(np.int16)).to(step.q_hat.device).view(torch.bfloat16))


def compare(ref: dict, o, o_lat, lse, heads=None, label="", lse_ref=None):
    """Check every (b, j) the oracle computed.  Returns the worst figures.
    lse_ref: optional dict (b, j) -> lse to compare lse with instead."""
    worst = {"max_abs": 0.0, "rel_l2": 0.0, "lse": 0.0, "lat_rel_l2": 0.0}
    for (b, j), (ro, rlse, rlat) in ref.items():
        hs = slice(None) if heads is None else list(heads)
        go, glat, glse = o[b, j][hs], o_lat[b, j][hs], lse[b, j][hs]
        if np.all(np.isneginf(rlse)):
            assert np.all(np.isneginf(glse)), (label, b, j, glse)
            assert np.all(go == 0) and np.all(glat == 0), (label, b, j)
            continue
        ro_b = O.round_to_bf16(ro)
        err = np.abs(go - ro_b)
        assert np.isfinite(go).all() and np.isfinite(glat).all(), (label, b, j)
        max_abs = float(err.max())
        rel = float(np.linalg.norm(go - ro) / max(np.linalg.norm(ro), 1e-30))
        lat_rel = float(np.linalg.norm(glat - rlat) / max(np.linalg.norm(rlat), 1e-30))
        if lse_ref is not None:
            rlse = lse_ref[(b, j)][1]
        lse_err = float(np.abs(glse - rlse).max())
        worst["max_abs"] = max(worst["max_abs"], max_abs)
        worst["rel_l2"] = max(worst["rel_l2"], rel)
        worst["lat_rel_l2"] = max(worst["lat_rel_l2"], lat_rel)
        worst["lse"] = max(worst["lse"], lse_err)
        assert max_abs <= ATOL_MAX, (label, b, j, "max abs", max_abs)
        assert rel <= REL_L2, (label, b, j, "rel L2", rel)
        assert lat_rel <= REL_L2, (label, b, j, "latent rel L2", lat_rel)
        assert lse_err <= LSE_TOL, (label, b, j, "lse", lse_err)
    return worst


def with_fp8(batch: W.Batch, garbage="finite") -> W.Batch:
    """FP8 / FP4 workloads drawn with fp8_source="float": attach the paged
    bytes made by the oracle's quantiser (codes-drawn batches have them)."""
    kv = batch.workload.kv_dtype
    if kv in ("fp8", "fp4") and "cache_" + kv not in batch.extra:
        enc = F if kv == "fp8" else F4
        batch.extra["cache_" + kv] = enc.quantize_pages(batch.latent_f32, batch.slot_valid,
                                                        rng_seed=batch.workload.seed,
                                                        garbage=garbage)
    return batch
