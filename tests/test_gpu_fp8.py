"""GPU parity of the FP8 latent cache (e4m3 values, one e8m0 scale per 32).

The decode reads each cached row as 576 e4m3 codes and 18 scale bytes
(GLM-4.7-Flash record, phantomic12 inference-research, the FlashMLA FP8
constraint: per-token inlined scales, RoPE dims quantised too) and attends
over e4m3 * 2^(scale - 127).  These checks run the CUDA path through the C
ABI against the oracle, which dequantises the same bytes in float64.
"""
import numpy as np
import pytest

import oracle as O
from oracle import fp8 as F
import workloads as W
from mla_testlib import (compare, ensure_built, gpu_outputs, make_step, oracle_q_hat,
                         upload_q_hat, with_fp8)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _run_and_compare(batch, sm_count=None, label="", requests=None, heads=None):
    """Outputs against the non-absorbed definition; lse against the absorbed
    form on the decode's own bf16 absorbed query (the oracle's, uploaded),
    because the bf16 rounding of q_hat alone moves the largest scores, and
    with them lse, by up to ~2e-3 on these FP8 rows."""
    q_hat = oracle_q_hat(batch)
    step = make_step(batch, sm_count=sm_count, absorb=False)
    upload_q_hat(step, q_hat)
    step.step()
    o, o_lat, lse = gpu_outputs(step)
    assert step.status() == 0, label
    ref = O.decode(batch, requests=requests, heads=heads)
    lse_ref = O.decode(batch, requests=requests, heads=heads, q_hat=q_hat)
    compare(ref, o, o_lat, lse, heads=heads, label=label, lse_ref=lse_ref)
    return step


@pytest.mark.parametrize("source", ["codes", "float"])
@pytest.mark.parametrize("garbage", ["finite", "nan"])
def test_fp8_small_matches_oracle(source, garbage):
    """Random codes over the whole code space, and the oracle's quantiser
    applied to N(0, 1) rows; dead slots hold finite garbage or NaN."""
    batch = W.generate(W.SMALL_WORKLOADS["fp8_small"], garbage=garbage, fp8_source=source)
    with_fp8(batch, garbage)
    _run_and_compare(batch, label=f"fp8/{source}/{garbage}")


@pytest.mark.parametrize("page_size,sm_count", [(128, None), (64, 7), (128, 40)])
def test_fp8_pages_and_splits(page_size, sm_count):
    """Both page sizes (a 64-row tile is a page or half of one) and forced
    splits of a request over CTAs (partials merged in the launch)."""
    w = W.with_overrides(W.SMALL_WORKLOADS["fp8_small"], page_size=page_size, seq_lo=1500,
                         seq_hi=4000, batch=3)
    _run_and_compare(W.generate(w), sm_count=sm_count, label=f"fp8/p{page_size}/c{sm_count}")


def test_fp8_dequant_is_exact():
    """One cached token per request: its softmax weight is exactly 1, so the
    latent output is the dequantised row itself, bit for bit.  The rows hold
    every finite e4m3 code under scales 2^-17 .. 2^8; the query selects one
    RoPE dim per head (q = 1 there), so the lse is that dim's value times
    sm_scale and checks the 64 RoPE dims too."""
    B, H = 8, 16
    w = W.with_overrides(W.SMALL_WORKLOADS["fp8_small"], batch=B, heads=H, seq_lens=(1,) * B)
    batch = W.generate(w)
    rng = np.random.default_rng(11)
    finite = np.array([c for c in range(256) if c & 0x7F != 0x7F], dtype=np.uint8)
    raw = batch.cache_fp8.reshape(batch.num_pages, w.page_size, F.ROW_BYTES).copy()
    rows = {}
    for b in range(B):
        page = batch.block_table[b, 0]
        codes = np.resize(np.roll(finite, 37 * b), 576)
        rng.shuffle(codes)
        raw[page, 0, :576] = codes
        raw[page, 0, 576:] = rng.integers(110, 136, size=18, dtype=np.uint8)
        rows[b] = F.dequant_rows(raw[page, 0])
    batch.extra["cache_fp8"] = raw.reshape(batch.num_pages, -1)
    q = np.zeros((B, 1, H, 576))
    for b in range(B):
        for h in range(H):
            q[b, 0, h, 512 + 4 * h + (b % 4)] = 1.0
    step = make_step(batch, absorb=False)
    upload_q_hat(step, q)
    step.step()
    _, o_lat, lse = gpu_outputs(step)
    assert step.status() == 0
    for b in range(B):
        expect = rows[b][:512].astype(np.float32)
        assert np.array_equal(expect.astype(np.float64), rows[b][:512])   # exact in f32
        for h in range(H):
            assert np.array_equal(o_lat[b, 0, h], expect), (b, h)
            s = rows[b][512 + 4 * h + (b % 4)] * w.sm_scale
            assert abs(lse[b, 0, h] - s) <= 1e-6 * abs(s) + 1e-30, (b, h)


def test_fp8_edge_lengths():
    """Lengths around the 8-row copy granule and the 64-row tile: a tail
    tile copies its live rows rounded up to 8.  As for bf16, the decode gets
    the oracle's bf16 absorbed query so T = 1 compares lse exactly."""
    w = W.with_overrides(W.SMALL_WORKLOADS["fp8_small"],
                         seq_lens=(0, 1, 7, 8, 9, 63, 64, 65, 127, 129), batch=10)
    batch = W.generate(w)
    q_hat = oracle_q_hat(batch)
    step = make_step(batch, absorb=False)
    upload_q_hat(step, q_hat)
    step.step()
    o, o_lat, lse = gpu_outputs(step)
    assert step.status() == 0
    compare(O.decode(batch), o, o_lat, lse, label="fp8-edges",
            lse_ref=O.decode(batch, q_hat=q_hat))


def test_fp8_bad_page_is_masked_and_reported():
    from head_latent_attention_paged_gb300 import MLA_STATUS_BAD_PAGE
    batch = W.generate(W.SMALL_WORKLOADS["fp8_small"])
    clean = make_step(batch)
    clean.step()
    _, lat_clean, _ = gpu_outputs(clean)
    bad = int(np.argmax(batch.seq_lens))
    assert batch.seq_lens[bad] > 64
    bt = batch.block_table.copy()
    bt[bad, 1] = batch.num_pages        # its second page: out of range
    batch.block_table = bt
    step = make_step(batch)
    step.step()
    _, lat, lse = gpu_outputs(step)
    assert step.status() & MLA_STATUS_BAD_PAGE
    for b in range(batch.workload.batch):
        if b != bad:
            assert np.array_equal(lat[b], lat_clean[b])
    assert np.isfinite(lat).all() and np.isfinite(lse).all()


def test_fp8_full_size_sampled():
    """The full FP8 workload (B=128, seq_lens U[2048, 16384], page 64) in
    the benchmark's launch configuration, sampled requests and heads."""
    batch = W.generate(W.WORKLOADS["fp8"])
    step = _run_and_compare(batch, requests=[0, 64, 127], heads=[0, 9, 19], label="fp8-full")
    o, _, lse = gpu_outputs(step)
    assert np.isfinite(o).all() and np.isfinite(lse).all()


def test_fp8_full_size_from_the_absmax_quantiser():
    """The FP8 workload as stated (B=128, seq_lens U[2048, 16384], page 64):
    an N(0, 1) latent quantised by the oracle's quantiser (one e8m0 scale per
    32 values from the group's absolute maximum), decoded in the benchmark's
    launch configuration; sampled requests and heads against the oracle on
    the same bytes."""
    batch = with_fp8(W.generate(W.WORKLOADS["fp8"], fp8_source="float"))
    batch.latent_f32 = None
    step = _run_and_compare(batch, requests=[0, 50, 101, 127], heads=[0, 6, 13, 19],
                            label="fp8-full-absmax")
    o, _, lse = gpu_outputs(step)
    assert np.isfinite(o).all() and np.isfinite(lse).all()


def test_gpu_quantiser_matches_oracle_on_full_size_rows():
    """The GPU quantiser the benchmark uses for its FP8 and FP4 caches
    (mla_cache_append over every slot) against the oracle's quantisers, byte
    for byte, on 4096 rows drawn from the full-size FP8 workload's latent."""
    from head_latent_attention_paged_gb300 import (MLA_KV_FP4_E2M1_E8M0, MLA_KV_FP8_E4M3_E8M0)
    from head_latent_attention_paged_gb300.runner import quantise_cache_on_device
    from oracle import fp4 as F4
    batch = W.generate(W.WORKLOADS["fp8"], fp8_source="float")
    rng = np.random.default_rng(17)
    rows = rng.choice(batch.latent_f32.shape[0] * batch.latent_f32.shape[1], size=4096, replace=False)
    flat = batch.latent_f32.reshape(-1, 576)[rows]
    bits = W.f32_to_bf16_bits(flat)
    lat = W.bf16_bits_to_f32(bits).reshape(64, 64, 576)     # 64 pages of the sampled rows
    for kv, enc in [(MLA_KV_FP8_E4M3_E8M0, F), (MLA_KV_FP4_E2M1_E8M0, F4)]:
        got = quantise_cache_on_device(lat, kv, "cuda:0").cpu().numpy().reshape(-1, enc.ROW_BYTES)
        want = enc.quantize_rows(lat.reshape(-1, 576).astype(np.float64))
        assert np.array_equal(got, want), (enc.__name__, int((got != want).any(axis=1).sum()))


def test_fp8_draft_pairs_full_size_sampled():
    """The FP8 workload with two causal draft tokens per request (an MTP
    draft pair over an FP8 cache): both drafts of a request form one row set
    of 40 rows that shares every staged page.  Benchmark launch
    configuration, sampled requests and heads."""
    batch = W.generate(W.WORKLOADS["mtp_fp8"])
    step = _run_and_compare(batch, requests=[0, 77, 127], heads=[0, 9, 19], label="mtp-fp8-full")
    assert step.plan.num_streams == 128
    o, _, lse = gpu_outputs(step)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
