"""GPU parity of the FP4 latent cache (e2m1 values, one e8m0 scale per 16).

Each cached row is 288 bytes of packed e2m1 codes and 36 scale bytes (this
build's reading of the FP4 variant of the inlined-scale latent in the
GLM-4.7-Flash record, engine-kernel constraint (2)); the decode attends over
e2m1 * 2^(scale - 127).  These checks run the CUDA path through the C ABI
against the oracle, which dequantises the same bytes in float64.
"""
import numpy as np
import pytest

import oracle as O
from oracle import fp4 as F4
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
    form on the decode's own bf16 absorbed query (the oracle's, uploaded)."""
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
def test_fp4_small_matches_oracle(source, garbage):
    """Codes drawn directly, and the oracle's quantiser applied to N(0, 1)
    rows; dead slots hold finite garbage or NaN scales."""
    batch = W.generate(W.SMALL_WORKLOADS["fp4_small"], garbage=garbage, fp8_source=source)
    with_fp8(batch, garbage)
    _run_and_compare(batch, label=f"fp4/{source}/{garbage}")


@pytest.mark.parametrize("page_size,sm_count", [(128, None), (64, 7), (128, 40), (32, 11),
                                                (16, None)])
def test_fp4_pages_and_splits(page_size, sm_count):
    """Every page size (a 64-row tile is a page, half of one, or 2 or 4
    pages) and forced splits of a request over CTAs."""
    w = W.with_overrides(W.SMALL_WORKLOADS["fp4_small"], page_size=page_size, seq_lo=1500,
                         seq_hi=4000, batch=3)
    _run_and_compare(W.generate(w), sm_count=sm_count, label=f"fp4/p{page_size}/c{sm_count}")


def test_fp4_dequant_is_exact():
    """One cached token per request: its softmax weight is exactly 1, so the
    latent output is the dequantised row itself, bit for bit.  The rows hold
    all 16 e2m1 codes under scales 2^-27 .. 2^13 (scale bytes above 128 take
    the two-factor path); the query selects one RoPE dim per head (q = 1
    there), so the lse is that dim's value times sm_scale and checks the 64
    RoPE dims too."""
    B, H = 8, 16
    w = W.with_overrides(W.SMALL_WORKLOADS["fp4_small"], batch=B, heads=H, seq_lens=(1,) * B)
    batch = W.generate(w)
    rng = np.random.default_rng(12)
    raw = batch.cache_fp4.reshape(batch.num_pages, w.page_size, F4.ROW_BYTES).copy()
    rows = {}
    for b in range(B):
        page = batch.block_table[b, 0]
        codes = np.resize(np.roll(np.arange(16, dtype=np.uint8), 5 * b), 576)
        rng.shuffle(codes)
        raw[page, 0, :F4.CODE_BYTES] = F4.pack_codes(codes)
        raw[page, 0, F4.CODE_BYTES:] = rng.integers(100, 141, size=F4.N_GROUPS, dtype=np.uint8)
        rows[b] = F4.dequant_rows(raw[page, 0])
    batch.extra["cache_fp4"] = raw.reshape(batch.num_pages, -1)
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


def test_fp4_edge_lengths():
    """Lengths around the 8-row copy granule and the 64-row tile."""
    w = W.with_overrides(W.SMALL_WORKLOADS["fp4_small"],
                         seq_lens=(0, 1, 7, 8, 9, 63, 64, 65, 127, 129), batch=10)
    batch = W.generate(w)
    q_hat = oracle_q_hat(batch)
    step = make_step(batch, absorb=False)
    upload_q_hat(step, q_hat)
    step.step()
    o, o_lat, lse = gpu_outputs(step)
    assert step.status() == 0
    compare(O.decode(batch), o, o_lat, lse, label="fp4-edges",
            lse_ref=O.decode(batch, q_hat=q_hat))


def test_fp4_bad_page_is_masked_and_reported():
    from head_latent_attention_paged_gb300 import MLA_STATUS_BAD_PAGE
    batch = W.generate(W.SMALL_WORKLOADS["fp4_small"])
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


def test_fp4_full_size_sampled():
    """The full FP4 workload (B=128, seq_lens U[2048, 16384], page 64) in
    the benchmark's launch configuration, sampled requests and heads."""
    batch = W.generate(W.WORKLOADS["fp4"])
    step = _run_and_compare(batch, requests=[0, 64, 127], heads=[0, 9, 19], label="fp4-full")
    o, _, lse = gpu_outputs(step)
    assert np.isfinite(o).all() and np.isfinite(lse).all()


@pytest.mark.parametrize("name,row_sets", [("fp8_small", 3), ("fp4_small", 3)])
def test_quantised_caches_with_draft_tokens(name, row_sets):
    """q_len 2 causal drafts over FP8 and FP4 caches, each draft with its own
    window: both drafts of a request in one row set, sharing every staged
    page."""
    w = W.with_overrides(W.SMALL_WORKLOADS[name], q_len=2, batch=3, seq_lo=60, seq_hi=700)
    step = _run_and_compare(W.generate(w), sm_count=11, label=f"{name}/q2")
    assert step.plan.num_streams == row_sets
