"""GPU parity of the cache append (mla_cache_append): each request's newest
token row written into the paged cache, bf16 as is or quantised to the FP8 or
FP4 layout on the GPU.  Compared byte for byte with the oracle's append, which
uses the oracle's quantisers, on the same bf16 rows."""
import numpy as np
import pytest

import oracle as O
from oracle import cache_append as CA
from oracle import fp8 as F
import workloads as W
from mla_testlib import compare, ensure_built, gpu_outputs, make_step, oracle_q_hat, upload_q_hat

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _special_rows(rng, B):
    """bf16 rows with groups that exercise the quantiser's edges."""
    x = rng.standard_normal((B, 576)).astype(np.float32)
    x[0, 0:32] = 0.0                                   # all-zero group
    x[0, 32:64] = 0.0
    x[0, 40] = -0.0                                    # zeros of both signs
    x[1, 0:32] = rng.uniform(-448, 448, 32)
    x[1, 5] = 448.0                                    # amax exactly 448: scale 1
    x[1, 32:64] = rng.uniform(-450, 450, 32)
    x[1, 33] = -450.0                                  # just above: scale 2
    x[2, 0:32] = rng.standard_normal(32) * 1e-30       # tiny
    x[2, 32:64] = rng.standard_normal(32) * 1e30       # huge
    x[2, 64:96] = rng.standard_normal(32) * 1e-38      # bf16 subnormals: scale clamps
    x[3, 0:32] = rng.choice([-3.0, -1.0, 0.5, 2.5, 7.0], 32)   # rounding ties after scaling
    # FP4 rounding ties (amax 6: scale 1): every midpoint of the e2m1 grid
    x[5, 0:16] = [6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, -0.75, -1.75,
                  -2.5, -3.5, -1.25, -0.0]
    x[5, 16:32] = np.array([12.0, 0.5, 1.5, 2.5, 3.5, 5.0, 7.0, 10.0, -0.5, -1.5, -2.5,
                            -3.5, -5.0, -7.0, -10.0, 0.1])            # amax 12: scale 2
    return W.f32_to_bf16_bits(x)


def _problem(batch, w, num_pages, max_pages, fp8):
    from head_latent_attention_paged_gb300 import (MLA_KV_BF16, MLA_KV_FP4_E2M1_E8M0,
                                                   MLA_KV_FP8_E4M3_E8M0, make_problem)
    kv = {"bf16": MLA_KV_BF16, "fp8": MLA_KV_FP8_E4M3_E8M0, "fp4": MLA_KV_FP4_E2M1_E8M0}[fp8] \
        if isinstance(fp8, str) else (MLA_KV_FP8_E4M3_E8M0 if fp8 else MLA_KV_BF16)
    return make_problem(batch, 1, w.heads, w.page_size, num_pages, max_pages, kv_dtype=kv)


@pytest.mark.parametrize("kv,page_size", [("bf16", 64), ("bf16", 128), ("fp8", 64), ("fp8", 128),
                                          ("fp4", 64), ("fp4", 128), ("fp4", 16)])
def test_append_matches_oracle_bytes(kv, page_size):
    from head_latent_attention_paged_gb300 import mla_cache_append
    base = W.SMALL_WORKLOADS[{"bf16": "dense_small", "fp8": "fp8_small", "fp4": "fp4_small"}[kv]]
    w = W.with_overrides(base, page_size=page_size, batch=6, seq_lo=1, seq_hi=500)
    batch = W.generate(w)
    rng = np.random.default_rng(7)
    rows = _special_rows(rng, w.batch)
    # positions: the next token after each context where the pages have room,
    # an in-context overwrite, and -1 (no append)
    seq = batch.seq_lens.astype(np.int32)
    pos = np.where(seq % page_size != 0, seq, seq - 1).astype(np.int32)   # a mapped slot
    pos[2] = 0
    pos[4] = -1
    cache = batch.cache_bf16 if kv == "bf16" else batch.cache_quant
    expect = CA.append_rows(cache, rows, pos, batch.block_table, page_size, kv)
    dev = torch.device("cuda", 0)
    cache_d = torch.from_numpy(cache.view(np.uint8).copy()).to(dev)
    rows_d = torch.from_numpy(rows.view(np.int16).copy()).to(dev)
    pos_d = torch.from_numpy(pos).to(dev)
    bt_d = torch.from_numpy(batch.block_table).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    mla_cache_append(_problem(w.batch, w, batch.num_pages, batch.block_table.shape[1], kv),
                     rows_d, pos_d, bt_d, cache_d, status)
    torch.cuda.synchronize()
    got = cache_d.cpu().numpy()
    assert int(status.item()) == 0
    assert np.array_equal(got, expect.view(np.uint8).reshape(got.shape))


def test_append_reports_bad_positions_and_pages():
    from head_latent_attention_paged_gb300 import (MLA_STATUS_BAD_INDEX, MLA_STATUS_BAD_PAGE,
                                                   mla_cache_append)
    w = W.with_overrides(W.SMALL_WORKLOADS["dense_small"], batch=3, seq_lo=100, seq_hi=200)
    batch = W.generate(w)
    rows = W.f32_to_bf16_bits(np.ones((3, 576), dtype=np.float32))
    max_tok = batch.block_table.shape[1] * w.page_size
    pos = np.array([max_tok, 5, 7], dtype=np.int32)       # row 0: past the pages
    bt = batch.block_table.copy()
    bt[1, 0] = -2                                          # row 1: bad page id
    dev = torch.device("cuda", 0)
    cache_d = torch.from_numpy(batch.cache_bf16.view(np.uint8).copy()).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    mla_cache_append(_problem(3, w, batch.num_pages, bt.shape[1], False),
                     torch.from_numpy(rows.view(np.int16)).to(dev), torch.from_numpy(pos).to(dev),
                     torch.from_numpy(bt).to(dev), cache_d, status)
    torch.cuda.synchronize()
    bits = int(status.item())
    assert bits & MLA_STATUS_BAD_INDEX and bits & MLA_STATUS_BAD_PAGE
    expect = CA.append_rows(batch.cache_bf16, rows, np.array([-1, -1, 7]), bt, w.page_size, "bf16")
    got = cache_d.cpu().numpy()
    assert np.array_equal(got, expect.view(np.uint8).reshape(got.shape))


@pytest.mark.parametrize("name", ["dense_small", "fp8_small", "fp4_small"])
def test_decode_sees_appended_token(name):
    """Append the next token of every request, then decode over seq_lens + 1:
    the result matches the oracle decode over the oracle-appended cache."""
    from head_latent_attention_paged_gb300 import mla_cache_append
    w = W.SMALL_WORKLOADS[name]
    batch = W.generate(w)
    room = batch.seq_lens < batch.block_table.shape[1] * w.page_size
    keep = np.flatnonzero(room & (batch.seq_lens % w.page_size != 0))   # next slot on a mapped page
    assert keep.size >= 2
    rng = np.random.default_rng(9)
    rows = W.f32_to_bf16_bits(rng.standard_normal((w.batch, 576)).astype(np.float32))
    pos = np.full(w.batch, -1, dtype=np.int32)
    pos[keep] = batch.seq_lens[keep]
    kv = w.kv_dtype
    cache = batch.cache_bf16 if kv == "bf16" else batch.cache_quant
    step = make_step(batch, absorb=False)
    q_hat = oracle_q_hat(batch)
    upload_q_hat(step, q_hat)
    mla_cache_append(step.problem, torch.from_numpy(rows.view(np.int16)).to(step.device),
                     torch.from_numpy(pos).to(step.device), step.block_table, step.cache)
    new_lens = batch.seq_lens.copy()
    new_lens[keep] += 1
    step.seq_lens.copy_(torch.from_numpy(new_lens).to(step.device))
    step.step()
    o, o_lat, lse = gpu_outputs(step)
    assert step.status() == 0
    appended = CA.append_rows(cache, rows, pos, batch.block_table, w.page_size, kv)
    if kv == "bf16":
        batch.cache_bf16 = appended
    else:
        batch.extra["cache_" + kv] = appended
    batch.seq_lens = new_lens
    reqs = list(keep)
    # lse against the absorbed form on the decode's own bf16 absorbed query
    # (the query is rounded to bf16 before the score)
    compare(O.decode(batch, requests=reqs), o, o_lat, lse, label=f"append/{name}",
            lse_ref=O.decode(batch, requests=reqs, q_hat=q_hat))
