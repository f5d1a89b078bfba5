"""GPU parity of the cache append (mla_cache_append): each request's newest
token row written into the paged cache, bf16 as is or quantised to the FP8 or
FP4 layout on the GPU.  Compared byte for byte with the oracle's append, which
uses the oracle's quantisers, on the same bf16 rows."""
import numpy as np
import pytest

import oracle as O
from oracle import cache_append as CA
from oracle import fp4 as F4
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


ROPE_THETA = 1.0e6   # GLM-4.7-Flash configuration clause


def _assert_same_cache(got, expect, kv, rope):
    """Byte for byte; with RoPE on, the rotated keys (float64 on both sides,
    rounded once) may differ where the two float64 rotations straddle a
    rounding boundary of the stored type: allowed for at most 0.5 % of the
    RoPE values, each by at most one step of that type."""
    if not rope:
        assert np.array_equal(got, expect.view(np.uint8).reshape(got.shape))
        return
    if kv == "bf16":
        g = got.view(np.uint16).reshape(-1, 576).astype(np.int64)
        e = expect.view(np.uint16).reshape(-1, 576).astype(np.int64)
        assert np.array_equal(g[:, :512], e[:, :512])
        d = np.abs(g[:, 512:] - e[:, 512:])
        assert d.max() <= 1 and (d > 0).mean() <= 5e-3, (int(d.max()), float((d > 0).mean()))
        return
    enc = F if kv == "fp8" else F4
    g = got.reshape(-1, enc.ROW_BYTES)
    e = expect.view(np.uint8).reshape(-1, enc.ROW_BYTES)
    diff_rows = np.flatnonzero((g != e).any(axis=1))
    gv, ev = enc.dequant_rows(g[diff_rows]), enc.dequant_rows(e[diff_rows])
    assert np.array_equal(gv[:, :512], ev[:, :512])
    bad = gv[:, 512:] != ev[:, 512:]
    assert bad.sum() <= 5e-3 * 64 * max(1, g.shape[0] // 1000), int(bad.sum())
    if bad.any():
        step = np.abs(ev[:, 512:]).max(axis=1, keepdims=True) / (8.0 if kv == "fp8" else 2.0)
        assert (np.abs(gv[:, 512:] - ev[:, 512:]) <= step + 1e-30).all()


@pytest.mark.parametrize("rope", [False, True])
@pytest.mark.parametrize("kv,page_size", [("bf16", 64), ("bf16", 128), ("fp8", 64), ("fp8", 128),
                                          ("fp4", 64), ("fp4", 128), ("fp4", 16)])
def test_append_matches_oracle_bytes(kv, page_size, rope):
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
    theta = ROPE_THETA if rope else 0.0
    expect = CA.append_rows(cache, rows, pos, batch.block_table, page_size, kv, rope_theta=theta)
    dev = torch.device("cuda", 0)
    cache_d = torch.from_numpy(cache.view(np.uint8).copy()).to(dev)
    rows_d = torch.from_numpy(rows.view(np.int16).copy()).to(dev)
    pos_d = torch.from_numpy(pos).to(dev)
    bt_d = torch.from_numpy(batch.block_table).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    mla_cache_append(_problem(w.batch, w, batch.num_pages, batch.block_table.shape[1], kv),
                     rows_d, pos_d, bt_d, cache_d, status, rope_theta=theta)
    torch.cuda.synchronize()
    got = cache_d.cpu().numpy()
    assert int(status.item()) == 0
    _assert_same_cache(got, expect, kv, rope)


def test_append_rope_at_long_positions():
    """Positions up to 131,071 (the long workload's contexts): the rotation
    angle of pair 0 reaches 2^17 radians; every stored RoPE key stays within
    one bf16 step of the float64 rotation."""
    from head_latent_attention_paged_gb300 import mla_cache_append
    B, P = 64, 128
    pages_per = 1024
    rng = np.random.default_rng(31)
    rows = W.f32_to_bf16_bits(rng.standard_normal((B, 576)).astype(np.float32))
    pos = rng.integers(0, pages_per * P, size=B).astype(np.int32)
    pos[:4] = [0, 1, 131071, 65536]
    # request b's position lands on physical page b; the other entries are
    # never read
    bt = np.zeros((B, pages_per), dtype=np.int32)
    bt[np.arange(B), pos // P] = np.arange(B, dtype=np.int32)
    num_pages = B
    w = W.with_overrides(W.SMALL_WORKLOADS["dense_small"], page_size=P)
    dev = torch.device("cuda", 0)
    cache_d = torch.zeros((num_pages, P, 576), dtype=torch.int16, device=dev)
    mla_cache_append(_problem(B, w, num_pages, pages_per, "bf16"),
                     torch.from_numpy(rows.view(np.int16)).to(dev), torch.from_numpy(pos).to(dev),
                     torch.from_numpy(bt).to(dev), cache_d, rope_theta=ROPE_THETA)
    torch.cuda.synchronize()
    got = cache_d.view(-1, 576)[torch.from_numpy(bt[np.arange(B), pos // P] * P + pos % P).to(dev)]
    got = got.cpu().numpy().view(np.uint16)
    want = np.stack([CA.rotate_row(rows[b], int(pos[b]), ROPE_THETA) for b in range(B)])
    assert np.array_equal(got[:, :512], rows[:, :512])
    d = np.abs(got[:, 512:].astype(np.int64) - want[:, 512:].astype(np.int64))
    assert d.max() <= 1 and (d > 0).mean() <= 5e-3


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
