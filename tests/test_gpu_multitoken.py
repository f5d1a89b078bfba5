"""GPU parity of the dense multi-token decode (speculative draft tokens that
share each staged page), over bf16, FP4 and FP8 caches.

With q_len = Q draft tokens per request and H heads, G = min(Q, 48 / H)
consecutive draft tokens of a request form one row set of G * H rows: every
64-token tile of the request's pages is staged once for all of them, and
each row keeps its own causal window (draft j sees positions 0 .. T - Q + j).
These checks run the CUDA path through the C ABI against the oracle, which
attends per (request, draft token, head) by the definition.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from mla_testlib import compare, ensure_built, gpu_outputs, make_step, oracle_q_hat, upload_q_hat

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


BASE = {"bf16": "dense_small", "fp4": "fp4_small", "fp8": "fp8_small"}


def _group(q_len, heads):
    g = min(q_len, 48 // heads)
    return g if g >= 2 else 1


def _run(batch, sm_count=None, label=""):
    w = batch.workload
    q_hat = oracle_q_hat(batch)
    step = make_step(batch, sm_count=sm_count, absorb=False)
    g = _group(w.q_len, w.heads)
    assert step.plan.num_streams == w.batch * -(-w.q_len // g), label
    upload_q_hat(step, q_hat)
    step.step()
    o, o_lat, lse = gpu_outputs(step)
    assert step.status() == 0, label
    compare(O.decode(batch), o, o_lat, lse, label=label, lse_ref=O.decode(batch, q_hat=q_hat))
    return o_lat, lse


@pytest.mark.parametrize("q_len,heads,causal,page_size,sm_count", [
    (2, 20, True, 64, None),     # G = 2: the GLM-4.7-Flash head count, one MTP draft pair
    (3, 20, True, 64, None),     # groups {0, 1} and {2}: a short last group
    (4, 20, False, 128, None),   # two full groups, no causal limit, 128-token pages
    (4, 12, True, 64, 9),        # G = 4 (48 rows), requests split over CTAs
    (2, 24, True, 32, 13),       # 48 rows, 32-token pages, splits
    (5, 8, True, 16, None),      # G = 5 (40 rows), 16-token pages
    (2, 32, True, 64, None),     # 48 / 32 = 1: one draft per row set
])
@pytest.mark.parametrize("kv", ["bf16", "fp4", "fp8"])
def test_multi_token_matches_oracle(q_len, heads, causal, page_size, sm_count, kv):
    base = W.SMALL_WORKLOADS[BASE[kv]]
    w = W.with_overrides(base, q_len=q_len, heads=heads, causal=causal, page_size=page_size,
                         batch=4, seq_lo=70, seq_hi=900)
    _run(W.generate(w), sm_count=sm_count,
         label=f"{kv}/q{q_len}/h{heads}/c{int(causal)}/p{page_size}")


@pytest.mark.parametrize("kv", ["bf16", "fp4", "fp8"])
def test_multi_token_short_contexts(kv):
    """Contexts shorter than the drafts: with T = 1 and Q = 3 the first two
    drafts see no position (o = 0, lse = -inf) while the last sees one; other
    lengths end inside and at the edges of a tile for some drafts only."""
    base = W.SMALL_WORKLOADS[BASE[kv]]
    w = W.with_overrides(base, q_len=3, heads=16,
                         seq_lens=(1, 2, 3, 64, 65, 66, 127, 0), batch=8)
    batch = W.generate(w, garbage="nan")
    o_lat, lse = _run(batch, label="short")
    assert np.isneginf(lse[0, 0]).all() and np.isneginf(lse[0, 1]).all()
    assert (o_lat[0, :2] == 0).all() and np.isfinite(lse[0, 2]).all()
    assert np.isneginf(lse[7]).all() and (o_lat[7] == 0).all()


def test_multi_token_one_hot_rows_are_exact():
    """A query that selects one cached position per draft and head by a score
    margin of hundreds of nats: each row's latent output is that token's
    c_kv bit for bit, so every row reads its own window and its own token."""
    B, Q, H = 3, 2, 20
    w = W.with_overrides(W.SMALL_WORKLOADS["dense_small"], q_len=Q, heads=H, batch=B,
                         seq_lo=150, seq_hi=400)
    batch = W.generate(w)
    rng = np.random.default_rng(3)
    q = np.zeros((B, Q, H, 576))
    picks = np.zeros((B, Q, H), dtype=np.int64)
    for b in range(B):
        T = int(batch.seq_lens[b])
        for j in range(Q):
            window = T - Q + j + 1
            for h in range(H):
                t = int(rng.integers(0, window))
                picks[b, j, h] = t
                page, slot = batch.block_table[b, t // w.page_size], t % w.page_size
                row = O.bf16_to_f64(batch.cache_bf16[page, slot])
                q[b, j, h] = O.round_to_bf16(row * 64.0)   # score ~ 64 * |row|^2 / 16
    step = make_step(batch, absorb=False)
    upload_q_hat(step, q)
    step.step()
    _, o_lat, _ = gpu_outputs(step)
    assert step.status() == 0
    for b in range(B):
        for j in range(Q):
            for h in range(H):
                t = picks[b, j, h]
                page, slot = batch.block_table[b, t // w.page_size], t % w.page_size
                expect = O.bf16_to_f64(batch.cache_bf16[page, slot, :512]).astype(np.float32)
                assert np.array_equal(o_lat[b, j, h], expect), (b, j, h)
