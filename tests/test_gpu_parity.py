"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Small workloads are compared element by element for every (request, query
token, head); the full-size workloads run in the benchmark's launch
configuration and are compared on sampled requests and heads.
"""
import numpy as np
import pytest

import oracle as O
import workloads as W
from mla_testlib import (compare, ensure_built, gpu_outputs, make_step, oracle_q_hat,
                         upload_q_hat, with_fp8)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _run_and_compare(batch, sm_count=None, absorb=True, requests=None, heads=None, label=""):
    step = make_step(batch, sm_count=sm_count, absorb=absorb)
    step.step()
    o, o_lat, lse = gpu_outputs(step)
    assert step.status() == 0, label
    ref = O.decode(batch, requests=requests, heads=heads)
    worst = compare(ref, o, o_lat, lse, heads=heads, label=label)
    return step, worst


@pytest.mark.parametrize("name", ["tiny", "dense_small", "long_small", "sparse_small", "mtp_small"])
@pytest.mark.parametrize("garbage", ["finite", "nan"])
def test_small_workloads_match_oracle(name, garbage):
    batch = with_fp8(W.generate(W.SMALL_WORKLOADS[name], garbage=garbage), garbage)
    _run_and_compare(batch, label=f"{name}/{garbage}")


@pytest.mark.parametrize("sm_count", [1, 3, 7, 40, 152])
def test_split_invariance(sm_count):
    """Every way of cutting the streams over CTAs (one split, many, uneven)
    matches the oracle, and the splits agree with each other to the bf16
    rounding of P: probabilities are rounded to bf16 (relative error up to
    2^-9) against each split's own running maximum, so two splits round
    differently; the latent outputs agree to 2e-3 relative L2 and lse to
    5e-4."""
    batch = W.generate(W.SMALL_WORKLOADS["long_small"])
    ref_step = make_step(batch, sm_count=1)
    ref_step.step()
    o1, lat1, lse1 = gpu_outputs(ref_step)
    step, _ = _run_and_compare(batch, sm_count=sm_count, label=f"split{sm_count}")
    o2, lat2, lse2 = gpu_outputs(step)
    assert np.linalg.norm(lat2 - lat1) <= 2e-3 * np.linalg.norm(lat1)
    assert np.abs(lse2 - lse1).max() <= 5e-4


@pytest.mark.parametrize("sm_count", [7, 40])
@pytest.mark.parametrize("q_len", [1, 3])
def test_merge_is_repeatable_and_matches_separate_combine(sm_count, q_len):
    """The merge launched by mla_decode_run and a separate combine pass over
    the same partials give the same o_lat and lse, and a second run on the
    same workspace gives identical results.  q_len 3: multi-token row sets
    (two drafts, then one)."""
    batch = W.generate(W.with_overrides(W.SMALL_WORKLOADS["long_small"], q_len=q_len))
    step = make_step(batch, sm_count=sm_count)
    step.run()
    _, lat1, lse1 = gpu_outputs(step)
    step.o_lat.fill_(float("nan"))
    step.lse.fill_(float("nan"))
    step.run()
    _, lat2, lse2 = gpu_outputs(step)
    assert np.array_equal(lat1, lat2) and np.array_equal(lse1, lse2)
    step.combine()
    _, lat3, lse3 = gpu_outputs(step)
    assert np.array_equal(lat3, lat1) and np.array_equal(lse3, lse1)


def test_plan_without_host_lengths_on_few_tiles():
    """A plan made without host lengths fills every SM (152 CTAs) while the
    device lengths hold fewer tiles than that: the kernels split the work
    over at most one CTA per tile, so every CTA between a row set's first
    and last tile owners holds a partial, and the merge sees all of them."""
    batch = W.generate(W.with_overrides(W.SMALL_WORKLOADS["dense_small"], batch=3,
                                        seq_lo=300, seq_hi=900))
    step = make_step(batch, sm_count=152, plan_with_host_lengths=False)
    assert step.plan.num_ctas == 152 and sum((int(t) + 63) // 64 for t in batch.seq_lens) < 152
    step.step()
    o, o_lat, lse = gpu_outputs(step)
    assert step.status() == 0
    compare(O.decode(batch), o, o_lat, lse, label="no-host-lengths")


@pytest.mark.parametrize("name", ["dense_small", "fp8_small", "mtp_small"])
def test_chained_launches_see_their_inputs(name):
    """The decode and the merge + W_UV kernel run as programmatic dependents
    of one another: each must read what the one before wrote.  Outputs are
    filled with NaN before every step; a step over split row sets must
    rewrite all of them with the same values every time."""
    w = W.with_overrides(W.SMALL_WORKLOADS[name], seq_lo=1500, seq_hi=4000, batch=3)
    batch = W.generate(w)
    ref = None
    for trial in range(10):
        step = make_step(batch, sm_count=7)
        step.o_lat.fill_(float("nan"))
        step.lse.fill_(float("nan"))
        step.out.fill_(float("nan"))
        step.step()
        o, lat, lse = gpu_outputs(step)
        assert np.isfinite(o).all() and np.isfinite(lat).all() and np.isfinite(lse).all(), trial
        if ref is None:
            ref = (o, lat, lse)
        else:
            assert all(np.array_equal(a, b) for a, b in zip(ref, (o, lat, lse))), trial


def test_absorb_matches_oracle():
    batch = W.generate(W.SMALL_WORKLOADS["dense_small"])
    step = make_step(batch)
    torch.cuda.synchronize()
    got = step.q_hat.float().cpu().numpy().reshape(batch.workload.batch, 1, 20, 576)
    for b in range(batch.workload.batch):
        qn = O.bf16_to_f64(batch.q_nope[b, 0])
        ref = O.absorb_query(qn, O.bf16_to_f64(batch.w_uk))
        err = np.abs(got[b, 0, :, :512] - ref)
        # one bf16 rounding of an fp32 sum: within one bf16 ulp
        assert (err <= np.abs(ref) * 2.0 ** -7 + 1e-6).all()
        assert np.array_equal(got[b, 0, :, 512:], O.bf16_to_f64(batch.q_rope[b, 0]))


def test_uv_projection_matches_float64():
    from head_latent_attention_paged_gb300 import mla_uv_proj
    rng = np.random.default_rng(3)
    for rows, H in [(1, 1), (64, 20), (130, 20), (200, 7)]:
        o_lat = rng.standard_normal((rows, H, 512)).astype(np.float32)
        w_bits = W.f32_to_bf16_bits(rng.standard_normal((H, 512, 256)).astype(np.float32) / np.sqrt(512))
        o_dev = torch.from_numpy(o_lat).cuda()
        w_dev = torch.from_numpy(w_bits.view(np.int16)).cuda().view(torch.bfloat16)
        out = torch.empty((rows, H, 256), dtype=torch.bfloat16, device="cuda")
        mla_uv_proj(o_dev, w_dev, out, rows, H, torch.cuda.current_stream())
        got = out.float().cpu().numpy()
        # o_lat enters the MMA as bf16: the reference rounds it the same way
        lat_b = O.round_to_bf16(o_lat.astype(np.float64))
        ref = np.einsum("rhk,hkn->rhn", lat_b, O.bf16_to_f64(w_bits))
        assert np.abs(got - O.round_to_bf16(ref)).max() <= 2e-2
        assert np.linalg.norm(got - ref) <= 5e-3 * np.linalg.norm(ref)


@pytest.mark.parametrize("page_size", [64, 128])
def test_one_hot_gather_is_bit_exact(page_size):
    """Each head's query selects one planted token by > 100 nats: the latent
    output must equal that token's cached latent row bit for bit, whatever
    page and slot the block table maps it to."""
    w = W.with_overrides(W.SMALL_WORKLOADS["dense_small"], page_size=page_size, batch=3,
                         seq_lo=300, seq_hi=900)
    batch = W.generate(w)
    H = w.heads
    rng = np.random.default_rng(0)
    step = make_step(batch, absorb=False)
    q = np.zeros((w.batch, 1, H, 576), dtype=np.float32)
    cache = batch.cache_bf16.copy()
    planted = {}
    for b in range(w.batch):
        T = int(batch.seq_lens[b])
        # positions spread over pages, including page edges and the last token
        cands = [0, page_size - 1, page_size, T - 1] + list(rng.choice(T, size=H, replace=False))
        for h in range(H):
            t = int(cands[h % len(cands)]) if h < 4 else int(cands[h])
            planted[(b, h)] = t
        # rope dims: head h uses dim 512 + h; planted rows carry 1 there, others 0
        for t in range(T):
            page, slot = batch.block_table[b, t // page_size], t % page_size
            cache[page, slot, 512:512 + H] = 0
        for h in range(H):
            t = planted[(b, h)]
            page, slot = batch.block_table[b, t // page_size], t % page_size
            cache[page, slot, 512 + h] = 0x3F80                 # bf16 1.0
            q[b, 0, h, 512 + h] = 2048.0          # score 2048 / 16 = 128 nats
    # a token planted for two heads carries both flags; distinct heads still
    # see exactly one live row with a large score
    step.cache.copy_(torch.from_numpy(cache.view(np.int16)).view(torch.bfloat16))
    step.q_hat.copy_(torch.from_numpy(W.f32_to_bf16_bits(q.reshape(-1, H, 576)).view(np.int16)).view(torch.bfloat16))
    step.step()
    _, o_lat, lse = gpu_outputs(step)
    for (b, h), t in planted.items():
        page, slot = batch.block_table[b, t // page_size], t % page_size
        expect = W.bf16_bits_to_f32(cache[page, slot, :512])
        assert np.array_equal(o_lat[b, 0, h], expect), (b, h, t)
        assert abs(lse[b, 0, h] - 128.0) < 1e-3


def test_page_relabelling_gives_identical_bits():
    batch = W.generate(W.SMALL_WORKLOADS["dense_small"])
    s1 = make_step(batch)
    s1.step()
    _, lat1, lse1 = gpu_outputs(s1)
    perm = np.random.default_rng(1).permutation(batch.num_pages)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(batch.num_pages)
    batch.cache_bf16 = batch.cache_bf16[perm]
    bt = batch.block_table.copy()
    bt[bt >= 0] = inv[bt[bt >= 0]]
    batch.block_table = bt
    s2 = make_step(batch)
    s2.step()
    _, lat2, lse2 = gpu_outputs(s2)
    assert np.array_equal(lat1, lat2) and np.array_equal(lse1, lse2)


def test_bad_page_is_masked_and_reported():
    from head_latent_attention_paged_gb300 import MLA_STATUS_BAD_PAGE
    batch = W.generate(W.SMALL_WORKLOADS["dense_small"])
    clean = make_step(batch)
    clean.step()
    _, lat_clean, _ = gpu_outputs(clean)
    bt = batch.block_table.copy()
    bt[2, 1] = batch.num_pages + 5        # request 2, second page: out of range
    bt[3, 0] = -3                         # request 3, first page: negative
    batch.block_table = bt
    step = make_step(batch)
    step.step()
    _, lat, lse = gpu_outputs(step)
    assert step.status() & MLA_STATUS_BAD_PAGE
    for b in (0, 1, 4):
        assert np.array_equal(lat[b], lat_clean[b])
    assert np.isfinite(lat).all() and np.isfinite(lse[[0, 1, 2, 4]]).all()
    step.clear_status()
    assert step.status() == 0


def test_bad_sparse_index_is_masked_and_reported():
    from head_latent_attention_paged_gb300 import MLA_STATUS_BAD_INDEX
    batch = W.generate(W.SMALL_WORKLOADS["sparse_small"])
    idx = batch.topk_idx.copy()
    live = np.flatnonzero(idx[1] >= 0)
    idx[1, live[0]] = 10 ** 6       # past the window
    idx[1, live[1]] = -7            # negative but not -1
    ref_idx = batch.topk_idx.copy()
    ref_idx[1, live[0]] = -1
    ref_idx[1, live[1]] = -1
    batch.topk_idx = idx
    step = make_step(batch)
    step.step()
    o, o_lat, lse = gpu_outputs(step)
    assert step.status() & MLA_STATUS_BAD_INDEX
    batch.topk_idx = ref_idx
    ref = O.decode(batch)
    compare(ref, o, o_lat, lse, label="bad-index")


def test_empty_and_single_token_requests():
    """Lengths 0, 1, one page, one page + 1.  At T = 1 the lse is the single
    score, so the bf16 rounding of the absorbed query alone moves it by up to a
    few 1e-3: the decode is fed the oracle's own bf16 absorbed query and its
    lse is compared with the oracle's absorbed form on exactly that query;
    outputs are compared with the non-absorbed definition."""
    w = W.with_overrides(W.SMALL_WORKLOADS["dense_small"], seq_lens=(0, 1, 64, 65, 0, 129),
                         batch=6)
    batch = W.generate(w)
    q_hat = oracle_q_hat(batch)
    step = make_step(batch, absorb=False)
    upload_q_hat(step, q_hat)
    step.step()
    o, o_lat, lse = gpu_outputs(step)
    assert step.status() == 0
    ref = O.decode(batch)
    lse_ref = O.decode(batch, q_hat=q_hat)
    compare(ref, o, o_lat, lse, label="edge-lengths", lse_ref=lse_ref)


def test_multi_token_causal_dense():
    """q_len 4 draft tokens on the dense path: token j sees T - 4 + j + 1."""
    w = W.with_overrides(W.SMALL_WORKLOADS["dense_small"], q_len=4, batch=3, seq_lo=60, seq_hi=300)
    _run_and_compare(W.generate(w), label="dense-q4")


# ---------------------------------------------------------------------------
# full-size workloads, benchmark launch configuration, sampled outputs
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("name,requests,heads", [
    ("dense", [0, 37, 63], [0, 7, 19]),
    ("long", [3], [0, 19]),
    ("sparse", [0, 31], [0, 11, 19]),
    ("mtp", [0, 40, 63], [0, 13, 19]),
])
def test_full_size_sampled(name, requests, heads):
    batch = W.generate(W.WORKLOADS[name])
    step = make_step(batch)
    step.step()
    o, o_lat, lse = gpu_outputs(step)
    assert step.status() == 0
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    ref = O.decode(batch, requests=requests, heads=heads)
    compare(ref, o, o_lat, lse, heads=heads, label=name)


def test_long_full_size_every_request_and_head():
    """The long-context workload (8 requests of 64K-128K tokens split over
    all SMs, ~19 partials per request) in full: every request and every head
    against the oracle's absorbed form (pinned equal to the definition), and
    request 5, heads 0 and 10, against the definition itself."""
    batch = W.generate(W.WORKLOADS["long"])
    step = make_step(batch)
    step.step()
    o, o_lat, lse = gpu_outputs(step)
    assert step.status() == 0
    compare(O.decode(batch, form="absorbed"), o, o_lat, lse, label="long-absorbed")
    compare(O.decode(batch, requests=[5], heads=[0, 10]), o, o_lat, lse, heads=[0, 10],
            label="long-definition")


@pytest.mark.parametrize("name,sm_count", [("dense_small", 7), ("long_small", 40),
                                           ("long_small", 152), ("mtp_small", 11),
                                           ("sparse_small", 5), ("tiny", None)])
def test_combine_with_w_uv_matches_separate_passes(name, sm_count):
    """The step's merge inside the W_UV launch against the merge kernel alone
    followed by the stand-alone mla_uv_proj (whose row block follows the
    device's SM count, not the plan's): the same o_lat and lse bits (one
    merge arithmetic; long_small on 152 CTAs splits a row set over more than
    32), outputs within one bf16 step; both against the oracle."""
    _merge_uv_against_separate_passes(W.generate(W.SMALL_WORKLOADS[name]), sm_count, name)


def _merge_uv_against_separate_passes(batch, sm_count, label):
    step = make_step(batch, sm_count=sm_count)
    step.run()
    step.uv()
    o1, lat1, lse1 = gpu_outputs(step)
    for t in (step.out, step.o_lat, step.lse):
        t.fill_(float("nan"))
    step.step()                        # attention pass, then merge + W_UV
    o2, lat2, lse2 = gpu_outputs(step)
    assert step.status() == 0
    assert np.array_equal(lat2.view(np.uint32), lat1.view(np.uint32))
    assert np.array_equal(lse2.view(np.uint32), lse1.view(np.uint32))
    assert np.abs(o2 - o1).max() <= 2.0 ** -7 * max(1.0, np.abs(o1).max())
    ref = O.decode(batch)
    compare(ref, o1, lat1, lse1, label=f"separate/{label}")
    compare(ref, o2, lat2, lse2, label=f"combine-uv/{label}")


@pytest.mark.parametrize("batch,q_len,sm_count", [(1, 1, 152), (17, 1, 39), (40, 1, 152),
                                                  (33, 2, 152), (1, 3, 60), (50, 2, 130)])
def test_merge_uv_ragged_row_blocks(batch, q_len, sm_count):
    """The merge inside the W_UV launch splits each row block's rows between
    the two CTAs of a cluster: one row (the second CTA merges none), 17 rows
    in a block of 64 (9 and 8), a last block of 8 or 2 rows, three drafts of
    one request, 100 rows in blocks of 48 (the last of 4); each row set split
    over many CTAs.  Same checks as above."""
    w = W.with_overrides(W.SMALL_WORKLOADS["long_small"], batch=batch, q_len=q_len)
    _merge_uv_against_separate_passes(W.generate(w), sm_count, f"{batch}x{q_len}/{sm_count}")


@pytest.mark.parametrize("name", ["dense_small", "mtp_small", "tiny"])
def test_run_with_w_uk_equals_absorbed_query(name):
    """mla_decode_run given the un-absorbed query and W_UK (absorbed into the
    workspace) gives the same bits as the run on mla_q_absorb's q_hat."""
    batch = W.generate(W.SMALL_WORKLOADS[name])
    step = make_step(batch, sm_count=9)
    step.step()
    o1, lat1, lse1 = gpu_outputs(step)
    for t in (step.out, step.o_lat, step.lse):
        t.fill_(float("nan"))
    step.attend(w_uk=True)
    step.combine(uv=True)
    o2, lat2, lse2 = gpu_outputs(step)
    assert np.array_equal(lat1.view(np.uint32), lat2.view(np.uint32))
    assert np.array_equal(lse1.view(np.uint32), lse2.view(np.uint32))
    assert np.array_equal(o1, o2)


@pytest.mark.parametrize("split_tokens", [256, 512, 1024])
def test_split_kv_by_length_matches_oracle(split_tokens):
    """Split-KV with a fixed share of about split_tokens tokens per CTA (the
    grid grows with the context: more CTAs than SMs run in waves)."""
    from mla_testlib import make_step as mk
    batch = W.generate(W.SMALL_WORKLOADS["long_small"])
    step = mk(batch, split_tokens=split_tokens)
    tiles = sum((int(t) + 63) // 64 for t in batch.seq_lens)
    assert step.plan.num_ctas == -(-tiles // (split_tokens // 64))
    step.step()
    o, o_lat, lse = gpu_outputs(step)
    assert step.status() == 0
    compare(O.decode(batch), o, o_lat, lse, label=f"split_tokens{split_tokens}")


@pytest.mark.parametrize("rows,heads", [(2, 4), (130, 20), (64, 32), (17, 1)])
def test_absorb_tensor_core_matches_float64(rows, heads):
    """Query absorption on the tensor cores: within one bf16 rounding of the
    float64 product, ragged row blocks and head counts included; the RoPE
    part is copied unchanged."""
    from head_latent_attention_paged_gb300 import make_problem, mla_decode_plan, mla_q_absorb
    rng = np.random.default_rng(rows * 100 + heads)
    q = W.f32_to_bf16_bits(rng.standard_normal((rows, heads, 256)).astype(np.float32))
    w_uk = W.f32_to_bf16_bits((rng.standard_normal((heads, 512, 192)) / np.sqrt(512)).astype(np.float32))
    plan = mla_decode_plan(make_problem(rows, 1, heads, 64, 10, 4), None, 152)
    dev = torch.device("cuda", 0)
    q_d = torch.from_numpy(q.view(np.int16)).to(dev)
    w_d = torch.from_numpy(w_uk.view(np.int16)).to(dev)
    out = torch.full((rows, heads, 576), -1, dtype=torch.int16, device=dev)
    mla_q_absorb(plan, q_d, w_d, out, torch.cuda.current_stream())
    torch.cuda.synchronize()
    got = O.bf16_to_f64(out.cpu().numpy().view(np.uint16))
    ref = np.einsum("hdk,rhk->rhd", O.bf16_to_f64(w_uk), O.bf16_to_f64(q[..., :192]))
    assert (np.abs(got[..., :512] - ref) <= np.abs(ref) * 2.0 ** -7 + 1e-6).all()
    assert np.array_equal(got[..., 512:], O.bf16_to_f64(q[..., 192:]))


@pytest.mark.parametrize("name,sm_count", [("dense_small", None), ("long_small", 40),
                                           ("mtp_small", 11), ("sparse_small", 5), ("tiny", None),
                                           ("fp8_small", 9), ("fp4_small", 152)])
def test_decode_step_matches_run_and_combine(name, sm_count):
    """mla_decode_step (one call) gives the bits of mla_decode_run followed by
    mla_combine with W_UV, twice in a row on one workspace; against the
    oracle with the decode's own bf16 absorbed query for lse."""
    batch = with_fp8(W.generate(W.SMALL_WORKLOADS[name]))
    step = make_step(batch, sm_count=sm_count, absorb=False)
    q_hat = oracle_q_hat(batch)
    upload_q_hat(step, q_hat)
    step.step_two_calls()
    o1, lat1, lse1 = gpu_outputs(step)
    for trial in range(2):
        for t in (step.out, step.o_lat, step.lse):
            t.fill_(float("nan"))
        step.step()
        o2, lat2, lse2 = gpu_outputs(step)
        assert step.status() == 0, trial
        assert np.array_equal(lat2.view(np.uint32), lat1.view(np.uint32)), trial
        assert np.array_equal(lse2.view(np.uint32), lse1.view(np.uint32)), trial
        assert np.array_equal(o2, o1), trial
    compare(O.decode(batch), o2, lat2, lse2, label=f"decode-step/{name}",
            lse_ref=O.decode(batch, q_hat=q_hat))


@pytest.mark.parametrize("name,q_len", [("dense_small", 1), ("fp8_small", 1), ("mtp_small", 2),
                                        ("fp4_small", 1)])
def test_more_row_sets_than_shared_memory_holds(name, q_len):
    """512 requests of short contexts: more row sets than the decode kernel
    keeps work-split prefixes for in shared memory, so a pre-pass writes the
    tile and cost prefixes to the workspace and the decode and the merge read
    them there.  Forced splits (40 CTAs), sampled requests on both sides of
    row set 256 against the oracle; the prefixes against the tile counts."""
    w = W.with_overrides(W.SMALL_WORKLOADS[name], batch=512, seq_lo=1, seq_hi=400, q_len=q_len)
    batch = W.generate(w)
    # contexts down to one token: the decode gets the oracle's bf16 absorbed
    # query, so lse compares against the absorbed form on exactly that query
    q_hat = oracle_q_hat(batch)
    step = make_step(batch, sm_count=40, absorb=False)
    upload_q_hat(step, q_hat)
    step.step()
    o, o_lat, lse = gpu_outputs(step)
    assert step.status() == 0
    pl = step.plan
    S = pl.num_streams
    assert S == 512
    words = step.workspace[pl.ws_prefix: pl.ws_prefix + 8 * (S + 1)].cpu().view(torch.int32).numpy()
    tiles, cost = words[:S + 1].astype(np.int64), words[S + 1:].astype(np.int64)
    nt = (batch.seq_lens.astype(np.int64) + 63) // 64      # one row set per request here
    assert tiles[0] == 0 and np.array_equal(np.diff(tiles), nt)
    dc = np.diff(cost)
    assert cost[0] == 0 and np.all(dc[nt == 0] == 0)
    fixed = dc[nt > 0] - 4 * nt[nt > 0]                       # a row set's fixed cost, one value
    assert fixed.min() == fixed.max() > 0
    req = [0, 3, 255, 256, 257, 400, 511]
    compare(O.decode(batch, requests=req), o, o_lat, lse, label=f"{name}-512",
            lse_ref=O.decode(batch, requests=req, q_hat=q_hat))


@pytest.mark.parametrize("name,batch,q_len", [("sparse_small", 80, 4), ("fp8_small", 160, 2)])
def test_prefix_pass_sparse_and_fp8_drafts(name, batch, q_len):
    """Row-set counts that need the prefix pre-pass in the sparse kernel (320
    row sets of one draft each) and in the FP8 multi-token kernel (160 draft
    pairs: too many prefixes for the shared memory beside its buffers);
    split over 40 CTAs, sampled requests against the oracle."""
    w = W.with_overrides(W.SMALL_WORKLOADS[name], batch=batch, q_len=q_len, seq_lo=200,
                         seq_hi=700)
    batch_ = W.generate(w)
    q_hat = oracle_q_hat(batch_)
    step = make_step(batch_, sm_count=40, absorb=False)
    assert step.plan.prefix_pass == 1
    upload_q_hat(step, q_hat)
    step.step()
    o, o_lat, lse = gpu_outputs(step)
    assert step.status() == 0
    req = [0, 1, batch // 2, batch - 1]
    compare(O.decode(batch_, requests=req), o, o_lat, lse, label=f"{name}-prefix",
            lse_ref=O.decode(batch_, requests=req, q_hat=q_hat))
