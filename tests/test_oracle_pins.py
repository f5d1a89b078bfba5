"""Pins for the CPU oracle: checks it against what the pages and the
mathematics fix, never against itself.

Each test names the kind of evidence: a value the pages print (golden
fixtures under tests/golden/), a closed form, an invariant, a special case
that reduces to a library routine, or brute force on a tiny case.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as O
from oracle import fp4 as F4
from oracle import fp8 as F
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand_problem(rng, H=3, n=17, Dc=O.D_C, Dr=O.D_R, Dn=O.D_NOPE, Dv=O.D_V):
    q_nope = rng.standard_normal((H, Dn))
    q_rope = rng.standard_normal((H, Dr))
    w_uk = rng.standard_normal((H, Dc, Dn)) / math.sqrt(Dc)
    w_uv = rng.standard_normal((H, Dc, Dv)) / math.sqrt(Dc)
    c_kv = rng.standard_normal((n, Dc))
    k_rope = rng.standard_normal((n, Dr))
    return q_nope, q_rope, w_uk, w_uv, c_kv, k_rope


# ---------------------------------------------------------------------------
# values the pages print
# ---------------------------------------------------------------------------
def test_kv_bytes_per_token_closed_form():
    g = _golden("kv_bytes_per_token.json")
    got = O.kv_cache_bytes_per_token(g["n_layers"], g["kv_lora_rank"], g["qk_rope_head_dim"],
                                     g["bytes_per_elem"])
    assert got == g["bytes_per_token_all_layers"]
    assert round(got / 1024, 1) == g["kib_per_token_rounded"]
    assert O.kv_cache_bytes_per_token(1) == g["bytes_per_token_one_layer"]
    # the generator's caches hold exactly that many bytes per token and layer
    b = W.generate(W.WORKLOADS["tiny"])
    assert b.cache_bf16.nbytes // (b.num_pages * b.workload.page_size) == g["bytes_per_token_one_layer"]
    assert W.FP8_ROW_BYTES == O.D_QK + O.D_QK // g["fp8_values_per_scale"] == F.ROW_BYTES


def test_topk_buffer_width_golden():
    for c in _golden("topk_width.json")["cases"]:
        assert O.topk_buffer_width(c["topk"], c["kpool"]) == c["width"], c
        assert O.topk_buffer_width(c["topk"], c["kpool"]) % 128 == 0


def test_paged_gather_golden():
    g = _golden("paged_gather.json")
    pages, slots = O.physical_rows(np.array(g["block_table_row"]), np.array(g["positions"]),
                                   g["page_size"])
    assert pages.tolist() == g["pages"]
    assert slots.tolist() == g["slots"]


def test_visibility_golden():
    g = _golden("visibility.json")
    for c in g["dense"]:
        got = O.visible_positions(c["T"], c["Q"], c["j"], causal=True)
        assert got.tolist() == c["visible"], c
    for c in g["sparse"]:
        got = O.visible_positions(c["T"], c["Q"], c["j"], causal=True,
                                  topk_row=np.array(c["row"]))
        assert got.tolist() == c["visible"], c
    # causal=0: every query token of a request sees the whole context
    for c in g["dense_non_causal"]:
        got = O.visible_positions(c["T"], c["Q"], c["j"], causal=False)
        assert got.tolist() == c["visible"], c
    for c in g["sparse_non_causal"]:
        got = O.visible_positions(c["T"], c["Q"], c["j"], causal=False,
                                  topk_row=np.array(c["row"]))
        assert got.tolist() == c["visible"], c


def test_bf16_codes_golden():
    """Hand-decoded bf16 bit patterns (normal, subnormal, signed zero,
    infinities, NaN) against the oracle's decoder."""
    for code, val in _golden("bf16_codes.json")["codes"]:
        got = O.bf16_to_f64(np.array([int(code, 16)], dtype=np.uint16))[0]
        if val == "nan":
            assert np.isnan(got), code
        elif val in ("inf", "-inf"):
            assert got == float(val), code
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), code


def test_bf16_decoder_all_patterns_match_torch():
    """All 65,536 bf16 bit patterns: the oracle's decoder agrees with torch's
    bfloat16 -> float64 conversion (a library routine), NaNs by class and
    zeros by sign."""
    torch = pytest.importorskip("torch")
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = O.bf16_to_f64(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert int(nan.sum()) == 2 * 127      # exponent field 255 with a non-zero mantissa
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def _hex(s):
    return int(s, 16)


def test_fp8_codes_golden():
    g = _golden("fp8_codes.json")
    for code, val in g["e4m3"]:
        got = F.e4m3_to_f64(np.array([_hex(code)], dtype=np.uint8))[0]
        if val == "nan":
            assert np.isnan(got)
        else:
            assert got == val and math.copysign(1, got) == math.copysign(1, val), code
    for code, val in g["e8m0"]:
        got = F.e8m0_to_f64(np.array([_hex(code)], dtype=np.uint8))[0]
        if val == "nan":
            assert np.isnan(got)
        else:
            assert got == val, code


def test_fp8_quantiser_golden_groups():
    row = np.zeros((1, F.D_QK))
    row[0, 0:32] = 448.0           # group 0
    row[0, 32] = 1.0               # group 1
    # group 2 all zero
    row[0, 96] = -896.0            # group 3
    q = F.quantize_rows(row)[0]
    vals, scales = q[:F.D_QK], q[F.D_QK:]
    assert scales[0] == 127 and (vals[0:32] == 0x7E).all()
    assert scales[1] == 119 and vals[32] == 0x78 and (vals[33:64] == 0).all()
    assert scales[2] == 0 and (vals[64:96] == 0).all()
    assert scales[3] == 128 and vals[96] == 0xFE and (vals[97:128] == 0).all()


def test_fp4_codes_golden():
    g = _golden("fp4_codes.json")
    for code, val in g["e2m1"]:
        got = F4.e2m1_to_f64(np.array([code]))[0]
        assert got == val and math.copysign(1, got) == math.copysign(1, val), code
    assert F4.ROW_BYTES == g["row_bytes_576"]
    # the same reading on the 512-value rows of the record gives its 288 bytes
    assert 512 // 2 + 512 // F4.GROUP == g["row_bytes_512"]
    pk = g["packing"]
    packed = F4.pack_codes(np.array(pk["codes"], dtype=np.uint8))
    assert [int(x) for x in packed] == [int(b, 16) for b in pk["bytes"]]
    assert list(F4.unpack_codes(packed)) == pk["codes"]
    for code, val in _golden("fp8_codes.json")["e8m0"]:
        got = F4.e8m0_to_f64(np.array([_hex(code)], dtype=np.uint8))[0]
        assert np.isnan(got) if val == "nan" else got == val, code


def test_fp4_quantiser_golden_groups():
    g = _golden("fp4_codes.json")["quantise_groups"]
    row = np.zeros((1, F4.D_QK))
    row[0, 0:16] = 6.0                                   # group 0
    row[0, 16] = 1.0                                     # group 1
    # group 2 all zero
    row[0, 48] = -12.0                                   # group 3
    ties = [float(v) for v in g[4]["group"].split(", ")]
    row[0, 64:80] = ties                                 # group 4
    q = F4.quantize_rows(row)[0]
    codes, scales = F4.unpack_codes(q[:F4.CODE_BYTES]), q[F4.CODE_BYTES:]
    assert scales[0] == g[0]["scale_byte"] and (codes[0:16] == 7).all()
    assert scales[1] == g[1]["scale_byte"] and codes[16] == g[1]["first_code"]
    assert (codes[17:32] == 0).all()
    assert scales[2] == g[2]["scale_byte"] and (codes[32:48] == 0).all()
    assert scales[3] == g[3]["scale_byte"] and codes[48] == g[3]["first_code"]
    assert (codes[49:64] == 0).all()
    assert scales[4] == g[4]["scale_byte"] and list(codes[64:80]) == g[4]["codes"]


def test_fp4_quantiser_brute_force_nearest_code():
    """Brute force over the 16 codes: each value's code is the one nearest
    to x / 2**e, ties to the even code; the scale is the smallest power of two
    that brings the group's amax to 6 or below; the round trip is within half
    the widest grid step (2**e)."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((48, F4.D_QK)) * np.exp(rng.uniform(-8, 8, size=(48, 1)))
    x[0, :40] = 0.0
    q = F4.quantize_rows(x)
    codes = F4.unpack_codes(q[:, :F4.CODE_BYTES]).astype(np.int64)
    e = q[:, F4.CODE_BYTES:].astype(np.int64) - 127
    grid = np.array([F4.e2m1_to_f64(np.array([c]))[0] for c in range(16)])
    for r in range(x.shape[0]):
        for gi in range(F4.N_GROUPS):
            xs = x[r, 16 * gi:16 * gi + 16]
            amax = np.abs(xs).max()
            if amax == 0:
                assert e[r, gi] == -127 and (codes[r, 16 * gi:16 * gi + 16] == 0).all()
                continue
            k = int(e[r, gi])
            assert amax / 2.0 ** k <= 6.0 < amax / 2.0 ** (k - 1)
            for i, v in enumerate(xs / 2.0 ** k):
                d = np.abs(grid - v)
                best = [c for c in range(16) if d[c] == d.min()]
                # the nearest magnitude, its sign from the value
                cand = [c for c in best if (c >= 8) == (np.signbit(v))] or best
                want = min(cand, key=lambda c: (c & 1, c))   # ties: even code
                assert codes[r, 16 * gi + i] == want, (r, gi, i, v)
    back = F4.dequant_rows(q)
    bound = np.repeat(2.0 ** e.astype(np.float64), 16, axis=1)
    assert (np.abs(back - x) <= bound + 1e-300).all()


# ---------------------------------------------------------------------------
# library routines
# ---------------------------------------------------------------------------
def test_e4m3_table_matches_torch():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    mine = F.e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])
    assert np.array_equal(np.signbit(mine[ok]), np.signbit(ref[ok]))


def test_e8m0_table_matches_torch():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e8m0fnu"):
        pytest.skip("torch lacks float8_e8m0fnu")
    codes = np.arange(256, dtype=np.uint8)
    mine = F.e8m0_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(mine), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(mine[ok], ref[ok])


def test_fp8_quantiser_round_trip_matches_torch_rounding():
    """x / 2**e rounded by torch's float8_e4m3fn cast (round to nearest even)
    must equal the quantiser's codes, and dequantising gives back the value
    within half a quantum."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, F.D_QK)) * np.exp(rng.uniform(-6, 6, size=(64, 1)))
    q = F.quantize_rows(x)
    scales = F.e8m0_to_f64(q[:, F.D_QK:])
    scaled = x / np.repeat(scales, 32, axis=1)
    assert np.abs(scaled).max() <= 448.0
    ref_codes = torch.from_numpy(scaled).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ref_codes, q[:, :F.D_QK])
    back = F.dequant_rows(q)
    amax = np.abs(x.reshape(64, 18, 32)).max(axis=2)
    # largest spacing in a group is 32 * 2**e (binade [256, 448] has spacing 32)
    bound = np.repeat(scales * 16.0, 32, axis=1)
    assert (np.abs(back - x) <= bound + 1e-300).all()
    # amax lands in (224, 448] after scaling: e is the smallest fitting power
    s_amax = amax / scales
    assert (s_amax <= 448.0).all() and (s_amax > 224.0).all()


def test_matches_torch_sdpa():
    """Softmax attention on the decompressed per-head K/V equals torch's
    scaled_dot_product_attention (float64, CPU); lse equals torch.logsumexp."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    q_nope, q_rope, w_uk, w_uv, c_kv, k_rope = _rand_problem(rng, H=4, n=50)
    scale = 1.0 / 16.0
    o, lse, o_lat = O.attend_non_absorbed(q_nope, q_rope, w_uk, w_uv, c_kv, k_rope, scale)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    for h in range(4):
        K = torch.cat([t(c_kv) @ t(w_uk[h]), t(k_rope)], dim=1)         # [n, 256]
        V = t(c_kv) @ t(w_uv[h])                                          # [n, 256]
        qv = torch.cat([t(q_nope[h]), t(q_rope[h])])[None, None, None, :]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qv, K[None, None], V[None, None], scale=scale)[0, 0, 0].numpy()
        assert np.allclose(o[h], ref, rtol=1e-12, atol=1e-13)
        ref_lse = torch.logsumexp((K @ qv[0, 0, 0]) * scale, dim=0).item()
        assert abs(lse[h] - ref_lse) < 1e-12
        # latent output up-projects to o
        assert np.allclose(o_lat[h] @ w_uv[h], o[h], rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# closed forms and special cases
# ---------------------------------------------------------------------------
def test_hand_worked_tiny_dims():
    """Dc=2, Dr=1, Dn=1, Dv=1, one head, two tokens, scale 1: every quantity
    worked by hand.  k_nope = c @ W_UK = [1, 3]; scores = [1*1 + 0*2, 3*1 + 1*2]
    = [1, 5]; v = c @ W_UV = [2, 4]."""
    q_nope = np.array([[1.0]])
    q_rope = np.array([[2.0]])
    w_uk = np.array([[[1.0], [0.0]]])
    w_uv = np.array([[[0.0], [1.0]]])
    c_kv = np.array([[1.0, 2.0], [3.0, 4.0]])
    k_rope = np.array([[0.0], [1.0]])
    o, lse, o_lat = O.attend_non_absorbed(q_nope, q_rope, w_uk, w_uv, c_kv, k_rope, 1.0)
    e1, e5 = math.exp(1.0), math.exp(5.0)
    assert abs(lse[0] - (5.0 + math.log1p(math.exp(-4.0)))) < 1e-14
    assert abs(o[0, 0] - (2 * e1 + 4 * e5) / (e1 + e5)) < 1e-14
    p0 = e1 / (e1 + e5)
    assert np.allclose(o_lat[0], [p0 * 1 + (1 - p0) * 3, p0 * 2 + (1 - p0) * 4], rtol=1e-14)


def test_single_token():
    rng = np.random.default_rng(1)
    q_nope, q_rope, w_uk, w_uv, c_kv, k_rope = _rand_problem(rng, H=2, n=1)
    o, lse, o_lat = O.attend_non_absorbed(q_nope, q_rope, w_uk, w_uv, c_kv, k_rope, 0.0625)
    for h in range(2):
        s0 = (c_kv[0] @ w_uk[h] @ q_nope[h] + k_rope[0] @ q_rope[h]) * 0.0625
        assert abs(lse[h] - s0) < 1e-12
        assert np.allclose(o[h], w_uv[h].T @ c_kv[0], rtol=1e-13, atol=1e-14)
        assert np.array_equal(o_lat[h], c_kv[0])


def test_zero_query_gives_mean_and_log_count():
    rng = np.random.default_rng(2)
    q_nope, q_rope, w_uk, w_uv, c_kv, k_rope = _rand_problem(rng, H=2, n=37)
    q_nope[:] = 0
    q_rope[:] = 0
    o, lse, o_lat = O.attend_non_absorbed(q_nope, q_rope, w_uk, w_uv, c_kv, k_rope, 0.0625)
    for h in range(2):
        assert abs(lse[h] - math.log(37)) < 1e-13
        assert np.allclose(o[h], (c_kv @ w_uv[h]).mean(axis=0), rtol=1e-12, atol=1e-14)
        assert np.allclose(o_lat[h], c_kv.mean(axis=0), rtol=1e-12, atol=1e-14)


def test_two_tokens_sigmoid():
    rng = np.random.default_rng(3)
    q_nope, q_rope, w_uk, w_uv, c_kv, k_rope = _rand_problem(rng, H=1, n=2)
    o, lse, _ = O.attend_non_absorbed(q_nope, q_rope, w_uk, w_uv, c_kv, k_rope, 0.0625)
    s = [(c_kv[t] @ w_uk[0] @ q_nope[0] + k_rope[t] @ q_rope[0]) * 0.0625 for t in range(2)]
    p0 = 1.0 / (1.0 + math.exp(s[1] - s[0]))
    v = c_kv @ w_uv[0]
    assert np.allclose(o[0], p0 * v[0] + (1 - p0) * v[1], rtol=1e-12, atol=1e-14)
    assert abs(lse[0] - max(s) - math.log1p(math.exp(min(s) - max(s)))) < 1e-13


def test_rope_only_and_nope_only_scores():
    """q_nope = 0 leaves the RoPE part alone in the scores; k_rope = q_rope = 0
    (the NoPE special case: vllm API docs, vllm.models.glm5next.common.model,
    load_weights: NoPE checkpoints zero-pad the RoPE rows) leaves the latent
    part alone, equal to an oracle run with the RoPE dims removed."""
    rng = np.random.default_rng(4)
    q_nope, q_rope, w_uk, w_uv, c_kv, k_rope = _rand_problem(rng, H=2, n=9)
    qn0 = np.zeros_like(q_nope)
    o, lse, _ = O.attend_non_absorbed(qn0, q_rope, w_uk, w_uv, c_kv, k_rope, 0.5)
    for h in range(2):
        s = (k_rope @ q_rope[h]) * 0.5
        m = s.max()
        assert abs(lse[h] - (m + math.log(np.exp(s - m).sum()))) < 1e-12
    o1, lse1, _ = O.attend_non_absorbed(q_nope, np.zeros_like(q_rope), w_uk, w_uv, c_kv,
                                        np.zeros_like(k_rope), 0.5)
    o2, lse2, _ = O.attend_non_absorbed(q_nope, q_rope[:, :0], w_uk, w_uv, c_kv,
                                        k_rope[:, :0], 0.5)
    assert np.allclose(o1, o2, rtol=1e-13, atol=1e-15) and np.allclose(lse1, lse2, rtol=1e-13)


def test_one_hot_dominant_token():
    """A token whose score exceeds all others by > 100 nats takes all the
    weight: o_lat equals its latent row (to float64 resolution)."""
    rng = np.random.default_rng(6)
    q_nope, q_rope, w_uk, w_uv, c_kv, k_rope = _rand_problem(rng, H=1, n=40)
    k_rope[17] = q_rope[0] * 40.0          # + 40 * |q_rope|^2 * scale >> 100
    o, lse, o_lat = O.attend_non_absorbed(q_nope, q_rope, w_uk, w_uv, c_kv, k_rope, 0.0625)
    assert np.allclose(o_lat[0], c_kv[17], rtol=1e-15, atol=1e-300)
    assert np.allclose(o[0], w_uv[0].T @ c_kv[17], rtol=1e-12)


def test_score_shift_invariance():
    """Adding the same vector u to every k_rope shifts every score by
    scale * q_rope . u: o is unchanged, lse moves by exactly that."""
    rng = np.random.default_rng(7)
    q_nope, q_rope, w_uk, w_uv, c_kv, k_rope = _rand_problem(rng, H=3, n=25)
    u = rng.standard_normal(O.D_R)
    o1, lse1, _ = O.attend_non_absorbed(q_nope, q_rope, w_uk, w_uv, c_kv, k_rope, 0.0625)
    o2, lse2, _ = O.attend_non_absorbed(q_nope, q_rope, w_uk, w_uv, c_kv, k_rope + u, 0.0625)
    assert np.allclose(o1, o2, rtol=1e-11, atol=1e-13)
    assert np.allclose(lse2 - lse1, (q_rope @ u) * 0.0625, rtol=1e-11, atol=1e-12)


def test_token_permutation_invariance():
    rng = np.random.default_rng(8)
    q_nope, q_rope, w_uk, w_uv, c_kv, k_rope = _rand_problem(rng, H=2, n=30)
    perm = rng.permutation(30)
    a = O.attend_non_absorbed(q_nope, q_rope, w_uk, w_uv, c_kv, k_rope, 0.0625)
    b = O.attend_non_absorbed(q_nope, q_rope, w_uk, w_uv, c_kv[perm], k_rope[perm], 0.0625)
    for x, y in zip(a, b):
        assert np.allclose(x, y, rtol=1e-12, atol=1e-14)


def test_absorbed_equals_non_absorbed():
    """Associativity: scoring W_UK q_nope against the latent, and up-projecting
    the latent-space output, is the same as decompressing K and V."""
    rng = np.random.default_rng(9)
    q_nope, q_rope, w_uk, w_uv, c_kv, k_rope = _rand_problem(rng, H=5, n=300)
    a = O.attend_non_absorbed(q_nope, q_rope, w_uk, w_uv, c_kv, k_rope, 0.0625)
    b = O.attend_absorbed(O.absorb_query(q_nope, w_uk), q_rope, w_uv, c_kv, k_rope, 0.0625)
    for x, y in zip(a, b):
        assert np.linalg.norm(x - y) <= 1e-10 * np.linalg.norm(x)


def test_absorb_query_brute_force():
    rng = np.random.default_rng(10)
    H, Dc, Dn = 2, 6, 3
    w_uk = rng.standard_normal((H, Dc, Dn))
    q = rng.standard_normal((H, Dn))
    got = O.absorb_query(q, w_uk)
    for h in range(H):
        for c in range(Dc):
            ref = sum(w_uk[h, c, n] * q[h, n] for n in range(Dn))
            assert abs(got[h, c] - ref) < 1e-13


def test_split_and_combine_equals_whole():
    """Attention over a token set equals the LSE-merge of attention over any
    partition of it (including an empty part)."""
    rng = np.random.default_rng(12)
    q_nope, q_rope, w_uk, w_uv, c_kv, k_rope = _rand_problem(rng, H=3, n=90)
    whole = O.attend_non_absorbed(q_nope, q_rope, w_uk, w_uv, c_kv, k_rope, 0.0625)
    cuts = [0, 13, 13, 64, 90]
    parts = [O.attend_non_absorbed(q_nope, q_rope, w_uk, w_uv, c_kv[a:b], k_rope[a:b], 0.0625)
             for a, b in zip(cuts[:-1], cuts[1:])]
    o, lse = O.combine_partials([p[2] for p in parts], [p[1] for p in parts])
    assert np.allclose(lse, whole[1], rtol=1e-13)
    assert np.allclose(o, whole[2], rtol=1e-12, atol=1e-14)


def test_empty_visible_set():
    rng = np.random.default_rng(13)
    q_nope, q_rope, w_uk, w_uv, c_kv, k_rope = _rand_problem(rng, H=2, n=0)
    o, lse, o_lat = O.attend_non_absorbed(q_nope, q_rope, w_uk, w_uv, c_kv, k_rope, 0.0625)
    assert (o == 0).all() and (o_lat == 0).all() and np.isneginf(lse).all()


def test_round_to_bf16_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(14)
    x = rng.standard_normal(10000) * np.exp(rng.uniform(-30, 30, 10000))
    x[:4] = [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]   # ties to even
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(O.round_to_bf16(x), ref)


# ---------------------------------------------------------------------------
# batch driver: paging and sparse handling
# ---------------------------------------------------------------------------
def test_decode_page_permutation_invariance():
    """Relabelling physical pages (with a consistent block table) leaves every
    output bit-identical."""
    w = W.with_overrides(W.SMALL_WORKLOADS["dense_small"], batch=2, heads=3)
    b = W.generate(w)
    ref = O.decode(b)
    perm = np.random.default_rng(0).permutation(b.num_pages)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(b.num_pages)
    b.cache_bf16 = b.cache_bf16[perm]        # new page i holds old page perm[i]
    bt = b.block_table.copy()
    bt[bt >= 0] = inv[bt[bt >= 0]]
    b.block_table = bt
    got = O.decode(b)
    for k in ref:
        for x, y in zip(ref[k], got[k]):
            assert np.array_equal(x, y)


def test_decode_sparse_full_window_equals_dense_and_minus_one_is_absent():
    w = W.with_overrides(W.SMALL_WORKLOADS["sparse_small"], batch=1, heads=2, q_len=2,
                         seq_lo=300, seq_hi=300, topk=0, topk_pad_slots=0)
    b = W.generate(w)
    dense = O.decode(b)
    # sparse rows listing each query token's full window in order, plus -1 pads
    ws = W.with_overrides(w, topk=300, topk_pad_slots=84)
    bs = W.generate(w)
    bs.workload = ws
    rows = np.full((2, 384), -1, dtype=np.int32)
    for j in range(2):
        vis = np.arange(300 - 2 + j + 1)
        slots = np.sort(np.random.default_rng(j).choice(384, size=len(vis), replace=False))
        rows[j, slots] = vis
    bs.topk_idx = rows
    sparse = O.decode(bs)
    for k in dense:
        for x, y in zip(dense[k], sparse[k]):
            assert np.allclose(x, y, rtol=1e-12, atol=1e-14)


def test_fp8_decode_uses_dequantised_bytes():
    """The FP8 path of the driver attends over exactly e4m3 * 2**(s-127) of the
    stored bytes: equal to the bf16-free float path on the dequantised rows."""
    w = W.with_overrides(W.SMALL_WORKLOADS["fp8_small"], batch=2, heads=2, seq_lo=70,
                         seq_hi=140)
    b = W.generate(w, fp8_source="float")
    b.extra["cache_fp8"] = F.quantize_pages(b.latent_f32, b.slot_valid)
    got = O.decode(b)
    raw = b.extra["cache_fp8"].reshape(b.num_pages, w.page_size, F.ROW_BYTES)
    for (bi, j), (o, lse, o_lat) in got.items():
        T = int(b.seq_lens[bi])
        pages, slots = O.physical_rows(b.block_table[bi], np.arange(T), w.page_size)
        rows = F.dequant_rows(raw[pages, slots])
        ref = O.attend_non_absorbed(O.bf16_to_f64(b.q_nope[bi, j]), O.bf16_to_f64(b.q_rope[bi, j]),
                                    O.bf16_to_f64(b.w_uk), O.bf16_to_f64(b.w_uv),
                                    rows[:, :512], rows[:, 512:], w.sm_scale)
        assert np.allclose(o, ref[0], rtol=1e-13, atol=1e-15)
        # dequantised rows stay close to the float latent they came from
        assert np.abs(rows - b.latent_f32[pages, slots]).max() < 0.07 * np.abs(rows).max()


def test_fp4_decode_uses_dequantised_bytes():
    """The FP4 path of the driver attends over exactly e2m1 * 2**(s-127) of the
    stored bytes: equal to the float path on the dequantised rows."""
    w = W.with_overrides(W.SMALL_WORKLOADS["fp4_small"], batch=2, heads=2, seq_lo=70,
                         seq_hi=140)
    b = W.generate(w, fp8_source="float")
    b.extra["cache_fp4"] = F4.quantize_pages(b.latent_f32, b.slot_valid)
    got = O.decode(b)
    raw = b.extra["cache_fp4"].reshape(b.num_pages, w.page_size, F4.ROW_BYTES)
    for (bi, j), (o, lse, o_lat) in got.items():
        T = int(b.seq_lens[bi])
        pages, slots = O.physical_rows(b.block_table[bi], np.arange(T), w.page_size)
        rows = F4.dequant_rows(raw[pages, slots])
        ref = O.attend_non_absorbed(O.bf16_to_f64(b.q_nope[bi, j]), O.bf16_to_f64(b.q_rope[bi, j]),
                                    O.bf16_to_f64(b.w_uk), O.bf16_to_f64(b.w_uv),
                                    rows[:, :512], rows[:, 512:], w.sm_scale)
        assert np.allclose(o, ref[0], rtol=1e-13, atol=1e-15)
        # FP4 keeps one fraction bit: within 2**e of the float latent
        assert np.abs(rows - b.latent_f32[pages, slots]).max() < 0.35 * np.abs(rows).max()


def test_generator_structure():
    """Block tables reference distinct in-range pages; live slots match
    seq_lens; sparse rows hold distinct in-window indices and -1 pads."""
    for name, w in W.SMALL_WORKLOADS.items():
        b = W.generate(w)
        used = b.block_table[b.block_table >= 0]
        assert len(np.unique(used)) == len(used) and used.max() < b.num_pages
        assert b.slot_valid.sum() == b.seq_lens.sum()
        if w.topk:
            for r in range(w.batch * w.q_len):
                bi, j = divmod(r, w.q_len)
                row = b.topk_idx[r]
                live = row[row >= 0]
                assert len(np.unique(live)) == len(live) == min(w.topk, int(b.seq_lens[bi]) - w.q_len + j + 1)
                assert live.max() <= int(b.seq_lens[bi]) - w.q_len + j
                assert (row == -1).sum() == w.topk_width - len(live)


def test_cache_append_places_rows_and_leaves_the_rest():
    """The appended row lands at page block_table[b, pos // P], slot pos % P
    (bf16: bit for bit; FP8: the quantiser's bytes, which dequantise to within
    half an e4m3 step of each value); every other byte is unchanged; -1 and
    out-of-range positions or pages append nothing."""
    from oracle import cache_append as CA
    rng = np.random.default_rng(5)
    P, num_pages, B = 64, 12, 5
    bt = rng.permutation(num_pages)[: B * 2].reshape(B, 2).astype(np.int32)
    bt[4, 1] = num_pages + 3                      # a page id outside the pool
    rows = W.f32_to_bf16_bits(rng.standard_normal((B, 576)).astype(np.float32))
    pos = np.array([0, 63, 64, -1, 100], dtype=np.int32)   # request 4 -> bad page
    cache = W.f32_to_bf16_bits(rng.standard_normal((num_pages, P, 576)).astype(np.float32))
    out = CA.append_rows(cache, rows, pos, bt, P, "bf16")
    written = {(int(bt[0, 0]), 0): 0, (int(bt[1, 0]), 63): 1, (int(bt[2, 1]), 0): 2}
    for (pg, sl), b in written.items():
        assert np.array_equal(out[pg, sl], rows[b])
    mask = np.ones((num_pages, P), dtype=bool)
    for (pg, sl) in written:
        mask[pg, sl] = False
    assert np.array_equal(out[mask], cache[mask])
    # FP8: same placement, quantised bytes
    raw = np.zeros((num_pages, P * F.ROW_BYTES), dtype=np.uint8)
    out8 = CA.append_rows(raw, rows, pos, bt, P, "fp8").reshape(num_pages, P, F.ROW_BYTES)
    for (pg, sl), b in written.items():
        got = F.dequant_rows(out8[pg, sl])
        x = O.bf16_to_f64(rows[b])
        scale = np.repeat(F.e8m0_to_f64(out8[pg, sl, 576:]), 32)
        # e4m3 has 3 fraction bits: |error| <= half a step <= 2^-4 * |value| + subnormal step
        assert np.all(np.abs(got - x) <= np.maximum(np.abs(x) * 2.0 ** -4, scale * 2.0 ** -10))
        assert np.array_equal(out8[pg, sl], F.quantize_rows(x[None, :])[0])
    mask8 = np.ones((num_pages, P), dtype=bool)
    for (pg, sl) in written:
        mask8[pg, sl] = False
    assert not out8[mask8].any()
    # FP4: same placement, 324-byte rows of the FP4 quantiser
    raw4 = np.zeros((num_pages, P * F4.ROW_BYTES), dtype=np.uint8)
    out4 = CA.append_rows(raw4, rows, pos, bt, P, "fp4").reshape(num_pages, P, F4.ROW_BYTES)
    for (pg, sl), b in written.items():
        x = O.bf16_to_f64(rows[b])
        assert np.array_equal(out4[pg, sl], F4.quantize_rows(x[None, :])[0])
        scale = np.repeat(F4.e8m0_to_f64(out4[pg, sl, F4.CODE_BYTES:]), 16)
        assert np.all(np.abs(F4.dequant_rows(out4[pg, sl]) - x) <= scale)
    assert not out4[mask8].any()


# ---------------------------------------------------------------------------
# RoPE on the cached key (append step)
# ---------------------------------------------------------------------------
from oracle import rope as R   # noqa: E402


def test_rope_golden_hand_worked():
    """Unit vectors rotated by hand from the closed form (golden fixture)."""
    g = _golden("rope.json")
    f = R.inverse_frequencies(g["dim"], g["theta"])
    assert f[1] == pytest.approx(g["inverse_frequency_pair_1"], rel=1e-15)
    assert f[16] == pytest.approx(g["inverse_frequency_pair_16"], rel=1e-15)
    for c in g["cases"]:
        x = np.zeros(g["dim"])
        x[c["x_index"]] = 1.0
        y = R.rope_rotate(x, c["pos"], g["theta"])
        want = np.zeros(g["dim"])
        for k, v in c["nonzero_out"].items():
            want[int(k)] = v
        np.testing.assert_allclose(y, want, rtol=0, atol=1e-12, err_msg=c["what"])


def test_rope_invariants():
    """Rotation preserves every pair's norm, position 0 is the identity, and
    q . k depends only on the difference of the two positions."""
    rng = np.random.default_rng(21)
    q, k = rng.standard_normal(64), rng.standard_normal(64)
    assert np.array_equal(R.rope_rotate(k, 0), k)
    y = R.rope_rotate(k, 123457)
    np.testing.assert_allclose(y[0::2] ** 2 + y[1::2] ** 2, k[0::2] ** 2 + k[1::2] ** 2, rtol=1e-12)
    for m, n, d in [(5, 2, 7), (131071, 65536, 1000), (0, 9, 40000)]:
        a = R.rope_rotate(q, m) @ R.rope_rotate(k, n)
        b = R.rope_rotate(q, m + d) @ R.rope_rotate(k, n + d)
        assert a == pytest.approx(b, rel=1e-9, abs=1e-9)
    # rotating by m then n is rotating by m + n
    np.testing.assert_allclose(R.rope_rotate(R.rope_rotate(k, 300), 700), R.rope_rotate(k, 1000),
                               rtol=0, atol=1e-12)


def test_rope_matches_complex_multiplication():
    """Each pair (x0, x1) read as the complex number x0 + i x1 is multiplied
    by exp(i a): an independent statement of the same rotation."""
    rng = np.random.default_rng(22)
    k = rng.standard_normal(64)
    pos = 4321
    z = (k[0::2] + 1j * k[1::2]) * np.exp(1j * pos * 1e6 ** (-np.arange(32) * 2 / 64))
    y = R.rope_rotate(k, pos)
    np.testing.assert_allclose(y[0::2], z.real, atol=1e-12)
    np.testing.assert_allclose(y[1::2], z.imag, atol=1e-12)


def test_append_rotates_only_the_rope_key():
    """With rope_theta the appended row's latent is stored unchanged and its
    RoPE key is the rotated key rounded to bf16; without it, the row as is."""
    from oracle import cache_append as CA
    rng = np.random.default_rng(23)
    rows = W.f32_to_bf16_bits(rng.standard_normal((2, 576)).astype(np.float32))
    cache = np.zeros((4, 64, 576), dtype=np.uint16)
    bt = np.array([[2, 0], [1, 3]], dtype=np.int32)
    out = CA.append_rows(cache, rows, np.array([70, 5]), bt, 64, "bf16", rope_theta=1e6)
    got0, got1 = out[0, 6], out[1, 5]
    assert np.array_equal(got0[:512], rows[0, :512]) and np.array_equal(got1[:512], rows[1, :512])
    for got, row, pos in [(got0, rows[0], 70), (got1, rows[1], 5)]:
        want = O.round_to_bf16(R.rope_rotate(O.bf16_to_f64(row[512:]), pos))
        assert np.array_equal(O.bf16_to_f64(got[512:]), want)
    plain = CA.append_rows(cache, rows, np.array([70, 5]), bt, 64, "bf16")
    assert np.array_equal(plain[0, 6], rows[0]) and np.array_equal(plain[1, 5], rows[1])
