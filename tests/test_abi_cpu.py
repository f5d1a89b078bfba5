"""The C ABI on the CPU: the library loads without a GPU, exports every entry
point the header declares, and rejects bad arguments with error codes before
any CUDA call."""
import ctypes
import os
import re

import numpy as np
import pytest

import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def m():
    from head_latent_attention_paged_gb300 import _build
    _build.build()
    import head_latent_attention_paged_gb300 as mod
    mod.load()
    return mod


def _declared_entry_points():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"MLA_API\s+[\w\s\*]+?\b(mla_\w+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol(m):
    declared = _declared_entry_points()
    assert {"mla_decode_plan", "mla_decode_run", "mla_combine", "mla_uv_proj"} <= declared
    lib = ctypes.CDLL(m.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert declared == set(m.EXPORTED)


def test_every_entry_point_has_declared_argument_types(m):
    """ctypes passes undeclared integer arguments as 32-bit ints, which would
    cut device pointers: every exported call must declare its argument
    types."""
    lib = m.load()
    for name in m.EXPORTED:
        assert getattr(lib, name).argtypes is not None, name


def test_version_and_strerror(m):
    assert m.version() == 20100
    for code in (0, -1, -2, -3, -4, -5, -99):
        assert isinstance(m.strerror(code), str) and m.strerror(code)


def _problem(m, **kw):
    base = dict(batch=4, q_len=1, num_heads=20, page_size=64, num_pages=100, max_pages_per_seq=30)
    base.update(kw)
    return m.make_problem(**base)


def test_plan_ok_and_workspace_layout(m):
    seq = np.array([100, 1000, 64, 0], dtype=np.int32)
    plan = m.mla_decode_plan(_problem(m), seq, 152)
    tiles = sum((int(t) + 63) // 64 for t in seq)
    assert plan.planned_tiles == tiles
    assert plan.num_ctas == min(152, tiles)
    assert plan.num_slots == 4 + plan.num_ctas - 1
    assert plan.ws_partial_o == 0
    assert plan.ws_partial_lse >= plan.num_slots * 20 * 512 * 4
    assert plan.ws_prefix >= plan.ws_partial_lse + plan.num_slots * 20 * 4
    assert plan.ws_status >= plan.ws_prefix + 2 * 4 * (4 + 1)
    assert plan.workspace_bytes > plan.ws_status
    assert plan.smem_bytes <= 232448
    # no host seq_lens: fill every SM
    assert m.mla_decode_plan(_problem(m), None, 152).num_ctas == 152


@pytest.mark.parametrize("kw", [dict(batch=257), dict(batch=65, q_len=4, num_heads=32),
                                dict(batch=200, q_len=4, kv_dtype=1), dict(batch=129, q_len=4),
                                dict(batch=4096), dict(batch=1000, kv_dtype=2)])
def test_plans_beyond_256_row_sets(m, kw):
    """More row sets than the decode kernel keeps prefixes for in shared
    memory: the plan leaves them out of its shared memory and sizes the
    workspace's prefix area, int32 [2][S + 1], for the pre-pass."""
    plan = m.mla_decode_plan(_problem(m, **kw), None, 152)
    assert plan.num_streams > 256
    assert plan.smem_bytes <= 232448
    assert plan.ws_status >= plan.ws_prefix + 8 * (plan.num_streams + 1)
    small = m.mla_decode_plan(_problem(m, **dict(kw, batch=2)), None, 152)
    assert plan.smem_bytes <= small.smem_bytes


@pytest.mark.parametrize("kw,S,prefix_pass", [
    (dict(batch=64), 64, 0), (dict(batch=256), 256, 0), (dict(batch=257), 257, 1),
    (dict(batch=150, q_len=2, kv_dtype=1), 150, 0),    # FP8 drafts: room for 150 rows' prefixes
    (dict(batch=160, q_len=2, kv_dtype=1), 160, 1),    # ... not for 160 beside its buffers
    (dict(batch=80, q_len=4, topk_width=2048), 320, 1),
])
def test_plan_reports_its_prefix_pass(m, kw, S, prefix_pass):
    """The decode kernel keeps the work split's per-row-set prefixes in
    shared memory when they fit (at most 256 row sets); otherwise each launch
    runs the one-block prefix pre-pass first, which the plan reports."""
    plan = m.mla_decode_plan(_problem(m, **kw), None, 152)
    assert plan.num_streams == S and plan.prefix_pass == prefix_pass
    assert plan.smem_bytes <= 232448

@pytest.mark.parametrize("kw,code", [
    (dict(page_size=96), -2), (dict(page_size=8), -2), (dict(page_size=256), -2), (dict(num_heads=0), -1),
    (dict(num_heads=33), -2), (dict(q_len=0), -1), (dict(batch=-1), -1),
    (dict(topk_width=100), -2), (dict(topk_width=-128), -1), (dict(kv_lora_rank=256), -2),
    (dict(rope_dim=32), -2), (dict(v_head_dim=128), -2), (dict(nope_dim=128), -2),
    (dict(causal=2), -1), (dict(sm_scale=0.0), -1), (dict(sm_scale=float("nan")), -1),
    (dict(num_pages=0), -1), (dict(max_pages_per_seq=0), -1), (dict(batch=2**20 + 1), -2),
    (dict(kv_dtype=1, topk_width=128), -2), (dict(kv_dtype=2, topk_width=128), -2),
    (dict(kv_dtype=3), -2), (dict(kv_dtype=-1), -2),
])
def test_plan_rejects(m, kw, code):
    with pytest.raises(m.MlaError) as e:
        m.mla_decode_plan(_problem(m, **kw), None, 152)
    assert e.value.code == code


def test_fp8_plan_fits_shared_memory(m):
    """FP8 caches plan like bf16 ones; the FP8 kernel's staging (two bf16
    tiles, each with its P in the RoPE chunk, two FP8 byte tiles and the
    RoPE part of q_hat for 32 M-rows) fits the 227 KB window at the largest
    head and row-set counts."""
    seq = np.array([100, 1000, 64, 0], dtype=np.int32)
    plan = m.mla_decode_plan(_problem(m, kv_dtype=m.MLA_KV_FP8_E4M3_E8M0), seq, 152)
    assert plan.planned_tiles == sum((int(t) + 63) // 64 for t in seq)
    big = m.mla_decode_plan(_problem(m, kv_dtype=m.MLA_KV_FP8_E4M3_E8M0, batch=256, num_heads=32),
                            None, 152)
    assert 2 * 73728 + 2 * 64 * 594 + 32 * 128 < big.smem_bytes <= 232448


def test_fp4_plan_fits_shared_memory(m):
    """FP4 caches (324-byte rows) plan like FP8 ones: the raw rows land in
    the bf16 stages, so the staging is the bf16 kernel's (three bf16 tiles
    and the RoPE part of q_hat, 64 rows x 128 B)."""
    seq = np.array([100, 1000, 64, 0], dtype=np.int32)
    plan = m.mla_decode_plan(_problem(m, kv_dtype=m.MLA_KV_FP4_E2M1_E8M0), seq, 152)
    assert plan.planned_tiles == sum((int(t) + 63) // 64 for t in seq)
    big = m.mla_decode_plan(_problem(m, kv_dtype=m.MLA_KV_FP4_E2M1_E8M0, batch=256, num_heads=32),
                            None, 152)
    assert 3 * 73728 < big.smem_bytes <= 232448
    assert big.smem_bytes == m.mla_decode_plan(
        _problem(m, batch=256, num_heads=32), None, 152).smem_bytes


@pytest.mark.parametrize("q_len,heads,group", [(1, 20, 1), (2, 20, 2), (3, 20, 2), (4, 12, 4),
                                               (2, 24, 2), (2, 32, 1), (6, 8, 6), (7, 8, 6)])
def test_multi_token_plan_groups_draft_tokens(m, q_len, heads, group):
    """Dense bf16 problems with q_len >= 2 group G = min(q_len, 48 / H)
    draft tokens of a request into one row set (G >= 2, else one per token);
    the partial slots hold G * H rows; every plan fits shared memory."""
    seq = np.array([100, 1000, 64, 0], dtype=np.int32)
    plan = m.mla_decode_plan(_problem(m, q_len=q_len, num_heads=heads), seq, 152)
    assert plan.num_streams == 4 * -(-q_len // group)
    rows = group * heads
    assert plan.ws_partial_lse >= plan.num_slots * rows * 512 * 4
    assert plan.ws_prefix >= plan.ws_partial_lse + plan.num_slots * rows * 4
    assert plan.smem_bytes <= 232448
    # FP4 and FP8 caches group drafts the same way
    for kv in (m.MLA_KV_FP4_E2M1_E8M0, m.MLA_KV_FP8_E4M3_E8M0):
        quant = m.mla_decode_plan(_problem(m, q_len=q_len, num_heads=heads, kv_dtype=kv), seq, 152)
        assert quant.num_streams == plan.num_streams and quant.smem_bytes <= 232448


def test_plan_rejects_negative_seq_len_and_bad_sm_count(m):
    with pytest.raises(m.MlaError) as e:
        m.mla_decode_plan(_problem(m), np.array([1, -2, 3, 4], dtype=np.int32), 152)
    assert e.value.code == -1
    with pytest.raises(m.MlaError) as e:
        m.mla_decode_plan(_problem(m), None, 0)
    assert e.value.code == -1


def test_calls_reject_null_and_misaligned_pointers_before_cuda(m):
    plan = m.mla_decode_plan(_problem(m), None, 152)
    A = 1 << 20    # an aligned fake address: never dereferenced, the call fails first
    run = m.mla_decode_run

    def code_of(fn, *args, **kw):
        with pytest.raises(m.MlaError) as e:
            fn(*args, **kw)
        return e.value.code

    # (plan, q, w_uk, kv, block_table, seq_lens, topk, workspace, o_lat, lse)
    assert code_of(run, plan, None, None, A, A, A, None, A, A, A) == -1
    assert code_of(run, plan, A, None, A, A, A, A, A, A, A) == -1        # dense given a top-k list
    assert code_of(run, plan, A + 8, None, A, A, A, None, A, A, A) == -3
    assert code_of(run, plan, A, A + 8, A, A, A, None, A, A, A) == -3    # W_UK misaligned
    assert code_of(run, plan, A, None, A, A, A, None, A, None, A) == -1  # outputs are required
    assert code_of(run, plan, A, None, A, A, A, None, A, A + 8, A) == -3
    # a workspace smaller than the plan's
    assert code_of(run, plan, A, None, A, A, A, None, A, A, A,
                   workspace_bytes=plan.workspace_bytes - 1) == -4
    assert code_of(m.mla_combine, plan, A, A, A + 4, A) == -3
    assert code_of(m.mla_combine, plan, A, A, A, A, workspace_bytes=16) == -4
    assert code_of(m.mla_combine, plan, A, A, A, A, w_uv=A, out=None) == -1   # W_UV needs out
    assert code_of(m.mla_combine, plan, A, A, A, A, w_uv=A + 2, out=A) == -3
    assert code_of(m.mla_uv_proj, A, A, A, -1, 20) == -1
    assert code_of(m.mla_uv_proj, A, A + 2, A, 4, 20) == -3
    assert code_of(m.mla_q_absorb, plan, A, None, A) == -1
    assert code_of(m.mla_q_absorb, plan, A, A, A + 2) == -3
    sparse = m.mla_decode_plan(_problem(m, topk_width=256), None, 152)
    assert code_of(run, sparse, A, None, A, A, A, None, A, A, A) == -1   # sparse without a list


def test_plan_split_tokens(m):
    """split_tokens > 0 sizes the grid by length (about split_tokens tokens
    per CTA; needs the host lengths; a multiple of 64), 0 is one CTA per SM;
    the workspace out-parameter matches the plan."""
    seq = np.array([100_000, 70_000, 1000, 0], dtype=np.int32)
    tiles = sum((int(t) + 63) // 64 for t in seq)
    for st in (256, 512, 1024):
        plan = m.mla_decode_plan(_problem(m, max_pages_per_seq=2000), seq, 152, split_tokens=st)
        assert plan.num_ctas == -(-tiles // (st // 64)) and plan.split_tokens == st
        assert plan.num_slots == plan.num_streams + plan.num_ctas - 1
    auto = m.mla_decode_plan(_problem(m, max_pages_per_seq=2000), seq, 152)
    assert auto.num_ctas == 152 and auto.split_tokens == 0
    for bad in (-64, 100):
        with pytest.raises(m.MlaError) as e:
            m.mla_decode_plan(_problem(m, max_pages_per_seq=2000), seq, 152, split_tokens=bad)
        assert e.value.code == -1
    with pytest.raises(m.MlaError) as e:   # a length split needs the host lengths
        m.mla_decode_plan(_problem(m), None, 152, split_tokens=512)
    assert e.value.code == -1


TILE_COST, STREAM_COST = 4, 7   # the kernels' cost weights (tile, stream start)


def _first_tile_at(tiles_pre, cost_pre, u):
    """Host restatement of the kernel's search: first tile whose cost
    position (stream cost start + STREAM_COST + k * TILE_COST) is >= u."""
    S = len(tiles_pre) - 1
    if u >= cost_pre[S]:
        return int(tiles_pre[S])
    s = int(np.searchsorted(cost_pre, u, side="right") - 1)
    off = u - cost_pre[s]
    k = 0 if off <= STREAM_COST else -(-(off - STREAM_COST) // TILE_COST)
    nt = tiles_pre[s + 1] - tiles_pre[s]
    return int(tiles_pre[s] + k) if k < nt else int(tiles_pre[s + 1])


@pytest.mark.parametrize("page_size", [16, 32, 64, 128])
def test_plan_accepts_every_supported_page_size(m, page_size):
    """Pages of 16 and 32 tokens (compressed layers: block_size / compress
    ratio) as well as 64 and 128."""
    seq = np.array([100, 1000, 64, 0], dtype=np.int32)
    plan = m.mla_decode_plan(_problem(m, page_size=page_size, num_pages=4000,
                                      max_pages_per_seq=1024 // page_size + 1), seq, 152)
    assert plan.planned_tiles == sum((int(t) + 63) // 64 for t in seq)


def test_cache_append_rejects_bad_arguments_before_cuda(m):
    A = 1 << 20    # an aligned fake address: never dereferenced, the call fails first
    prob = _problem(m)
    with pytest.raises(m.MlaError) as e:
        m.mla_cache_append(prob, None, A, A, A)
    assert e.value.code == -1
    with pytest.raises(m.MlaError) as e:
        m.mla_cache_append(prob, A + 8, A, A, A)
    assert e.value.code == -3
    with pytest.raises(m.MlaError) as e:
        m.mla_cache_append(_problem(m, page_size=96), A, A, A, A)
    assert e.value.code == -2
    for theta in (-1.0, 0.5, float("nan"), float("inf")):
        with pytest.raises(m.MlaError) as e:
            m.mla_cache_append(prob, A, A, A, A, rope_theta=theta)
        assert e.value.code == -1


def test_stream_split_matches_kernel_rule():
    """Host restatement of the cost-weighted split the kernels use: tile k of
    stream s sits at cost position P_s + 7 + 4k (P_s: cost of the streams
    before it, a stream with n > 0 tiles costing 7 + 4n); CTA c owns the
    tiles at positions [c*U/C, (c+1)*U/C).  The tile ranges the decode
    derives by search partition the tiles in order, the owner formula the
    merge uses agrees with them, partial slot s + c is unique, and a CTA
    that opens more streams gets fewer tiles."""
    rng = np.random.default_rng(0)
    for _ in range(200):
        S = int(rng.integers(1, 40))
        tiles = rng.integers(0, 30, size=S)
        tiles[rng.random(S) < 0.2] = 0
        T = int(tiles.sum())
        if T == 0:
            continue
        C = int(rng.integers(1, min(T, 200) + 1))
        cost = np.where(tiles > 0, STREAM_COST + TILE_COST * tiles, 0)
        tpre = np.concatenate([[0], np.cumsum(tiles)])
        cpre = np.concatenate([[0], np.cumsum(cost)])
        U = int(cpre[-1])
        bounds = [_first_tile_at(tpre, cpre, (c * U) // C) for c in range(C + 1)]
        assert bounds[0] == 0 and bounds[-1] == T and all(np.diff(bounds) >= 0)
        owner = np.empty(T, dtype=np.int64)
        for c in range(C):
            owner[bounds[c]:bounds[c + 1]] = c
        slots = set()
        for s in range(S):
            for k in range(int(tiles[s])):
                x = int(cpre[s]) + STREAM_COST + TILE_COST * k
                c = ((x + 1) * C - 1) // U
                assert c == owner[tpre[s] + k]
                slots.add((s, c))
        keys = [s + c for s, c in slots]
        assert len(keys) == len(set(keys)) and max(keys) < S + C - 1 + 1


def test_bounded_wait_selftest_rejects_bad_arguments_before_cuda(m):
    A = 1 << 20
    for status, limit, waited, code in [(None, 1000, None, -1), (A, 0, None, -1),
                                        (A, 2_000_000_000, None, -1), (A + 2, 1000, None, -3),
                                        (A, 1000, A + 4, -3)]:
        with pytest.raises(m.MlaError) as e:
            m.mla_selftest_bounded_wait(status, limit, waited)
        assert e.value.code == code


def test_row_set_count_counts_grouped_drafts(m):
    """Row sets, not query tokens: 64 requests with 8 drafts of 6 heads are
    64 grouped row sets (G = 8), over every cache type."""
    plan = m.mla_decode_plan(_problem(m, batch=64, q_len=8, num_heads=6), None, 152)
    assert plan.num_streams == 64
    for kv in (m.MLA_KV_FP4_E2M1_E8M0, m.MLA_KV_FP8_E4M3_E8M0):
        assert m.mla_decode_plan(_problem(m, batch=64, q_len=8, num_heads=6, kv_dtype=kv), None,
                                 152).num_streams == 64
    plan = m.mla_decode_plan(_problem(m, batch=128, q_len=4), None, 152)   # G = 2
    assert plan.num_streams == 256


def _stream_geom(s, q_len, group):
    """Host restatement of the row-set geometry the kernels use."""
    ng = -(-q_len // group)
    b, gi = divmod(s, ng)
    j0 = gi * group
    return b, j0, min(group, q_len - j0)


@pytest.mark.parametrize("batch,q_len,heads", [(3, 1, 20), (3, 2, 20), (2, 3, 20), (2, 5, 8),
                                               (4, 7, 8), (2, 4, 12), (3, 2, 32)])
def test_row_sets_partition_the_query_rows(m, batch, q_len, heads):
    """Every (request, draft, head) output row belongs to exactly one row
    set, as the contiguous block (b * Q + j0) * H .. + nq * H; the plan's row
    set count matches the grouping rule."""
    plan = m.mla_decode_plan(_problem(m, batch=batch, q_len=q_len, num_heads=heads), None, 152)
    S = plan.num_streams
    g_rule = min(q_len, 48 // heads)
    group = g_rule if g_rule >= 2 else 1
    assert S == batch * -(-q_len // group)
    seen = np.zeros(batch * q_len * heads, dtype=np.int64)
    for s in range(S):
        b, j0, nq = _stream_geom(s, q_len, group)
        assert 0 <= b < batch and nq >= 1
        first = (b * q_len + j0) * heads
        seen[first:first + nq * heads] += 1
        assert nq * heads <= 48 or group == 1
    assert (seen == 1).all()


def test_plain_c_consumer_builds_and_plans(tmp_path):
    """The header is valid C99 on its own, and a C program linked against the
    library can plan a decode and read error strings (no GPU needed)."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    from head_latent_attention_paged_gb300 import LIB_PATH
    libdir = os.path.dirname(LIB_PATH)
    src = os.path.join(ROOT, "tests", "c_consumer", "plan_check.c")
    exe = str(tmp_path / "plan_check")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    src, "-o", exe, "-L", libdir, "-lmla_gb300", f"-Wl,-rpath,{libdir}"],
                   check=True, capture_output=True)
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    assert "plan_check ok" in out.stdout
