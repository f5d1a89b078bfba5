"""mla_decode_run_static: the decode pass for callers that cannot allocate.

Callers that run inside a CUDA graph capture, or inside a runtime that only
hands out the input and output buffers it owns, cannot allocate the
workspace mla_decode_run needs; this entry point keeps its scratch in the
library's own fixed-size device array instead.  These checks call it
through the C ABI and compare it with mla_decode_run (which takes a
caller-allocated workspace) on the same inputs, twice in a row so that the
second call runs over the scratch contents the first one left behind.

This file is collected last on purpose: a failure here leaves every other
test already run.
"""
import numpy as np
import pytest

import workloads as W
from mla_testlib import ensure_built, make_step

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _bits(x):
    return np.ascontiguousarray(x).view(np.uint32)


@pytest.mark.parametrize("name,sm_count", [("dense_small", None), ("long_small", 40),
                                           ("sparse_small", 7), ("mtp_small", 11),
                                           ("fp8_small", 5)])
def test_static_scratch_matches_workspace_entry_point(name, sm_count):
    """Same kernels, plan and split as mla_decode_run + mla_combine: o_lat and
    lse must agree bit for bit (NaN and infinity patterns included), on two
    calls in a row."""
    from head_latent_attention_paged_gb300 import mla_decode_run_static
    batch = W.generate(W.SMALL_WORKLOADS[name])
    step = make_step(batch, sm_count=sm_count)
    step.run()                                   # caller-allocated workspace
    torch.cuda.synchronize()
    ref_lat, ref_lse = step.o_lat.cpu().numpy(), step.lse.cpu().numpy()
    assert step.status() == 0
    status = torch.full((1,), 0xFFFF, dtype=torch.int32, device=step.device)
    for _ in range(2):                           # two calls in a row
        step.o_lat.fill_(float("nan"))
        step.lse.fill_(float("nan"))
        mla_decode_run_static(step.plan, step.q_hat, step.cache, step.block_table, step.seq_lens,
                              step.topk_idx, step.o_lat, step.lse, status, step.stream)
        torch.cuda.synchronize()
        assert np.array_equal(_bits(step.o_lat.cpu().numpy()), _bits(ref_lat))
        assert np.array_equal(_bits(step.lse.cpu().numpy()), _bits(ref_lse))
        assert int(status.item()) == 0


def test_static_scratch_matches_oracle():
    """The allocation-free call against the CPU oracle directly (o through the
    stand-alone W_UV projection of its o_lat)."""
    import oracle as O
    from head_latent_attention_paged_gb300 import mla_decode_run_static, mla_uv_proj
    from mla_testlib import compare, gpu_outputs
    batch = W.generate(W.SMALL_WORKLOADS["long_small"])
    step = make_step(batch, sm_count=9)
    for _ in range(2):
        step.o_lat.fill_(float("nan"))
        step.out.fill_(float("nan"))
        mla_decode_run_static(step.plan, step.q_hat, step.cache, step.block_table, step.seq_lens,
                              step.topk_idx, step.o_lat, step.lse, None, step.stream)
        mla_uv_proj(step.o_lat, step.w_uv, step.out, step.rows, step.H, step.stream)
        o, o_lat, lse = gpu_outputs(step)
        compare(O.decode(batch), o, o_lat, lse, label="static")


def test_rejected_static_call_queues_nothing():
    """A call rejected for a misaligned output returns its error; the next
    valid call still gives the workspace path's bits."""
    from head_latent_attention_paged_gb300 import (MLA_ERR_MISALIGNED, MlaError,
                                                   mla_decode_run_static)
    batch = W.generate(W.SMALL_WORKLOADS["dense_small"])
    step = make_step(batch, sm_count=13)
    step.run()
    torch.cuda.synchronize()
    ref_lat, ref_lse = step.o_lat.cpu().numpy(), step.lse.cpu().numpy()
    with pytest.raises(MlaError) as e:
        mla_decode_run_static(step.plan, step.q_hat, step.cache, step.block_table, step.seq_lens,
                              None, step.o_lat.data_ptr() + 4, step.lse, None, step.stream)
    assert e.value.code == MLA_ERR_MISALIGNED
    step.o_lat.fill_(float("nan"))
    mla_decode_run_static(step.plan, step.q_hat, step.cache, step.block_table, step.seq_lens,
                          None, step.o_lat, step.lse, None, step.stream)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(step.o_lat.cpu().numpy()), _bits(ref_lat))
    assert np.array_equal(_bits(step.lse.cpu().numpy()), _bits(ref_lse))


def test_static_scratch_rejects_plans_larger_than_the_array():
    from head_latent_attention_paged_gb300 import (MLA_ERR_WORKSPACE_TOO_SMALL, MlaError,
                                                   make_problem, mla_decode_plan,
                                                   mla_decode_run_static)
    # 256 row sets x 32 heads over 152 CTAs needs ~26 MiB of partials
    plan = mla_decode_plan(make_problem(256, 1, 32, 64, 1000, 10), None, 152)
    assert plan.workspace_bytes > 16 << 20
    A = 1 << 20   # never dereferenced: the size check fails first
    with pytest.raises(MlaError) as e:
        mla_decode_run_static(plan, A, A, A, A, None, A, A)
    assert e.value.code == MLA_ERR_WORKSPACE_TOO_SMALL
