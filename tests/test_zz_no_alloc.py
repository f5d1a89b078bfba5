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
from mla_testlib import ATOL_MAX, LSE_TOL, REL_L2, ensure_built, make_step

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _close(a_lat, a_lse, b_lat, b_lse):
    live = np.isfinite(a_lse)
    assert np.array_equal(live, np.isfinite(b_lse))
    assert np.abs(b_lat - a_lat).max() <= ATOL_MAX
    assert np.linalg.norm(b_lat - a_lat) <= REL_L2 * max(np.linalg.norm(a_lat), 1e-30)
    assert np.abs(b_lse[live] - a_lse[live]).max(initial=0.0) <= LSE_TOL


@pytest.mark.parametrize("name,sm_count", [("dense_small", None), ("long_small", 40),
                                           ("sparse_small", 7), ("mtp_small", 11)])
def test_static_scratch_matches_workspace_entry_point(name, sm_count):
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
        _close(ref_lat, ref_lse, step.o_lat.cpu().numpy(), step.lse.cpu().numpy())
        assert int(status.item()) == 0


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
