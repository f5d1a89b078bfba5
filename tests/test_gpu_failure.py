"""Failure detection without a fault: the bounded waits every kernel uses
give up after their limit and report MLA_STATUS_TIMEOUT through a status
word the host reads, and the CUDA context stays usable afterwards."""
import numpy as np
import pytest

import workloads as W
from mla_testlib import compare, ensure_built, gpu_outputs, make_step
import oracle as O

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.mark.parametrize("limit_ns", [1_000, 2_000_000, 50_000_000])
def test_wait_that_nothing_completes_times_out(limit_ns):
    from head_latent_attention_paged_gb300 import MLA_STATUS_TIMEOUT, mla_selftest_bounded_wait
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    mla_selftest_bounded_wait(status, limit_ns, waited)
    torch.cuda.synchronize()
    assert int(status.item()) & MLA_STATUS_TIMEOUT
    w = int(waited.item())
    assert limit_ns <= w <= limit_ns + 20_000_000, w


def test_context_usable_after_a_timeout():
    """A decode after the timed-out wait runs and matches the oracle; its own
    status word is clean (the timeout was reported where it happened)."""
    from head_latent_attention_paged_gb300 import mla_selftest_bounded_wait
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    mla_selftest_bounded_wait(status, 5_000_000)
    batch = W.generate(W.SMALL_WORKLOADS["dense_small"])
    step = make_step(batch)
    step.step()
    o, o_lat, lse = gpu_outputs(step)
    assert int(status.item()) != 0 and step.status() == 0
    compare(O.decode(batch), o, o_lat, lse, label="after-timeout")
