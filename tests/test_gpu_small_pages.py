"""GPU parity with pages smaller than a 64-token tile: 16 and 32 tokens, the
compressed-layer page block size (block_size / compress_ratio, e.g. 32 at
block_size 64 for a ratio-2 layer: GLM-4.7-Flash record, phantomic12
inference-research, the engine-kernel constraint on page-block sizes).  A
tile then spans 64 / P pages of the block table, each staged separately."""
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


def _run(batch, sm_count=None, label=""):
    q_hat = oracle_q_hat(batch)
    step = make_step(batch, sm_count=sm_count, absorb=False)
    upload_q_hat(step, q_hat)
    step.step()
    o, o_lat, lse = gpu_outputs(step)
    assert step.status() == 0, label
    compare(O.decode(batch), o, o_lat, lse, label=label, lse_ref=O.decode(batch, q_hat=q_hat))


@pytest.mark.parametrize("page_size", [16, 32])
@pytest.mark.parametrize("name,garbage,sm_count", [
    ("dense_small", "finite", None), ("dense_small", "nan", 7),
    ("fp8_small", "finite", None), ("fp8_small", "nan", 7),
    ("sparse_small", "finite", None),
])
def test_small_pages_match_oracle(page_size, name, garbage, sm_count):
    w = W.with_overrides(W.SMALL_WORKLOADS[name], page_size=page_size)
    _run(W.generate(w, garbage=garbage), sm_count=sm_count, label=f"{name}/p{page_size}/{garbage}")


@pytest.mark.parametrize("page_size", [16, 32])
def test_small_pages_edge_lengths(page_size):
    """Lengths ending inside the first, second and last page of a tile."""
    w = W.with_overrides(W.SMALL_WORKLOADS["dense_small"], page_size=page_size,
                         seq_lens=(1, 15, 16, 17, 31, 33, 47, 63, 64, 65, 100), batch=11)
    _run(W.generate(w), label=f"edges/p{page_size}")
