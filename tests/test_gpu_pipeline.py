"""The host <-> device pipeline (runner.HostPipeline): packed input and
output copies on their own streams, double-buffered across steps.  Its
outputs must equal those of the same step run directly on the compute
stream with separately copied inputs."""
import numpy as np
import pytest

import workloads as W
from mla_testlib import ensure_built, gpu_outputs, make_step

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _built():
    ensure_built()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


@pytest.mark.parametrize("name", ["dense_small", "sparse_small", "fp8_small", "mtp_small"])
def test_pipeline_matches_direct_step(name):
    from head_latent_attention_paged_gb300 import mla_cache_append
    from head_latent_attention_paged_gb300.runner import HostPipeline
    batch = W.generate(W.SMALL_WORKLOADS[name])
    w = batch.workload
    rng = np.random.default_rng(21)
    rows = W.f32_to_bf16_bits(rng.standard_normal((w.batch, 576)).astype(np.float32))
    pos = (batch.seq_lens.astype(np.int64) - 1).clip(min=-1).astype(np.int32)
    # direct: append the rows, then one step
    ref = make_step(batch)
    mla_cache_append(ref.problem, torch.from_numpy(rows.view(np.int16)).to(ref.device),
                     torch.from_numpy(pos).to(ref.device), ref.block_table, ref.cache)
    ref.step()
    o_ref, _, lse_ref = gpu_outputs(ref)
    assert ref.status() == 0
    # pipelined: five steps with the same inputs (each appends the same rows)
    step = make_step(batch)
    q_bits = step.q_hat.view(torch.int16).cpu().numpy()
    pipe = HostPipeline(step, q_hat_bits=q_bits, block_table=batch.block_table,
                        seq_lens=batch.seq_lens, new_rows=rows, positions=pos,
                        topk_idx=batch.topk_idx)
    for k in range(5):
        step.out.fill_(float("nan"))   # the buffer set's previous outputs must be rewritten
        pipe.submit(k)
    pipe.drain(4)
    torch.cuda.synchronize()
    assert step.status() == 0
    for k in (3, 4):
        o_bits, lse = pipe.host_outputs(k)
        o = (o_bits.astype(np.uint32) << 16).view(np.float32).reshape(o_ref.shape)
        assert np.array_equal(o, o_ref), (name, k)
        assert np.array_equal(lse.reshape(lse_ref.shape), lse_ref), (name, k)
    assert pipe.h2d_bytes > 0 and pipe.d2h_bytes == o_ref.size * 2 + lse_ref.size * 4


def test_captured_pipeline_matches_direct_step():
    """The same pipelined sequence captured in one CUDA graph and replayed
    twice gives the direct step's outputs."""
    from head_latent_attention_paged_gb300 import mla_cache_append
    from head_latent_attention_paged_gb300.runner import HostPipeline
    batch = W.generate(W.SMALL_WORKLOADS["dense_small"])
    w = batch.workload
    rng = np.random.default_rng(22)
    rows = W.f32_to_bf16_bits(rng.standard_normal((w.batch, 576)).astype(np.float32))
    pos = (batch.seq_lens.astype(np.int64) - 1).clip(min=-1).astype(np.int32)
    ref = make_step(batch)
    mla_cache_append(ref.problem, torch.from_numpy(rows.view(np.int16)).to(ref.device),
                     torch.from_numpy(pos).to(ref.device), ref.block_table, ref.cache)
    ref.step()
    o_ref, _, lse_ref = gpu_outputs(ref)
    step = make_step(batch)
    pipe = HostPipeline(step, q_hat_bits=step.q_hat.view(torch.int16).cpu().numpy(),
                        block_table=batch.block_table, seq_lens=batch.seq_lens, new_rows=rows,
                        positions=pos)
    stream = torch.cuda.current_stream()
    for k in range(2):
        pipe.submit(k, stream)
    pipe.drain(1, stream)
    torch.cuda.synchronize()
    graph = pipe.capture(2, 6)
    for _ in range(2):
        pipe.host_out[0].zero_()
        pipe.host_out[1].zero_()
        graph.replay()
        torch.cuda.synchronize()
        for k in (6, 7):
            o_bits, lse = pipe.host_outputs(k)
            o = (o_bits.astype(np.uint32) << 16).view(np.float32).reshape(o_ref.shape)
            assert np.array_equal(o, o_ref) and np.array_equal(lse.reshape(lse_ref.shape), lse_ref)
    assert step.status() == 0
