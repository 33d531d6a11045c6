"""Failure paths of the decode step, exercised without faulting the GPU.

* A fused token whose grid-barrier waits cannot complete: a diagnostics call
  shortens the wait bound to 1 ms and raises every barrier target of the next
  token beyond what the blocks can reach.  Every block's wait runs out, the
  kernel records the timeout, stops working and ends; the status query maps the
  record to DQ_ERR_TIMEOUT; the same model then decodes correctly again (the
  kernel zeroes its barrier counters on the way out).
* An allocation failure injected on the host: dq_model_create returns
  DQ_ERR_ALLOC and no handle, then succeeds once the injection is used up.
* A fused token captured into a CUDA graph and replayed: its launch arguments
  depend only on the call, so replays with new inputs match the oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

from quantised_gemv_norm_gb300 import synth

pytestmark = pytest.mark.gpu

GEMV_TOL = 2e-3
DQ_ERR_UNSUPPORTED, DQ_ERR_TIMEOUT, DQ_ERR_ALLOC = -4, -6, -7


@pytest.fixture(scope="module")
def dq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantised_gemv_norm_gb300 import build, dq as dqmod

    build.build()
    dqmod.load()
    yield dqmod
    assert dqmod.device_error() == 0


def cuda(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def normwise(y, r):
    y = np.asarray(y, np.float64)
    r = np.asarray(r, np.float64)
    return float(np.max(np.abs(y - r)) / np.max(np.abs(r)))


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _small_model(seed, max_ctx=32):
    return synth.make_model(seed, n_layers=2, hidden=2048, ffn=4096, n_q_heads=16, n_kv_heads=4, head_dim=128,
                            vocab=400, max_ctx=max_ctx, qwen3_attention=True)


@pytest.mark.parametrize("pos", [0, 5])  # the attention folded into the O phase, and its own phase
def test_fused_barrier_timeout_reports_and_model_recovers(dq, orc, pos):
    from quantised_gemv_norm_gb300 import upload

    m = _small_model(31)
    kv = synth.make_kv_cache(31, m, pos)
    w = upload.to_device(m, kv)
    model = dq.Model(**upload.model_kwargs(m), weights=w, flags=dq.MODEL_FUSED)
    assert model.fused
    lib = dq.load()
    x = synth.decode_input(31, m.hidden)
    ref = orc.decode_step(m, x, pos, kv.copy())
    assert lib.dq_check_device(_stream()) == 0
    assert lib.dq_model_debug_waits(model._h, 1_000_000, 1000) == 0  # 1 ms bound, unreachable barriers
    model.step(cuda(x), pos)
    assert lib.dq_check_device(_stream()) == DQ_ERR_TIMEOUT
    assert lib.dq_check_device(_stream()) == 0  # the check cleared the record
    for _ in range(2):  # the same model, still with the 1 ms bound, decodes correctly again
        logits = model.step(cuda(x), pos).cpu().numpy()
        assert lib.dq_check_device(_stream()) == 0
        assert normwise(logits, ref) <= GEMV_TOL
    model.close()


def test_debug_waits_argument_errors(dq):
    from quantised_gemv_norm_gb300 import upload

    m = _small_model(32)
    w = upload.to_device(m, synth.make_kv_cache(32, m, 0))
    lib = dq.load()
    graph_model = dq.Model(**upload.model_kwargs(m), weights=w, flags=0)
    assert lib.dq_model_debug_waits(graph_model._h, 1_000_000, 0) == DQ_ERR_UNSUPPORTED
    graph_model.close()
    fused = dq.Model(**upload.model_kwargs(m), weights=w, flags=dq.MODEL_FUSED)
    assert lib.dq_model_debug_waits(fused._h, 10, 0) == -2  # below 1 us
    assert lib.dq_model_debug_waits(fused._h, 1_000_000, -1) == -2
    assert lib.dq_model_debug_waits(None, 1_000_000, 0) == -1
    fused.close()


@pytest.mark.parametrize("flags", [0, 2])
def test_model_create_reports_allocation_failure(dq, flags):
    from quantised_gemv_norm_gb300 import upload

    m = _small_model(33)
    w = upload.to_device(m, synth.make_kv_cache(33, m, 0))
    lib = dq.load()
    assert lib.dq_debug_fail_next_allocs(1) == 0
    with pytest.raises(dq.DQError) as e:
        dq.Model(**upload.model_kwargs(m), weights=w, flags=flags)
    assert e.value.status == DQ_ERR_ALLOC
    model = dq.Model(**upload.model_kwargs(m), weights=w, flags=flags)  # the injection is used up
    logits = model.step(cuda(synth.decode_input(33, m.hidden)), 0)
    assert bool(torch.isfinite(logits).all())
    model.close()
    assert lib.dq_debug_fail_next_allocs(-1) == -2


def test_fused_decode_step_replays_from_a_cuda_graph(dq, orc):
    from quantised_gemv_norm_gb300 import upload

    m = _small_model(34)
    pos = 6
    kv = synth.make_kv_cache(34, m, pos)
    w = upload.to_device(m, kv)
    model = dq.Model(**upload.model_kwargs(m), weights=w, flags=dq.MODEL_FUSED)
    assert model.fused
    x_dev = torch.empty(m.hidden, dtype=torch.float32, device="cuda")
    logits = torch.empty(m.vocab, dtype=torch.float32, device="cuda")
    x_dev.copy_(cuda(synth.decode_input(34, m.hidden, 0)))
    model.step(x_dev, pos, logits)  # one eager token first
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        model.step(x_dev, pos, logits)
    kv_host = kv.copy()
    for t in range(1, 4):  # each replay is a new token at the same position (it rewrites cache row pos)
        x = synth.decode_input(34, m.hidden, t)
        x_dev.copy_(cuda(x))
        graph.replay()
        torch.cuda.synchronize()
        ref = orc.decode_step(m, x, pos, kv_host)
        assert normwise(logits.cpu().numpy(), ref) <= GEMV_TOL, t
    assert dq.device_error() == 0
    model.close()
