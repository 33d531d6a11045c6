"""The attention entry point that allocates nothing (dq_attention_decode_static).

It is meant for callers that cannot call cudaMalloc: inference-server plugins
whose host process owns all device memory through its own pool, and embedded or
real-time deployments that fix their device memory at start-up.  Its scratch is
a static device array inside the library, shared by every call.  The checks
compare it with the fp64 oracle and with the entry point that takes a caller
workspace, on two calls in a row (the second call finds the first call's
partials and counters in the shared array).  This file is collected last on
purpose, so a stop-at-first-failure run has already run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

ATTN_TOL = 1e-4  # the attention tests' bar: max|out - ref| / max|ref|


def _inputs(seed, n_q, n_kv, max_ctx):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((n_q, 128)).astype(np.float32)
    k = rng.standard_normal((n_kv, max_ctx, 128)).astype(np.float16)
    v = rng.standard_normal((n_kv, max_ctx, 128)).astype(np.float16)
    return q, k, v


def _normwise(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.abs(a - b).max() / np.abs(b).max())


@pytest.fixture(scope="module")
def dq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantised_gemv_norm_gb300 import build, dq as dqmod

    build.build()
    dqmod.load()
    return dqmod


def _call_static(lib, q, k, v, out, n_q, n_kv, max_ctx, n_keys):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.dq_attention_decode_static(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                          ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                          n_q, n_kv, 128, max_ctx, n_keys, stream)


@pytest.mark.parametrize("n_q,n_kv,n_keys", [(32, 8, 513), (32, 8, 40), (64, 64, 1024), (64, 8, 1)])
def test_static_scratch_matches_oracle_and_workspace_version_twice(dq, orc, n_q, n_kv, n_keys):
    lib = dq.load()
    max_ctx = 1024
    qh, kh, vh = _inputs(n_keys, n_q, n_kv, max_ctx)
    ref = orc.attention(qh, kh.view(np.uint16), vh.view(np.uint16), n_keys)  # fp64 oracle
    q, k, v = (torch.from_numpy(a).cuda() for a in (qh, kh, vh))
    ws = dq.attention_decode(q, k, v, n_keys).cpu().numpy()  # the existing entry point, caller workspace
    assert _normwise(ws, ref) <= ATTN_TOL
    for _ in range(2):  # two calls in a row share the static array
        out = torch.full_like(q, float("nan"))
        assert _call_static(lib, q, k, v, out, n_q, n_kv, max_ctx, n_keys) == 0
        torch.cuda.synchronize()
        got = out.cpu().numpy()
        assert _normwise(got, ref) <= ATTN_TOL
        assert _normwise(got, ws) <= ATTN_TOL
    assert dq.device_error() == 0


def test_static_scratch_rejects_sizes_beyond_its_array(dq):
    lib = dq.load()
    qh, kh, vh = _inputs(1, 128, 16, 64)
    q, k, v = (torch.from_numpy(a).cuda() for a in (qh, kh, vh))
    assert _call_static(lib, q, k, v, q, 128, 16, 64, 8) == -2  # DQ_ERR_SHAPE: n_q > 64
    qh, kh, vh = _inputs(2, 128, 128, 64)
    q, k, v = (torch.from_numpy(a).cuda() for a in (qh, kh, vh))
    assert _call_static(lib, q, k, v, q, 128, 128, 64, 8) == -2  # DQ_ERR_SHAPE: n_kv > 64
