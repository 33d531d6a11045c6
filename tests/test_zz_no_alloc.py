"""The attention entry point that allocates nothing (dq_attention_decode_static).

It is meant for callers that cannot call cudaMalloc: code running while a stream
is captured under a mode that forbids allocation, server plugins whose host owns
all device memory, or deployments that fix device memory at start-up.  Its
scratch is a static device array inside the library.  This file is collected
last on purpose, so a stop-at-first-failure run has already run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _inputs(seed, n_q, n_kv, max_ctx):
    rng = np.random.default_rng(seed)
    q = torch.from_numpy(rng.standard_normal((n_q, 128)).astype(np.float32)).cuda()
    k = torch.from_numpy(rng.standard_normal((n_kv, max_ctx, 128)).astype(np.float16)).cuda()
    v = torch.from_numpy(rng.standard_normal((n_kv, max_ctx, 128)).astype(np.float16)).cuda()
    return q, k, v


def _normwise(a, b):
    a = a.double().cpu()
    b = b.double().cpu()
    return float((a - b).abs().max() / b.abs().max())


@pytest.fixture(scope="module")
def dq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantised_gemv_norm_gb300 import build, dq as dqmod

    build.build()
    dqmod.load()
    return dqmod


@pytest.mark.parametrize("n_q,n_kv,n_keys", [(32, 8, 513), (32, 8, 40), (64, 64, 1024)])
def test_static_scratch_matches_workspace_version_twice(dq, n_q, n_kv, n_keys):
    lib = dq.load()
    q, k, v = _inputs(n_keys, n_q, n_kv, 1024)
    ref = dq.attention_decode(q, k, v, n_keys)  # the existing entry point, caller workspace
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):  # two calls in a row share the static array
        out = torch.full_like(q, float("nan"))
        st = lib.dq_attention_decode_static(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                            ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                            n_q, n_kv, 128, 1024, n_keys, stream)
        assert st == 0
        torch.cuda.synchronize()
        assert _normwise(out, ref) <= 1e-4
    assert dq.device_error() == 0


def test_static_scratch_rejects_sizes_beyond_its_array(dq):
    lib = dq.load()
    q, k, v = _inputs(1, 128, 16, 64)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.dq_attention_decode_static(ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                                        ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(q.data_ptr()),
                                        128, 16, 128, 64, 8, stream)
    assert st == -2  # DQ_ERR_SHAPE: n_q > 64
