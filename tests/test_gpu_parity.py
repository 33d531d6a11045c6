"""GPU parity: every C-ABI entry point against the CPU oracle on the same seeded
inputs, at sizes that span several tiles with ragged tails and at the full
configuration sizes.  Tolerances:
  norms      |y - r| <= 1e-5 * max(1, |r|) elementwise
  GEMV       max|y - r| / max|r| <= 2e-3 (bf16 in / fp32 accumulate bar)
  dequant    bit-exact
  attention  max|o - r| / max|r| <= 1e-4 (fp16 data, fp32 arithmetic)
  decode     logits max|y - r| / max|r| <= 2e-3
"""
import ctypes
import os

import numpy as np
import pytest
import torch

from quantised_gemv_norm_gb300 import synth

pytestmark = pytest.mark.gpu

GEMV_TOL = 2e-3


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
    return float(np.max(np.abs(y - r)) / max(np.max(np.abs(r)), 1e-300))


# ---------------------------------------------------------------- norms


@pytest.mark.parametrize("rows,n", [(64, 2048), (3, 1000), (5, 4097), (2, 1), (1, 12288)])
def test_rmsnorm(dq, orc, rows, n):
    x, g, _ = synth.norm_inputs(0, rows, n)
    y = dq.rmsnorm(cuda(x), cuda(g), 1e-6).cpu().numpy()
    r = orc.rmsnorm(x, g, 1e-6)
    assert np.all(np.abs(y - r) <= 1e-5 * np.maximum(1.0, np.abs(r)))


@pytest.mark.parametrize("rows,n", [(64, 2048), (3, 1000), (5, 4097), (1, 12288)])
def test_layernorm(dq, orc, rows, n):
    x, g, b = synth.norm_inputs(1, rows, n)
    y = dq.layernorm(cuda(x), cuda(g), cuda(b), 1e-6).cpu().numpy()
    r = orc.layernorm(x, g, b, 1e-6)
    assert np.all(np.abs(y - r) <= 1e-5 * np.maximum(1.0, np.abs(r)))


@pytest.mark.parametrize("threads", [1, 2, 8, 32, 64, 256, 1024])
def test_norm_thread_sweep(dq, orc, threads):
    x, g, b = synth.norm_inputs(2, 4, 2048)
    y = dq.rmsnorm(cuda(x), cuda(g), 1e-6, threads=threads).cpu().numpy()
    r = orc.rmsnorm(x, g, 1e-6)
    assert np.all(np.abs(y - r) <= 1e-5 * np.maximum(1.0, np.abs(r)))
    y = dq.layernorm(cuda(x), cuda(g), cuda(b), 1e-6, threads=threads).cpu().numpy()
    r = orc.layernorm(x, g, b, 1e-6)
    assert np.all(np.abs(y - r) <= 1e-5 * np.maximum(1.0, np.abs(r)))


def test_rmsnorm_in_place(dq, orc):
    x, g, _ = synth.norm_inputs(3, 8, 2048)
    t = cuda(x)
    dq.rmsnorm(t, cuda(g), 1e-6, out=t)
    r = orc.rmsnorm(x, g, 1e-6)
    assert np.all(np.abs(t.cpu().numpy() - r) <= 1e-5 * np.maximum(1.0, np.abs(r)))


# ------------------------------------------------------------ dequant


def test_dequant_bit_exact(dq, orc):
    rng = np.random.default_rng(11)
    b4 = synth.q4k_blocks(rng, 3001)
    b6 = synth.q6k_blocks(rng, 3001)
    y4 = dq.dequant_q4k(cuda(b4)).cpu().numpy()
    y6 = dq.dequant_q6k(cuda(b6)).cpu().numpy()
    r4 = orc.dequant_q4k(b4).astype(np.float32)
    r6 = orc.dequant_q6k(b6).astype(np.float32)
    assert np.array_equal(y4.view(np.uint32), r4.view(np.uint32))
    assert np.array_equal(y6.view(np.uint32), r6.view(np.uint32))


def test_dequant_q2k_bit_exact_and_hand_built(dq, orc):
    b2 = synth.q2k_blocks(np.random.default_rng(12), 3001)
    y2 = dq.dequant_q2k(cuda(b2)).cpu().numpy()
    r2 = orc.dequant_q2k(b2).astype(np.float32)
    assert np.array_equal(y2.view(np.uint32), r2.view(np.uint32))
    blk = orc.pack_q2k(0x3C00, 0x3800, [7] * 16, [15] * 16, [0] * 256)
    assert np.all(dq.dequant_q2k(cuda(blk)).cpu().numpy() == -7.5)
    q = [n % 4 for n in range(256)]
    blk = orc.pack_q2k(0x3C00, 0x3800, list(range(16)), [15 - j for j in range(16)], q)
    assert np.array_equal(dq.dequant_q2k(cuda(blk)).cpu().numpy().astype(np.float64), orc.dequant_q2k(blk))


def test_dequant_hand_built(dq, orc):
    blk = orc.pack_q6k(0x0400, [-128] * 16, [63] * 256)
    assert np.all(dq.dequant_q6k(cuda(blk)).cpu().numpy() == -0.2421875)
    blk = orc.pack_q4k(0x3C00, 0x3800, [5] * 8, [63] * 8, [0] * 256)
    assert np.all(dq.dequant_q4k(cuda(blk)).cpu().numpy() == -31.5)


# --------------------------------------------------------------- GEMV


BF16_SHAPES = [(512, 4096), (1003, 4096), (7, 8), (33, 1024), (1024, 4096), (4096, 4096), (12288, 4096),
               (4096, 12288), (151936, 4096)]


@pytest.mark.parametrize("rows,K", BF16_SHAPES)
def test_gemv_bf16(dq, orc, rows, K):
    W, x = synth.bf16_gemv_inputs(4, rows, K)
    y = dq.gemv_bf16(cuda(W.view(np.int16)), cuda(x.view(np.int16))).cpu().numpy()
    r = orc.gemv_bf16(W, x)
    assert normwise(y, r) <= GEMV_TOL


Q4K_SHAPES = [(300, 4096), (1, 4096), (37, 256), (129, 768), (257, 2048), (64, 12288), (8, 16384),
              (12288, 4096), (4096, 4096), (6144, 4096), (4096, 12288)]


@pytest.mark.parametrize("rows,K", Q4K_SHAPES)
def test_gemv_q4k(dq, orc, rows, K):
    W = synth.quant_matrix(5, synth.FMT_Q4K, rows, K)
    x = synth.activation(5, K)
    y = dq.gemv_q4k(cuda(W), cuda(x)).cpu().numpy()
    r = orc.gemv_q4k(W, x, rows, K)
    assert normwise(y, r) <= GEMV_TOL


Q6K_SHAPES = [(300, 4096), (1, 2048), (77, 6144), (4096, 12288), (151936, 4096), (5, 16384)]


@pytest.mark.parametrize("rows,K", Q6K_SHAPES)
def test_gemv_q6k(dq, orc, rows, K):
    W = synth.quant_matrix(6, synth.FMT_Q6K, rows, K)
    x = synth.activation(6, K)
    y = dq.gemv_q6k(cuda(W), cuda(x)).cpu().numpy()
    r = orc.gemv_q6k(W, x, rows, K)
    assert normwise(y, r) <= GEMV_TOL


Q2K_SHAPES = [(300, 4096), (1, 1024), (77, 3072), (12288, 4096), (4096, 12288), (151936, 4096), (5, 16384)]


@pytest.mark.parametrize("rows,K", Q2K_SHAPES)
def test_gemv_q2k(dq, orc, rows, K):
    W = synth.quant_matrix(8, synth.FMT_Q2K, rows, K)
    x = synth.activation(8, K)
    y = dq.gemv_q2k(cuda(W), cuda(x)).cpu().numpy()
    r = orc.gemv_q2k(W, x, rows, K)
    assert normwise(y, r) <= GEMV_TOL


@pytest.mark.parametrize("fmt,rows,K", [(0, 4096, 4096), (1, 12288, 4096), (1, 37, 256), (2, 300, 4096),
                                         (3, 77, 3072)])
def test_gemv_static_weights_flag(dq, orc, fmt, rows, K):
    """The static-weights flag only moves the first weight copies before the wait on
    the previous kernel: the result is the default entry point's, bit for bit, and the
    oracle's within the GEMV tolerance.  Two calls each, after another GEMV on the
    stream."""
    if fmt == dq.FMT_BF16:
        Wn, xn = synth.bf16_gemv_inputs(4, rows, K)
        W, x = cuda(Wn.view(np.int16)), cuda(xn.view(np.int16))
        r = orc.gemv_bf16(Wn, xn)
    else:
        Wn = synth.quant_matrix(9, fmt, rows, K)
        xn = synth.activation(9, K)
        W, x = cuda(Wn), cuda(xn)
        r = [None, orc.gemv_q4k, orc.gemv_q6k, orc.gemv_q2k][fmt](Wn, xn, rows, K)
    base = dq.gemv_ex(fmt, W, x).cpu().numpy()
    for _ in range(2):
        dq.gemv_ex(fmt, W, x)
        y = dq.gemv_ex(fmt, W, x, flags=dq.GEMV_STATIC_WEIGHTS).cpu().numpy()
        assert np.array_equal(y.view(np.uint32), base.view(np.uint32))
    assert normwise(base, r) <= GEMV_TOL


def test_gemv_q2k_integer_weights_and_extreme_activation(dq, orc):
    # d = dmin = 1: integer weights; a zero group, a tiny group and an outlier in x
    rng = np.random.default_rng(14)
    rows, K = 40, 2048
    blocks = [orc.pack_q2k(0x3C00, 0x3C00, rng.integers(0, 16, 16), rng.integers(0, 16, 16), rng.integers(0, 4, 256))
              for _ in range(rows * K // 256)]
    W = np.concatenate(blocks).reshape(rows, -1)
    x = synth.activation(14, K)
    x[:32] = 0.0
    x[32:64] *= 1e-6
    x[100] = 1e4
    y = dq.gemv_q2k(cuda(W), cuda(x)).cpu().numpy()
    assert normwise(y, orc.gemv_q2k(W, x, rows, K)) <= GEMV_TOL
    assert dq.device_error() == 0


def test_gemv_quant_condition_aware(dq, orc):
    # error against sum_k |W_rk x_k|, per row (well inside the bar for 15-bit activations)
    rows, K = 513, 4096
    for fmt, fn, deq in ((synth.FMT_Q4K, dq.gemv_q4k, orc.dequant_q4k), (synth.FMT_Q6K, dq.gemv_q6k, orc.dequant_q6k),
                         (synth.FMT_Q2K, dq.gemv_q2k, orc.dequant_q2k)):
        W = synth.quant_matrix(7, fmt, rows, K)
        x = synth.activation(7, K)
        y = fn(cuda(W), cuda(x)).cpu().numpy().astype(np.float64)
        Wd = deq(W).reshape(rows, K)
        r = Wd @ x.astype(np.float64)
        cond = np.abs(Wd) @ np.abs(x.astype(np.float64))
        assert np.max(np.abs(y - r) / cond) <= 1e-4


def test_gemv_extreme_activation(dq, orc):
    # a group whose values span 12 orders of magnitude, a zero group and an outlier
    rows, K = 40, 4096
    W = synth.quant_matrix(8, synth.FMT_Q4K, rows, K)
    x = synth.activation(8, K)
    x[:32] = 0.0
    x[32:64] *= 1e-6
    x[100] = 1e4
    y = dq.gemv_q4k(cuda(W), cuda(x)).cpu().numpy()
    assert normwise(y, orc.gemv_q4k(W, x, rows, K)) <= GEMV_TOL


# ---------------------------------------------------------- attention


def _attn_inputs(seed, n_q, n_kv, max_ctx, n_keys):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((n_q, 128)).astype(np.float32)
    k = rng.standard_normal((n_kv, max_ctx, 128)).astype(np.float16)
    v = rng.standard_normal((n_kv, max_ctx, 128)).astype(np.float16)
    return q, k, v


@pytest.mark.parametrize("n_q,n_kv,n_keys", [(32, 8, 1), (32, 8, 7), (32, 8, 32), (32, 8, 33), (32, 8, 64), (32, 8, 65), (32, 8, 513),
                                             (32, 8, 1024), (16, 2, 100), (8, 8, 17)])
def test_attention(dq, orc, n_q, n_kv, n_keys):
    q, k, v = _attn_inputs(n_keys, n_q, n_kv, 1024, n_keys)
    ws = dq.attention_workspace(n_q, n_kv)
    qt, kt, vt = cuda(q), cuda(k), cuda(v)
    for _ in range(2):  # the workspace must come back zeroed and reusable
        o = dq.attention_decode(qt, kt, vt, n_keys, workspace=ws).cpu().numpy()
        r = orc.attention(q.astype(np.float64), k.view(np.uint16), v.view(np.uint16), n_keys)
        assert normwise(o, r) <= 1e-4


def test_rope_table(dq, orc):
    # row p, pair i: the rotation the oracle applies to the unit vector e_i is (cos, sin) of that angle
    max_ctx, hd, theta = 40960, 128, 1.0e6
    tab = dq.rope_table(max_ctx, hd, theta).cpu().numpy().astype(np.float64)
    for p in (0, 1, 7, 1000, 32767, 40959):
        for i in range(hd // 2):
            e = np.zeros(hd)
            e[i] = 1.0
            r = orc.rope(e, p, theta)
            assert abs(tab[p, i, 0] - r[i]) <= 1.2e-7 and abs(tab[p, i, 1] - r[i + hd // 2]) <= 1.2e-7, (p, i)
    assert np.all(tab[0, :, 0] == 1.0) and np.all(tab[0, :, 1] == 0.0)


@pytest.mark.parametrize("n_q,n_kv,n_keys", [(32, 8, 1), (32, 8, 64), (32, 8, 65), (16, 2, 1100), (8, 8, 3000)])
def test_attention_decode_rope(dq, orc, n_q, n_kv, n_keys):
    max_ctx, theta, eps = 3072, 1.0e6, 1e-6
    rng = np.random.default_rng(700 + n_keys)
    q = (rng.standard_normal((n_q, 128)) * 3.0).astype(np.float32)
    k_new = (rng.standard_normal((n_kv, 128)) * 3.0).astype(np.float32)
    q_norm = rng.normal(1.0, 0.1, 128).astype(np.float32)
    k_norm = rng.normal(1.0, 0.1, 128).astype(np.float32)
    k = rng.standard_normal((n_kv, max_ctx, 128)).astype(np.float16)
    v = rng.standard_normal((n_kv, max_ctx, 128)).astype(np.float16)
    pos = n_keys - 1
    k[:, pos, :] = 0  # written by the call
    rope = dq.rope_table(max_ctx, 128, theta)
    kt = cuda(k)
    o = dq.attention_decode_rope(cuda(q), cuda(k_new), kt, cuda(v), cuda(q_norm), cuda(k_norm), rope, n_keys,
                                 eps=eps).cpu().numpy()
    # oracle: normalise and rotate each head, append the key in fp16, attend
    qr = np.stack([orc.rope(orc.head_rmsnorm(q[h], q_norm, eps), pos, theta) for h in range(n_q)])
    kref = np.stack([orc.rope(orc.head_rmsnorm(k_new[g], k_norm, eps), pos, theta) for g in range(n_kv)])
    k_ref = k.copy()
    k_ref[:, pos, :] = kref.astype(np.float16)
    r = orc.attention(qr, k_ref.view(np.uint16), v.view(np.uint16), n_keys)
    assert normwise(o, r) <= 1e-4
    got = kt.cpu().numpy()
    # the appended key: the fp16 rounding of a value within fp32 arithmetic of the exact one
    assert np.max(np.abs(got[:, pos, :].astype(np.float64) - kref)) <= np.max(np.abs(kref)) * 2.0 ** -10
    assert np.array_equal(np.delete(got, pos, axis=1).view(np.uint16), np.delete(k, pos, axis=1).view(np.uint16))
    assert dq.device_error() == 0


# ------------------------------------------------------------- M-sweep


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8, 16, 64])
def test_matmul_q4k(dq, orc, M):
    rows, K = 12288, 4096
    W = synth.quant_matrix(9, synth.FMT_Q4K, rows, K)
    X = np.stack([synth.activation(9, K, m) for m in range(M)])
    R = orc.matmul_q4k(W, X, rows, K)
    for path in (dq.MATMUL_AUTO, dq.MATMUL_CUDA_CORE, dq.MATMUL_TENSOR):
        Y = dq.matmul_q4k(cuda(W), cuda(X), path=path).cpu().numpy()
        for m in range(M):
            assert normwise(Y[m], R[m]) <= GEMV_TOL, (path, m)


@pytest.mark.parametrize("rows,K,M", [(1000, 256, 3), (20000, 512, 17), (152, 1024, 33), (77, 2048, 64)])
def test_matmul_q4k_tensor_shapes(dq, orc, rows, K, M):
    # ragged row tiles, a single block column, several 128-row tiles per block, one row per block
    W = synth.quant_matrix(11, synth.FMT_Q4K, rows, K)
    X = np.stack([synth.activation(11, K, m) for m in range(M)])
    R = orc.matmul_q4k(W, X, rows, K)
    Y = dq.matmul_q4k(cuda(W), cuda(X), path=dq.MATMUL_TENSOR).cpu().numpy()
    for m in range(M):
        assert normwise(Y[m], R[m]) <= GEMV_TOL, m
    assert dq.device_error() == 0


@pytest.mark.parametrize("rows,K,M", [(12288, 4096, 1), (12288, 4096, 16), (12288, 4096, 64), (128, 4096, 3),
                                      (300, 768, 5), (1000, 2048, 8), (20000, 512, 17), (77, 2048, 2),
                                      (256, 16384, 4), (40000, 256, 33)])
def test_matmul_q4k_split(dq, orc, rows, K, M):
    """K split across blocks: the 12288 x 4096 table (tiles shared by two or three
    blocks), one tile shared by 16 blocks, two tiles of 64 block columns shared by 64
    blocks each, ragged last tiles, fewer stages than SMs, and single-column rows
    where every block takes whole tiles.  Against the oracle at the GEMV bar; a second call on the same workspace
    (its tile counts left at zero) gives the same bits."""
    W = synth.quant_matrix(13, synth.FMT_Q4K, rows, K)
    X = np.stack([synth.activation(13, K, m) for m in range(M)])
    R = orc.matmul_q4k(W, X, rows, K)
    Wd, Xd = cuda(W), cuda(X)
    ws = dq.matmul_split_workspace(M, rows, K)
    Y = dq.matmul_q4k_split(Wd, Xd, ws).cpu().numpy()
    for m in range(M):
        assert normwise(Y[m], R[m]) <= GEMV_TOL, m
    Y2 = dq.matmul_q4k_split(Wd, Xd, ws).cpu().numpy()
    assert np.array_equal(Y.view(np.uint32), Y2.view(np.uint32))
    assert int(ws[:65536].view(torch.int32).abs().sum()) == 0  # the counts are back at zero
    assert dq.device_error() == 0


@pytest.mark.parametrize("M", [8, 32, 64])
def test_matmul_q4k_split_graph_replay(dq, M):
    """Two calls captured in one CUDA graph (dependent launches, and above 16 tokens
    the activation pre-pass) and the graph replayed twice: every replay gives the
    eager call's bits, and the counts are back at zero after each."""
    rows, K = 12288, 4096
    W = cuda(synth.quant_matrix(15, synth.FMT_Q4K, rows, K))
    X = cuda(np.stack([synth.activation(15, K, m) for m in range(M)]))
    ws = dq.matmul_split_workspace(M, rows, K)
    ref = dq.matmul_q4k_split(W, X, ws).clone()
    Y1 = torch.empty_like(ref)
    Y2 = torch.empty_like(ref)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            dq.matmul_q4k_split(W, X, ws, out=Y1)
            dq.matmul_q4k_split(W, X, ws, out=Y2)
    torch.cuda.synchronize()
    for _ in range(2):
        Y1.zero_()
        Y2.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(Y1, ref) and torch.equal(Y2, ref)
        assert int(ws[:65536].view(torch.int32).abs().sum()) == 0
    assert dq.device_error() == 0


def test_matmul_q4k_split_workspace_reuse(dq, orc):
    """One workspace, sized for the largest, serves calls of several shapes in turn."""
    ws = dq.matmul_split_workspace(64, 12288, 4096)
    for rows, K, M in ((12288, 4096, 16), (300, 768, 5), (128, 4096, 64), (12288, 4096, 2)):
        W = synth.quant_matrix(14, synth.FMT_Q4K, rows, K)
        X = np.stack([synth.activation(14, K, m) for m in range(M)])
        R = orc.matmul_q4k(W, X, rows, K)
        Y = dq.matmul_q4k_split(cuda(W), cuda(X), ws).cpu().numpy()
        for m in range(M):
            assert normwise(Y[m], R[m]) <= GEMV_TOL, (rows, K, M, m)
    assert dq.device_error() == 0


# -------------------------------------------------------------- decode


def _log_margin(case, pos, err, tol):
    """Append one measured decode error to the file named by DQ_PARITY_LOG (if set)."""
    path = os.environ.get("DQ_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write("%s pos=%d err=%.3e tol=%.1e margin=%.1fx\n" % (case, pos, err, tol, tol / max(err, 1e-300)))


def _run_decode(dq, orc, m, kv, positions, use_graph=True, seed=0, flags=0, fused=None, w=None):
    """Decode `positions` on the GPU and in the oracle; returns the GPU logits per step.

    Bar per step: max|gpu - oracle| / max|oracle| <= 2e-3 (the GEMV bar), on
    every model.  `fused` (when not None) is the expected execution mode of the
    model.
    """
    from quantised_gemv_norm_gb300 import upload

    if w is None:
        w = upload.to_device(m, kv)
    else:
        w["kv_cache"].copy_(torch.from_numpy(kv.view(np.int16)).to("cuda"))
    model = dq.Model(**upload.model_kwargs(m), weights=w, use_graph=use_graph, flags=flags)
    if fused is not None:
        assert model.fused == fused
        assert model.launches_per_step == (1 if fused else 2 + 5 * m.n_layers)
    kv_host = kv.copy()
    outs = []
    case = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    for t, pos in enumerate(positions):
        x = synth.decode_input(seed, m.hidden, t)
        logits = model.step(cuda(x), pos).cpu().numpy()
        outs.append(logits)
        ref = orc.decode_step(m, x, pos, kv_host)
        err = normwise(logits, ref)
        _log_margin(case, pos, err, GEMV_TOL)
        assert err <= GEMV_TOL, (pos, err)
        # the cache rows this token appended: fp16 values of k and v
        got = w["kv_cache"].cpu().numpy().view(np.float16)[:, :, :, pos, :].astype(np.float64)
        want = kv_host.view(np.float16)[:, :, :, pos, :].astype(np.float64)
        assert normwise(got, want) <= GEMV_TOL
    model.close()
    assert dq.device_error() == 0
    return outs


MODES = {"fused": (2, True), "kernels": (0, False)}  # flags (DQ_MODEL_FUSED = 2), expected fused


@pytest.mark.parametrize("mode", ["fused", "kernels"])
def test_decode_small_model_steps(dq, orc, mode):
    m = synth.make_model(21, n_layers=2, hidden=2048, ffn=4096, n_q_heads=8, n_kv_heads=2, head_dim=128,
                         vocab=1000, max_ctx=64)
    kv = synth.make_kv_cache(21, m, 0)
    flags, fused = MODES[mode]
    _run_decode(dq, orc, m, kv, [0, 1, 2, 3], flags=flags, fused=fused)


@pytest.mark.parametrize("mode", ["fused", "kernels"])
def test_decode_small_model_attention_chunks(dq, orc, mode):
    # contexts around the attention's chunking: two chunks (64 keys), three, and 32 chunks of 35 keys
    m = synth.make_model(23, n_layers=2, hidden=2048, ffn=4096, n_q_heads=16, n_kv_heads=4, head_dim=128,
                         vocab=300, max_ctx=1200)
    kv = synth.make_kv_cache(23, m, 1100)
    flags, fused = MODES[mode]
    _run_decode(dq, orc, m, kv, [63, 64, 1100], flags=flags, fused=fused)


def test_decode_small_model_eager_equals_graph(dq, orc):
    # same kernels, same order: the CUDA graph and eager launches agree bit for bit
    m = synth.make_model(22, n_layers=2, hidden=2048, ffn=4096, n_q_heads=8, n_kv_heads=2, head_dim=128,
                         vocab=777, max_ctx=40)
    kv = synth.make_kv_cache(22, m, 30)
    eager = _run_decode(dq, orc, m, kv, [30, 31], use_graph=False, fused=False)
    graph = _run_decode(dq, orc, m, kv, [30, 31], use_graph=True, fused=False)
    for a, b in zip(eager, graph):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_decode_fused_is_deterministic(dq, orc):
    # the fused token kernel reduces in a fixed order: two runs agree bit for bit
    m = synth.make_model(24, n_layers=2, hidden=2048, ffn=4096, n_q_heads=8, n_kv_heads=2, head_dim=128,
                         vocab=500, max_ctx=80)
    kv = synth.make_kv_cache(24, m, 70)
    a = _run_decode(dq, orc, m, kv, [70, 71], flags=2, fused=True)
    b = _run_decode(dq, orc, m, kv, [70, 71], flags=2, fused=True)
    for x, y in zip(a, b):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32))


def test_decode_shape_outside_fused_kernel_runs_kernels(dq, orc):
    # hidden 6144 is beyond the fused kernel's activation registers: separate kernels run
    m = synth.make_model(25, n_layers=1, hidden=6144, ffn=2048, n_q_heads=8, n_kv_heads=2, head_dim=128,
                         vocab=256, max_ctx=16)
    kv = synth.make_kv_cache(25, m, 3)
    _run_decode(dq, orc, m, kv, [3], flags=2, fused=False)


@pytest.mark.parametrize("mode", ["fused", "kernels"])
def test_decode_small_model_qwen3_attention(dq, orc, mode):
    # per-head q/k RMSNorm and rotary embedding: the first positions, one and two chunks, 16 chunks
    m = synth.make_model(26, n_layers=2, hidden=2048, ffn=4096, n_q_heads=16, n_kv_heads=4, head_dim=128,
                         vocab=300, max_ctx=1200, qwen3_attention=True)
    kv = synth.make_kv_cache(26, m, 1100)
    flags, fused = MODES[mode]
    _run_decode(dq, orc, m, kv, [0, 1, 2, 63, 64, 1100], flags=flags, fused=fused)


@pytest.mark.parametrize("qwen3", [False, True])
@pytest.mark.parametrize("mode", ["fused", "kernels"])
def test_decode_short_context_fold_boundary(dq, orc, mode, qwen3):
    # the fused kernel folds the attention into the O phase up to 4 keys (pos 3) and
    # runs the attention phase from 5 keys on; both sides of the boundary, and the
    # cache rows written by the fold (block 0) are read back by the next steps
    m = synth.make_model(28, n_layers=2, hidden=2048, ffn=4096, n_q_heads=16, n_kv_heads=4, head_dim=128,
                         vocab=400, max_ctx=32, qwen3_attention=qwen3)
    kv = synth.make_kv_cache(28, m, 1)
    flags, fused = MODES[mode]
    _run_decode(dq, orc, m, kv, [1, 2, 3, 4, 5], flags=flags, fused=fused)


@pytest.mark.parametrize("mode", ["fused", "kernels"])
def test_decode_many_attention_items_per_block(dq, orc, mode):
    # 32 KV heads x 32 key chunks = 1024 attention items: in the fused kernel every
    # pair of warp groups runs several, the merging chunks after the plain ones
    m = synth.make_model(35, n_layers=2, hidden=2048, ffn=2048, n_q_heads=32, n_kv_heads=32, head_dim=128,
                         vocab=300, max_ctx=1200, qwen3_attention=True)
    kv = synth.make_kv_cache(35, m, 1100)
    flags, fused = MODES[mode]
    _run_decode(dq, orc, m, kv, [1100, 1101], flags=flags, fused=fused)


@pytest.mark.parametrize("n_q,n_kv", [(16, 2), (8, 8)])
@pytest.mark.parametrize("mode", ["fused", "kernels"])
def test_decode_group_sizes(dq, orc, mode, n_q, n_kv):
    # 8 query heads per KV head (two attention items fill the fused block's 16 warps) and
    # one (two warps work); short, one-chunk and many-chunk contexts
    m = synth.make_model(29, n_layers=2, hidden=2048, ffn=4096, n_q_heads=n_q, n_kv_heads=n_kv, head_dim=128,
                         vocab=300, max_ctx=700, qwen3_attention=True)
    kv = synth.make_kv_cache(29, m, 650)
    flags, fused = MODES[mode]
    _run_decode(dq, orc, m, kv, [2, 40, 650, 699], flags=flags, fused=fused)  # 699: last row


@pytest.mark.parametrize("mode", ["fused", "kernels"])
def test_decode_step_argument_errors(dq, orc, mode):
    # positions outside the cache and null buffers are refused before any launch
    from quantised_gemv_norm_gb300 import upload

    m = synth.make_model(30, n_layers=1, hidden=2048, ffn=2048, n_q_heads=8, n_kv_heads=2, head_dim=128,
                         vocab=256, max_ctx=16)
    w = upload.to_device(m, synth.make_kv_cache(30, m, 0))
    model = dq.Model(**upload.model_kwargs(m), weights=w, flags=MODES[mode][0])
    x = cuda(synth.decode_input(30, m.hidden))
    for pos in (-1, m.max_ctx, m.max_ctx + 5):
        with pytest.raises(dq.DQError) as e:
            model.step(x, pos)
        assert e.value.status == -2
    lib = dq.load()
    assert lib.dq_decode_step(model._h, None, 0, ctypes.c_void_p(x.data_ptr()), None) == -1
    logits = model.step(x, m.max_ctx - 1)  # the last row is valid
    assert bool(torch.isfinite(logits).all())
    model.close()
    assert dq.device_error() == 0


@pytest.mark.parametrize("mode", ["fused", "kernels"])
def test_decode_step_host_matches_device_step(dq, orc, mode):
    # the host-buffer entry point: same logits bit for bit as the device one, and its
    # argument errors (pinned and pageable host buffers both work)
    from quantised_gemv_norm_gb300 import upload

    m = synth.make_model(36, n_layers=2, hidden=2048, ffn=2048, n_q_heads=8, n_kv_heads=2, head_dim=128,
                         vocab=300, max_ctx=16, qwen3_attention=True)
    kv = synth.make_kv_cache(36, m, 3)
    w = upload.to_device(m, kv)
    model = dq.Model(**upload.model_kwargs(m), weights=w, flags=MODES[mode][0])
    x = synth.decode_input(36, m.hidden)
    ref = orc.decode_step(m, x, 3, kv.copy())
    dev = model.step(cuda(x), 3).cpu().numpy()
    for pinned in (True, False):
        xh = torch.from_numpy(x.copy())
        out = torch.empty(m.vocab, dtype=torch.float32)
        if pinned:
            xh, out = xh.pin_memory(), out.pin_memory()
        got = model.step_host(xh, 3, out).numpy()
        assert np.array_equal(got.view(np.uint32), dev.view(np.uint32))
        assert normwise(got, ref) <= GEMV_TOL
    lib = dq.load()
    xh = torch.from_numpy(x.copy())
    assert lib.dq_decode_step_host(model._h, None, 0, ctypes.c_void_p(xh.data_ptr()), None) == -1
    assert lib.dq_decode_step_host(model._h, ctypes.c_void_p(xh.data_ptr()), m.max_ctx,
                                   ctypes.c_void_p(xh.data_ptr()), None) == -2
    model.close()
    assert dq.device_error() == 0


def test_decode_qwen3_attention_modes_agree(dq, orc):
    # the fused kernel and the separate kernels compute the same norm, rotation and cache row
    m = synth.make_model(27, n_layers=2, hidden=2048, ffn=4096, n_q_heads=8, n_kv_heads=2, head_dim=128,
                         vocab=500, max_ctx=300, qwen3_attention=True)
    kv = synth.make_kv_cache(27, m, 257)
    a = _run_decode(dq, orc, m, kv, [257, 258], flags=2, fused=True)
    b = _run_decode(dq, orc, m, kv, [257, 258], flags=0, fused=False)
    for x, y in zip(a, b):
        assert normwise(x, y) <= GEMV_TOL


_QWEN = {}


def _qwen3():
    # the Qwen3-8B shape with Qwen3's attention inputs (q/k head norms, rotary base 1e6)
    if "m" not in _QWEN:
        from quantised_gemv_norm_gb300 import upload
        m = synth.make_model(1, max_ctx=1024, qwen3_attention=True, **synth.QWEN3_8B)
        _QWEN["m"] = m
        _QWEN["w"] = upload.to_device(m, synth.make_kv_cache(1, m, 0))
    return _QWEN["m"], _QWEN["w"]


@pytest.mark.parametrize("mode", ["fused", "kernels"])
def test_decode_qwen3_8b_shape_empty_cache(dq, orc, mode):
    m, w = _qwen3()
    kv = synth.make_kv_cache(1, m, 0)
    flags, fused = MODES[mode]
    _run_decode(dq, orc, m, kv, [0], flags=flags, fused=fused, w=w)


@pytest.mark.parametrize("mode", ["fused", "kernels"])
def test_decode_qwen3_8b_shape_512_context(dq, orc, mode):
    m, w = _qwen3()
    kv = synth.make_kv_cache(2, m, 512)
    flags, fused = MODES[mode]
    _run_decode(dq, orc, m, kv, [512], flags=flags, fused=fused, w=w)


_LAYER_REF = {}


@pytest.mark.parametrize("pos", [0, 512])
@pytest.mark.parametrize("mode", ["fused", "kernels"])
def test_decode_qwen3_8b_shape_layer_residuals(dq, orc, mode, pos):
    # the residual stream after l layers (the hidden state that enters layer l), GPU
    # against oracle at the decode bar, for the Qwen3-8B-shaped stack cut after l
    # layers (same weights and cache): an error in one layer that the vocabulary
    # table damps would still show here
    import dataclasses

    from quantised_gemv_norm_gb300 import upload

    m, w = _qwen3()
    kv = synth.make_kv_cache(2, m, pos)
    w["kv_cache"].copy_(torch.from_numpy(kv.view(np.int16)).to("cuda"))
    x = synth.decode_input(3, m.hidden)
    per_layer = ("attn_norm", "wqkv", "wo", "ffn_norm", "wgate", "wup", "wdown", "down_fmt", "q_norm", "k_norm")
    vocab = 1024
    case = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    for n in (1, 2, 9, 18, 36):
        ms = dataclasses.replace(m, n_layers=n, vocab=vocab, wvocab=m.wvocab[:vocab],
                                 **{k: getattr(m, k)[:n] for k in per_layer})
        if (pos, n) not in _LAYER_REF:
            _, hid = orc.decode_step(ms, x, pos, np.ascontiguousarray(kv[:n]), want_hidden=True)
            _LAYER_REF[(pos, n)] = hid
        ref = _LAYER_REF[(pos, n)]
        ws = {k: (v[:n] if isinstance(v, list) else v) for k, v in w.items()}
        ws["wvocab"] = w["wvocab"][:vocab]
        model = dq.Model(**upload.model_kwargs(ms), weights=ws, flags=MODES[mode][0])
        assert model.fused == MODES[mode][1]
        model.step(cuda(x), pos)
        got = model.buffer(0, m.hidden).cpu().numpy()
        model.close()
        err = normwise(got, ref)
        _log_margin("%s layers=%d" % (case, n), pos, err, GEMV_TOL)
        assert err <= GEMV_TOL, (n, err)
    assert dq.device_error() == 0
