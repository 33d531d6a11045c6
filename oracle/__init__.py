"""CPU oracle for the decode hot path -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
Python binding) never imports, links or runs it.  It shares no code with the
CUDA path: it is plain C (``dq_oracle.c``, fp64 accumulation) behind ctypes.

Every function here takes numpy arrays on the host and returns numpy float64
results.  The formats and formulas are documented at the top of dq_oracle.c.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dq_oracle.c")
_LIB = os.path.join(_HERE, "libdq_oracle.so")
_lib = None

Q4K_BLOCK_BYTES = 144
Q6K_BLOCK_BYTES = 210
Q2K_BLOCK_BYTES = 84


def build(force: bool = False) -> str:
    """Compile dq_oracle.c into libdq_oracle.so next to it (plain gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".%d.tmp" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    i32, i64, f64 = ctypes.c_int, ctypes.c_longlong, ctypes.c_double
    sig = {
        "oracle_half_to_double": (f64, [ctypes.c_uint16]),
        "oracle_double_to_half": (ctypes.c_uint16, [f64]),
        "oracle_bf16_to_double": (f64, [ctypes.c_uint16]),
        "oracle_unpack_q4k": (None, [P, P, P, P, P, P]),
        "oracle_pack_q4k": (None, [ctypes.c_uint16, ctypes.c_uint16, P, P, P, P]),
        "oracle_unpack_q6k": (None, [P, P, P, P]),
        "oracle_pack_q6k": (None, [ctypes.c_uint16, P, P, P]),
        "oracle_dequant_q4k": (None, [P, i64, P]),
        "oracle_unpack_q2k": (None, [P, P, P, P, P, P]),
        "oracle_pack_q2k": (None, [ctypes.c_uint16, ctypes.c_uint16, P, P, P, P]),
        "oracle_dequant_q2k": (None, [P, i64, P]),
        "oracle_gemv_q2k": (None, [P, P, P, i32, i32]),
        "oracle_dequant_q6k": (None, [P, i64, P]),
        "oracle_gemv_bf16": (None, [P, P, P, i32, i32]),
        "oracle_gemv_q4k": (None, [P, P, P, i32, i32]),
        "oracle_gemv_q6k": (None, [P, P, P, i32, i32]),
        "oracle_matmul_q4k": (None, [P, P, P, i32, i32, i32]),
        "oracle_rmsnorm": (None, [P, P, P, i32, i32, f64]),
        "oracle_layernorm": (None, [P, P, P, P, i32, i32, f64]),
        "oracle_attention": (None, [P, P, P, P, i32, i32, i32, i32, i32]),
        "oracle_silu": (f64, [f64]),
        "oracle_head_rmsnorm": (None, [P, P, i32, f64]),
        "oracle_rope": (None, [P, i32, i32, f64]),
        "oracle_decode_step": (None, [P, P, i32, P, P]),
        "oracle_num_threads": (i32, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return _load().oracle_num_threads()


# ------------------------------------------------------------------ scalars


def half_to_double(bits: int) -> float:
    return _load().oracle_half_to_double(int(bits))


def double_to_half(v: float) -> int:
    return int(_load().oracle_double_to_half(float(v)))


def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(int(bits))


def silu(z: float) -> float:
    return _load().oracle_silu(float(z))


# ------------------------------------------------------------- block codecs


def unpack_q4k(block: np.ndarray):
    """-> (d, dmin, sc[8], m[8], q[256]) of one 144-byte Q4_K block."""
    blk = _c(block, np.uint8)
    assert blk.size == Q4K_BLOCK_BYTES
    d = ctypes.c_double()
    dmin = ctypes.c_double()
    sc = np.zeros(8, np.int32)
    m = np.zeros(8, np.int32)
    q = np.zeros(256, np.int32)
    _load().oracle_unpack_q4k(_p(blk), ctypes.byref(d), ctypes.byref(dmin), _p(sc), _p(m), _p(q))
    return d.value, dmin.value, sc, m, q


def pack_q4k(d_bits: int, dmin_bits: int, sc, m, q) -> np.ndarray:
    out = np.zeros(Q4K_BLOCK_BYTES, np.uint8)
    _load().oracle_pack_q4k(int(d_bits), int(dmin_bits), _p(_c(sc, np.int32)), _p(_c(m, np.int32)),
                            _p(_c(q, np.int32)), _p(out))
    return out


def unpack_q2k(block: np.ndarray):
    """-> (d, dmin, sc[16], m[16], q[256]) of one 84-byte Q2_K block."""
    blk = _c(block, np.uint8)
    assert blk.size == Q2K_BLOCK_BYTES
    d = ctypes.c_double()
    dmin = ctypes.c_double()
    sc = np.zeros(16, np.int32)
    m = np.zeros(16, np.int32)
    q = np.zeros(256, np.int32)
    _load().oracle_unpack_q2k(_p(blk), ctypes.byref(d), ctypes.byref(dmin), _p(sc), _p(m), _p(q))
    return d.value, dmin.value, sc, m, q


def pack_q2k(d_bits: int, dmin_bits: int, sc, m, q) -> np.ndarray:
    out = np.zeros(Q2K_BLOCK_BYTES, np.uint8)
    _load().oracle_pack_q2k(int(d_bits), int(dmin_bits), _p(_c(sc, np.int32)), _p(_c(m, np.int32)),
                            _p(_c(q, np.int32)), _p(out))
    return out


def dequant_q2k(blocks: np.ndarray) -> np.ndarray:
    b = _c(blocks, np.uint8).reshape(-1)
    assert b.size % Q2K_BLOCK_BYTES == 0
    n = b.size // Q2K_BLOCK_BYTES
    out = np.empty(n * 256, np.float64)
    _load().oracle_dequant_q2k(_p(b), n, _p(out))
    return out


def unpack_q6k(block: np.ndarray):
    """-> (d, sc[16], q[256]) of one 210-byte Q6_K block."""
    blk = _c(block, np.uint8)
    assert blk.size == Q6K_BLOCK_BYTES
    d = ctypes.c_double()
    sc = np.zeros(16, np.int32)
    q = np.zeros(256, np.int32)
    _load().oracle_unpack_q6k(_p(blk), ctypes.byref(d), _p(sc), _p(q))
    return d.value, sc, q


def pack_q6k(d_bits: int, sc, q) -> np.ndarray:
    out = np.zeros(Q6K_BLOCK_BYTES, np.uint8)
    _load().oracle_pack_q6k(int(d_bits), _p(_c(sc, np.int32)), _p(_c(q, np.int32)), _p(out))
    return out


def dequant_q4k(blocks: np.ndarray) -> np.ndarray:
    b = _c(blocks, np.uint8).reshape(-1)
    assert b.size % Q4K_BLOCK_BYTES == 0
    n = b.size // Q4K_BLOCK_BYTES
    out = np.empty(n * 256, np.float64)
    _load().oracle_dequant_q4k(_p(b), n, _p(out))
    return out


def dequant_q6k(blocks: np.ndarray) -> np.ndarray:
    b = _c(blocks, np.uint8).reshape(-1)
    assert b.size % Q6K_BLOCK_BYTES == 0
    n = b.size // Q6K_BLOCK_BYTES
    out = np.empty(n * 256, np.float64)
    _load().oracle_dequant_q6k(_p(b), n, _p(out))
    return out


# --------------------------------------------------------------------- GEMV


def gemv_bf16(W_bits: np.ndarray, x_bits: np.ndarray) -> np.ndarray:
    """W: uint16 bf16 bits [rows, K]; x: uint16 bf16 bits [K] -> float64 [rows]."""
    W = _c(W_bits, np.uint16)
    x = _c(x_bits, np.uint16).reshape(-1)
    rows, K = W.shape
    assert x.size == K
    y = np.empty(rows, np.float64)
    _load().oracle_gemv_bf16(_p(W), _p(x), _p(y), rows, K)
    return y


def _gemv_quant(fn, bpb, W, x, rows, K):
    Wb = _c(W, np.uint8).reshape(-1)
    assert K % 256 == 0 and Wb.size == rows * (K // 256) * bpb
    xf = _c(x, np.float32).reshape(-1)
    assert xf.size == K
    y = np.empty(rows, np.float64)
    fn(_p(Wb), _p(xf), _p(y), rows, K)
    return y


def gemv_q4k(W: np.ndarray, x: np.ndarray, rows: int, K: int) -> np.ndarray:
    return _gemv_quant(_load().oracle_gemv_q4k, Q4K_BLOCK_BYTES, W, x, rows, K)


def gemv_q2k(W: np.ndarray, x: np.ndarray, rows: int, K: int) -> np.ndarray:
    return _gemv_quant(_load().oracle_gemv_q2k, Q2K_BLOCK_BYTES, W, x, rows, K)


def gemv_q6k(W: np.ndarray, x: np.ndarray, rows: int, K: int) -> np.ndarray:
    return _gemv_quant(_load().oracle_gemv_q6k, Q6K_BLOCK_BYTES, W, x, rows, K)


def matmul_q4k(W: np.ndarray, X: np.ndarray, rows: int, K: int) -> np.ndarray:
    """X: float32 [M, K] -> float64 [M, rows]."""
    Wb = _c(W, np.uint8).reshape(-1)
    Xf = _c(X, np.float32)
    M = Xf.shape[0]
    assert Xf.shape[1] == K and Wb.size == rows * (K // 256) * Q4K_BLOCK_BYTES
    Y = np.empty((M, rows), np.float64)
    _load().oracle_matmul_q4k(_p(Wb), _p(Xf), _p(Y), M, rows, K)
    return Y


# -------------------------------------------------------------------- norms


def rmsnorm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    xf = _c(x, np.float32)
    rows, n = xf.shape
    y = np.empty((rows, n), np.float64)
    _load().oracle_rmsnorm(_p(xf), _p(_c(gamma, np.float32)), _p(y), rows, n, float(eps))
    return y


def layernorm(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float) -> np.ndarray:
    xf = _c(x, np.float32)
    rows, n = xf.shape
    y = np.empty((rows, n), np.float64)
    _load().oracle_layernorm(_p(xf), _p(_c(gamma, np.float32)), _p(_c(beta, np.float32)), _p(y),
                             rows, n, float(eps))
    return y


# ---------------------------------------------------------------- attention


def attention(q: np.ndarray, k_plane: np.ndarray, v_plane: np.ndarray, n_keys: int) -> np.ndarray:
    """q: [n_q, hd] (float64); k/v planes: fp16 bits [n_kv, max_ctx, hd] -> [n_q, hd]."""
    qd = _c(q, np.float64)
    n_q, hd = qd.shape
    kc = _c(k_plane, np.uint16)
    vc = _c(v_plane, np.uint16)
    n_kv, max_ctx, hd2 = kc.shape
    assert hd2 == hd and vc.shape == kc.shape and 1 <= n_keys <= max_ctx
    out = np.empty((n_q, hd), np.float64)
    _load().oracle_attention(_p(qd), _p(kc), _p(vc), _p(out), n_q, n_kv, hd, max_ctx, int(n_keys))
    return out


# -------------------------------------------------------------- decode step


class _Model(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("ffn", ctypes.c_int),
        ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
        ("vocab", ctypes.c_int), ("max_ctx", ctypes.c_int), ("eps", ctypes.c_double),
        ("attn_norm", ctypes.c_void_p), ("wqkv", ctypes.c_void_p), ("wo", ctypes.c_void_p),
        ("ffn_norm", ctypes.c_void_p), ("wgate", ctypes.c_void_p), ("wup", ctypes.c_void_p),
        ("wdown", ctypes.c_void_p), ("down_fmt", ctypes.c_void_p), ("out_norm", ctypes.c_void_p),
        ("wvocab", ctypes.c_void_p), ("kv_cache", ctypes.c_void_p),
        ("q_norm", ctypes.c_void_p), ("k_norm", ctypes.c_void_p), ("rope_theta", ctypes.c_double),
    ]


def head_rmsnorm(v: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """Per-head RMSNorm of one head vector (Qwen3 QK-norm); returns a new array."""
    out = np.array(v, dtype=np.float64, copy=True)
    _load().oracle_head_rmsnorm(_p(out), _p(_c(w, np.float32)), out.size, float(eps))
    return out


def rope(v: np.ndarray, pos: int, theta: float) -> np.ndarray:
    """Rotary position embedding of one head vector (rotate-half pairing); new array."""
    out = np.array(v, dtype=np.float64, copy=True)
    _load().oracle_rope(_p(out), out.size, int(pos), float(theta))
    return out


def decode_step(model, x_in: np.ndarray, pos: int, kv_cache: np.ndarray, want_hidden: bool = False):
    """One decode token on the host.

    ``model`` is any object with the attributes of a synthetic model (see the
    input generator): n_layers, hidden, ffn, n_q_heads, n_kv_heads, head_dim,
    vocab, max_ctx, eps, and per-layer lists attn_norm, wqkv, wo, ffn_norm,
    wgate, wup, wdown, down_fmt, plus out_norm and wvocab, all numpy arrays;
    optionally per-layer q_norm and k_norm and rope_theta (Qwen3 attention inputs).
    ``kv_cache`` (uint16 fp16 bits [L, 2, n_kv, max_ctx, hd]) is updated in place
    at ``pos``.  Returns float64 logits (and the final hidden state if asked).
    """
    L = model.n_layers
    keep = []

    def ptr_array(arrs, dtype):
        cs = [_c(a, dtype) for a in arrs]
        keep.extend(cs)
        arr = (ctypes.c_void_p * L)(*[c.ctypes.data for c in cs])
        keep.append(arr)
        return ctypes.cast(arr, ctypes.c_void_p)

    assert kv_cache.dtype == np.uint16 and kv_cache.flags["C_CONTIGUOUS"]
    assert kv_cache.shape == (L, 2, model.n_kv_heads, model.max_ctx, model.head_dim)
    down_fmt = np.asarray(model.down_fmt, np.int32)
    out_norm = _c(model.out_norm, np.float32)
    wvocab = _c(model.wvocab, np.uint8)
    m = _Model(L, model.hidden, model.ffn, model.n_q_heads, model.n_kv_heads, model.head_dim,
               model.vocab, model.max_ctx, float(model.eps),
               ptr_array(model.attn_norm, np.float32), ptr_array(model.wqkv, np.uint8),
               ptr_array(model.wo, np.uint8), ptr_array(model.ffn_norm, np.float32),
               ptr_array(model.wgate, np.uint8), ptr_array(model.wup, np.uint8),
               ptr_array(model.wdown, np.uint8), down_fmt.ctypes.data, out_norm.ctypes.data,
               wvocab.ctypes.data, kv_cache.ctypes.data,
               ptr_array(model.q_norm, np.float32) if getattr(model, "q_norm", None) else None,
               ptr_array(model.k_norm, np.float32) if getattr(model, "k_norm", None) else None,
               float(getattr(model, "rope_theta", 0.0) or 0.0))
    xin = _c(x_in, np.float32).reshape(-1)
    assert xin.size == model.hidden
    logits = np.empty(model.vocab, np.float64)
    hidden = np.empty(model.hidden, np.float64) if want_hidden else None
    _load().oracle_decode_step(ctypes.byref(m), _p(xin), int(pos), _p(logits),
                               _p(hidden) if want_hidden else None)
    del keep
    return (logits, hidden) if want_hidden else logits
