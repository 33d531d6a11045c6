"""Thin ctypes binding over libdq.so (argument marshalling only).

Every function takes torch tensors that live on the current CUDA device,
passes their data pointers and the current torch stream to the C ABI, and
raises DQError on a non-zero status.  All computation happens in the CUDA
kernels of libdq.so; there is no fallback: if the library is missing or no GPU
is present, the calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdq.so")

FMT_BF16, FMT_Q4K, FMT_Q6K, FMT_Q2K = 0, 1, 2, 3
Q4K_BLOCK_BYTES, Q6K_BLOCK_BYTES, Q2K_BLOCK_BYTES = 144, 210, 84

# name -> (restype, argtypes); the same names as include/dq.h
P, I, LL, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_float, ctypes.c_size_t
D = ctypes.c_double
SIGNATURES = {
    "dq_status_string": (ctypes.c_char_p, [I]),
    "dq_last_cuda_error": (I, []),
    "dq_device_error": (I, [P]),
    "dq_check_device": (I, [P]),
    "dq_model_debug_waits": (I, [P, ctypes.c_ulonglong, I]),
    "dq_debug_fail_next_allocs": (I, [I]),
    "dq_rmsnorm": (I, [P, P, P, I, I, F, P]),
    "dq_layernorm": (I, [P, P, P, P, I, I, F, P]),
    "dq_rmsnorm_threads": (I, [P, P, P, I, I, F, I, P]),
    "dq_layernorm_threads": (I, [P, P, P, P, I, I, F, I, P]),
    "dq_debug_trace": (I, [P]),
    "dq_gemv_bf16": (I, [P, P, P, I, I, P]),
    "dq_gemv_q4k": (I, [P, P, P, I, I, P]),
    "dq_gemv_q6k": (I, [P, P, P, I, I, P]),
    "dq_gemv_q2k": (I, [P, P, P, I, I, P]),
    "dq_gemv_ex": (I, [I, P, P, P, I, I, I, P]),
    "dq_dequant_q4k": (I, [P, P, LL, P]),
    "dq_dequant_q6k": (I, [P, P, LL, P]),
    "dq_dequant_q2k": (I, [P, P, LL, P]),
    "dq_attention_workspace_bytes": (SZ, [I, I]),
    "dq_attention_decode": (I, [P, P, P, P, I, I, I, I, I, P, SZ, P]),
    "dq_attention_decode_static": (I, [P, P, P, P, I, I, I, I, I, P]),
    "dq_rope_table": (I, [P, I, I, D, P]),
    "dq_attention_decode_rope": (I, [P, P, P, P, P, P, P, P, F, I, I, I, I, I, P, SZ, P]),
    "dq_matmul_q4k": (I, [P, P, P, I, I, I, P]),
    "dq_matmul_q4k_path": (I, [P, P, P, I, I, I, I, P]),
    "dq_matmul_q4k_split": (I, [P, P, P, I, I, I, P, LL, P]),
    "dq_matmul_q4k_split_workspace_bytes": (LL, [I, I, I]),
    "dq_model_create": (I, [P, P]),
    "dq_decode_step": (I, [P, P, I, P, P]),
    "dq_decode_step_host": (I, [P, P, I, P, P]),
    "dq_model_launches_per_step": (I, [P]),
    "dq_model_fused": (I, [P]),
    "dq_model_enqueue_kernel": (I, [P, I, I, P]),
    "dq_model_buffer": (I, [P, I, P]),
    "dq_model_destroy": (I, [P]),
}

_lib = None


class DQError(RuntimeError):
    def __init__(self, fn: str, status: int):
        lib = _lib
        msg = lib.dq_status_string(status).decode() if lib else str(status)
        extra = ""
        if lib and status == -5:
            extra = " (cudaError %d)" % lib.dq_last_cuda_error()
        super().__init__("%s failed: %s [%d]%s" % (fn, msg, status, extra))
        self.status = status


def load(path: str = LIB_PATH):
    """Load libdq.so; raises if it is missing (build it with __graft_entry__.build())."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("libdq.so not found at %s: build the CUDA extension first" % path)
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(fn: str, status: int):
    if status != 0:
        raise DQError(fn, status)


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t: torch.Tensor):
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def device_error() -> int:
    """Synchronise the current stream and read/clear the device error flag."""
    lib = load()
    v = lib.dq_device_error(_stream())
    if v < 0:
        raise DQError("dq_device_error", v)
    return v


# ---------------------------------------------------------------- norms


def rmsnorm(x: torch.Tensor, gamma: torch.Tensor, eps: float, out=None, threads: int | None = None):
    lib = load()
    rows, n = x.shape
    out = torch.empty_like(x) if out is None else out
    if threads is None:
        st = lib.dq_rmsnorm(_ptr(x), _ptr(gamma), _ptr(out), rows, n, eps, _stream())
    else:
        st = lib.dq_rmsnorm_threads(_ptr(x), _ptr(gamma), _ptr(out), rows, n, eps, threads, _stream())
    _check("dq_rmsnorm", st)
    return out


def layernorm(x, gamma, beta, eps: float, out=None, threads: int | None = None):
    lib = load()
    rows, n = x.shape
    out = torch.empty_like(x) if out is None else out
    if threads is None:
        st = lib.dq_layernorm(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(out), rows, n, eps, _stream())
    else:
        st = lib.dq_layernorm_threads(_ptr(x), _ptr(gamma), _ptr(beta), _ptr(out), rows, n, eps, threads,
                                      _stream())
    _check("dq_layernorm", st)
    return out


# ----------------------------------------------------------------- GEMV


def quant_K(fmt: int, row_bytes: int) -> int:
    bpb = {FMT_Q4K: Q4K_BLOCK_BYTES, FMT_Q6K: Q6K_BLOCK_BYTES, FMT_Q2K: Q2K_BLOCK_BYTES}[fmt]
    if row_bytes % bpb:
        raise ValueError("row bytes %d is not a whole number of blocks" % row_bytes)
    return row_bytes // bpb * 256


def gemv_bf16(W: torch.Tensor, x: torch.Tensor, out=None):
    """W: bf16/int16 [rows, K]; x: bf16/int16 [K] -> fp32 [rows]."""
    lib = load()
    rows, K = W.shape
    out = torch.empty(rows, dtype=torch.float32, device=W.device) if out is None else out
    _check("dq_gemv_bf16", lib.dq_gemv_bf16(_ptr(W), _ptr(x), _ptr(out), rows, K, _stream()))
    return out


def gemv_q4k(W: torch.Tensor, x: torch.Tensor, out=None):
    """W: uint8 [rows, K/256*144]; x: fp32 [K] -> fp32 [rows]."""
    lib = load()
    rows = W.shape[0]
    K = quant_K(FMT_Q4K, W.shape[1])
    out = torch.empty(rows, dtype=torch.float32, device=W.device) if out is None else out
    _check("dq_gemv_q4k", lib.dq_gemv_q4k(_ptr(W), _ptr(x), _ptr(out), rows, K, _stream()))
    return out


def gemv_q6k(W: torch.Tensor, x: torch.Tensor, out=None):
    lib = load()
    rows = W.shape[0]
    K = quant_K(FMT_Q6K, W.shape[1])
    out = torch.empty(rows, dtype=torch.float32, device=W.device) if out is None else out
    _check("dq_gemv_q6k", lib.dq_gemv_q6k(_ptr(W), _ptr(x), _ptr(out), rows, K, _stream()))
    return out


def dequant_q4k(blocks: torch.Tensor, out=None):
    lib = load()
    n = blocks.numel() // Q4K_BLOCK_BYTES
    out = torch.empty(n * 256, dtype=torch.float32, device=blocks.device) if out is None else out
    _check("dq_dequant_q4k", lib.dq_dequant_q4k(_ptr(blocks), _ptr(out), n, _stream()))
    return out


def dequant_q6k(blocks: torch.Tensor, out=None):
    lib = load()
    n = blocks.numel() // Q6K_BLOCK_BYTES
    out = torch.empty(n * 256, dtype=torch.float32, device=blocks.device) if out is None else out
    _check("dq_dequant_q6k", lib.dq_dequant_q6k(_ptr(blocks), _ptr(out), n, _stream()))
    return out


def gemv_q2k(W: torch.Tensor, x: torch.Tensor, out=None):
    lib = load()
    rows = W.shape[0]
    K = quant_K(FMT_Q2K, W.shape[1])
    out = torch.empty(rows, dtype=torch.float32, device=W.device) if out is None else out
    _check("dq_gemv_q2k", lib.dq_gemv_q2k(_ptr(W), _ptr(x), _ptr(out), rows, K, _stream()))
    return out


GEMV_STATIC_WEIGHTS = 1


def gemv_ex(fmt: int, W: torch.Tensor, x: torch.Tensor, out=None, flags: int = 0):
    """The four GEMVs through dq_gemv_ex.  flags: GEMV_STATIC_WEIGHTS when the kernel
    before this call on the stream does not write W (the copies of W may then start
    before that kernel completes)."""
    lib = load()
    rows = W.shape[0]
    K = W.shape[1] if fmt == FMT_BF16 else quant_K(fmt, W.shape[1])
    out = torch.empty(rows, dtype=torch.float32, device=W.device) if out is None else out
    _check("dq_gemv_ex", lib.dq_gemv_ex(int(fmt), _ptr(W), _ptr(x), _ptr(out), rows, K, int(flags), _stream()))
    return out


def dequant_q2k(blocks: torch.Tensor, out=None):
    lib = load()
    n = blocks.numel() // Q2K_BLOCK_BYTES
    out = torch.empty(n * 256, dtype=torch.float32, device=blocks.device) if out is None else out
    _check("dq_dequant_q2k", lib.dq_dequant_q2k(_ptr(blocks), _ptr(out), n, _stream()))
    return out


MATMUL_AUTO, MATMUL_CUDA_CORE, MATMUL_TENSOR = 0, 1, 2


def matmul_q4k(W: torch.Tensor, X: torch.Tensor, out=None, path: int = MATMUL_AUTO):
    """W: uint8 [rows, K/256*144]; X: fp32 [M, K] -> fp32 [M, rows].

    ``path``: MATMUL_AUTO (CUDA cores up to M = 2, tensor cores above),
    MATMUL_CUDA_CORE (one GEMV per token) or MATMUL_TENSOR (one read of W)."""
    lib = load()
    rows = W.shape[0]
    K = quant_K(FMT_Q4K, W.shape[1])
    M = X.shape[0]
    out = torch.empty((M, rows), dtype=torch.float32, device=W.device) if out is None else out
    _check("dq_matmul_q4k_path",
           lib.dq_matmul_q4k_path(_ptr(W), _ptr(X), _ptr(out), M, rows, K, int(path), _stream()))
    return out


def matmul_split_workspace(M: int, rows: int, K: int, device=None) -> torch.Tensor:
    """A zero-filled workspace for matmul_q4k_split of this shape (reusable by
    later calls on the same stream whose shapes fit)."""
    lib = load()
    nbytes = lib.dq_matmul_q4k_split_workspace_bytes(M, rows, K)
    if nbytes < 0:
        _check("dq_matmul_q4k_split_workspace_bytes", int(nbytes))
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")


def matmul_q4k_split(W: torch.Tensor, X: torch.Tensor, workspace: torch.Tensor, out=None):
    """The tensor-core product with K split across blocks (every 128-row tile
    full); ``workspace`` from matmul_split_workspace."""
    lib = load()
    rows = W.shape[0]
    K = quant_K(FMT_Q4K, W.shape[1])
    M = X.shape[0]
    out = torch.empty((M, rows), dtype=torch.float32, device=W.device) if out is None else out
    _check("dq_matmul_q4k_split",
           lib.dq_matmul_q4k_split(_ptr(W), _ptr(X), _ptr(out), M, rows, K, _ptr(workspace), workspace.numel(),
                                   _stream()))
    return out


# ------------------------------------------------------------ attention


def attention_workspace(n_q: int, n_kv: int, device=None) -> torch.Tensor:
    lib = load()
    nbytes = lib.dq_attention_workspace_bytes(n_q, n_kv)
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")


def attention_decode(q: torch.Tensor, k_plane: torch.Tensor, v_plane: torch.Tensor, n_keys: int,
                     workspace: torch.Tensor | None = None, out=None):
    """q: fp32 [n_q, 128]; k/v planes: fp16 [n_kv, max_ctx, 128] -> fp32 [n_q, 128]."""
    lib = load()
    n_q, hd = q.shape
    n_kv, max_ctx, _ = k_plane.shape
    ws = attention_workspace(n_q, n_kv, q.device) if workspace is None else workspace
    out = torch.empty_like(q) if out is None else out
    st = lib.dq_attention_decode(_ptr(q), _ptr(k_plane), _ptr(v_plane), _ptr(out), n_q, n_kv, hd, max_ctx,
                                 n_keys, _ptr(ws), ws.numel(), _stream())
    _check("dq_attention_decode", st)
    return out


def attention_decode_static(q: torch.Tensor, k_plane: torch.Tensor, v_plane: torch.Tensor, n_keys: int, out=None):
    """As attention_decode, with the library's static scratch (no allocation by the library)."""
    lib = load()
    n_q, hd = q.shape
    n_kv, max_ctx, _ = k_plane.shape
    out = torch.empty_like(q) if out is None else out
    st = lib.dq_attention_decode_static(_ptr(q), _ptr(k_plane), _ptr(v_plane), _ptr(out), n_q, n_kv, hd, max_ctx,
                                        n_keys, _stream())
    _check("dq_attention_decode_static", st)
    return out


def rope_table(max_ctx: int, head_dim: int = 128, theta: float = 1.0e6, device=None) -> torch.Tensor:
    """fp32 [max_ctx, head_dim // 2, 2]: (cos, sin) of p / theta^(2i / head_dim)."""
    lib = load()
    t = torch.empty((max_ctx, head_dim // 2, 2), dtype=torch.float32, device=device or "cuda")
    _check("dq_rope_table", lib.dq_rope_table(_ptr(t), int(max_ctx), int(head_dim), float(theta), _stream()))
    return t


def attention_decode_rope(q: torch.Tensor, k_new: torch.Tensor, k_plane: torch.Tensor, v_plane: torch.Tensor,
                          q_norm: torch.Tensor, k_norm: torch.Tensor, rope: torch.Tensor, n_keys: int,
                          eps: float = 1e-6, workspace: torch.Tensor | None = None, out=None):
    """Qwen3 attention inputs: q fp32 [n_q, 128] and k_new fp32 [n_kv, 128] as projected are
    head-normalised and rotated to position n_keys - 1; k_plane row n_keys - 1 is written."""
    lib = load()
    n_q, hd = q.shape
    n_kv, max_ctx, _ = k_plane.shape
    ws = attention_workspace(n_q, n_kv, q.device) if workspace is None else workspace
    out = torch.empty_like(q) if out is None else out
    st = lib.dq_attention_decode_rope(_ptr(q), _ptr(k_new), _ptr(k_plane), _ptr(v_plane), _ptr(out), _ptr(q_norm),
                                      _ptr(k_norm), _ptr(rope), float(eps), n_q, n_kv, hd, max_ctx, int(n_keys),
                                      _ptr(ws), ws.numel(), _stream())
    _check("dq_attention_decode_rope", st)
    return out


# --------------------------------------------------------------- model


def _wrap_device_f32(ptr: int, numel: int) -> torch.Tensor:
    """A torch tensor over existing device memory (no copy, no ownership)."""
    class _CAI:
        __cuda_array_interface__ = {"shape": (numel,), "typestr": "<f4", "data": (ptr, False), "version": 3,
                                    "strides": None}
    return torch.as_tensor(_CAI(), device="cuda")


class _Desc(ctypes.Structure):
    _fields_ = [
        ("n_layers", I), ("hidden", I), ("ffn", I), ("n_q_heads", I), ("n_kv_heads", I), ("head_dim", I),
        ("vocab", I), ("max_ctx", I), ("eps", F),
        ("attn_norm", P), ("wqkv", P), ("wo", P), ("ffn_norm", P), ("wgate", P), ("wup", P), ("wdown", P),
        ("down_fmt", P), ("out_norm", P), ("wvocab", P), ("kv_cache", P), ("use_graph", I), ("flags", I),
        ("q_norm", P), ("k_norm", P), ("rope_theta", D),
    ]


MODEL_NO_PDL = 1
MODEL_FUSED = 2  # run the token as one persistent kernel where the shape allows


class Model:
    """A decode-step handle over device-resident weights.

    ``weights`` is a dict of torch CUDA tensors: per-layer lists ``attn_norm``,
    ``wqkv``, ``wo``, ``ffn_norm``, ``wgate``, ``wup``, ``wdown`` and the list
    ``down_fmt`` (ints), plus ``out_norm``, ``wvocab`` and ``kv_cache``
    (fp16/int16 [L, 2, n_kv, max_ctx, hd]).  The handle borrows them: keep
    them alive (this object holds references).  With the Qwen3 attention
    inputs, ``weights`` also holds per-layer lists ``q_norm`` and ``k_norm``
    (fp32 [hd]) and ``rope_theta`` is the rotary base (> 1).
    """

    def __init__(self, n_layers, hidden, ffn, n_q_heads, n_kv_heads, head_dim, vocab, max_ctx, eps, weights,
                 use_graph: bool = True, flags: int = 0, rope_theta: float = 0.0):
        lib = load()
        self.weights = weights
        self.hidden, self.vocab, self.max_ctx = hidden, vocab, max_ctx
        self._keep = []

        def arr(tensors):
            a = (ctypes.c_void_p * n_layers)(*[t.data_ptr() for t in tensors])
            self._keep.append(a)
            return ctypes.cast(a, ctypes.c_void_p)

        fmts = (ctypes.c_int * n_layers)(*[int(f) for f in weights["down_fmt"]])
        self._keep.append(fmts)
        d = _Desc(n_layers, hidden, ffn, n_q_heads, n_kv_heads, head_dim, vocab, max_ctx, eps,
                  arr(weights["attn_norm"]), arr(weights["wqkv"]), arr(weights["wo"]), arr(weights["ffn_norm"]),
                  arr(weights["wgate"]), arr(weights["wup"]), arr(weights["wdown"]),
                  ctypes.cast(fmts, ctypes.c_void_p), weights["out_norm"].data_ptr(), weights["wvocab"].data_ptr(),
                  weights["kv_cache"].data_ptr(), 1 if use_graph else 0, int(flags))
        if weights.get("q_norm"):
            d.q_norm = arr(weights["q_norm"])
            d.k_norm = arr(weights["k_norm"])
            d.rope_theta = float(rope_theta)
        h = ctypes.c_void_p()
        _check("dq_model_create", lib.dq_model_create(ctypes.byref(d), ctypes.byref(h)))
        self._h = h
        self.launches_per_step = lib.dq_model_launches_per_step(h)
        self.fused = bool(lib.dq_model_fused(h))

    def step(self, x_in: torch.Tensor, pos: int, logits: torch.Tensor | None = None) -> torch.Tensor:
        lib = load()
        logits = torch.empty(self.vocab, dtype=torch.float32, device=x_in.device) if logits is None else logits
        _check("dq_decode_step", lib.dq_decode_step(self._h, _ptr(x_in), int(pos), _ptr(logits), _stream()))
        return logits

    def step_raw(self, x_ptr: int, pos: int, logits_ptr: int, stream_handle: int):
        """Pointer-level call (no tensor checks), for timing loops."""
        _check("dq_decode_step", _lib.dq_decode_step(self._h, ctypes.c_void_p(x_ptr), int(pos),
                                                     ctypes.c_void_p(logits_ptr), ctypes.c_void_p(stream_handle)))

    def step_host(self, x_host: torch.Tensor, pos: int, logits_host: torch.Tensor) -> torch.Tensor:
        """One token from host memory (fp32 CPU tensors, page-locked for asynchronous
        copies): the C call copies x in, runs the token, copies the logits out and
        waits for the stream."""
        if x_host.device.type != "cpu" or logits_host.device.type != "cpu":
            raise ValueError("step_host takes CPU tensors")
        if not (x_host.is_contiguous() and logits_host.is_contiguous()):
            raise ValueError("tensors must be contiguous")
        if x_host.dtype != torch.float32 or logits_host.dtype != torch.float32:
            raise ValueError("step_host takes fp32 tensors")
        if x_host.numel() < self.hidden or logits_host.numel() < self.vocab:
            raise ValueError("step_host: x needs hidden and logits vocab elements")
        _check("dq_decode_step_host", _lib.dq_decode_step_host(self._h, ctypes.c_void_p(x_host.data_ptr()), int(pos),
                                                               ctypes.c_void_p(logits_host.data_ptr()), _stream()))
        return logits_host

    KERNEL_KINDS = ("qkv", "attention", "o_proj", "gate_up", "down", "vocab")

    def enqueue_kernel(self, layer: int, kind: int, stream_handle: int | None = None):
        """Launch one of the token's kernels alone (diagnostics / per-kernel timing)."""
        s = ctypes.c_void_p(stream_handle) if stream_handle is not None else _stream()
        _check("dq_model_enqueue_kernel", _lib.dq_model_enqueue_kernel(self._h, int(layer), int(kind), s))

    def buffer(self, which: int, numel: int) -> torch.Tensor:
        """A torch view (fp32) of one model activation buffer: 0 x, 1 q, 2 attn, 3 act."""
        p = ctypes.c_void_p()
        _check("dq_model_buffer", _lib.dq_model_buffer(self._h, int(which), ctypes.byref(p)))
        return _wrap_device_f32(p.value, numel)

    def close(self):
        if getattr(self, "_h", None):
            load().dq_model_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
