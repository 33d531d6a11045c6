"""Test-side error model of the decode step's activation format (not the oracle).

The CUDA path feeds every quantised GEMV a fixed-point copy of its input: per
32-element group, x ~= s * xi with |xi| <= 16383 (15 bits), or, for the q|k|v
projection (and the O projection of the separate kernels), x ~= s * (xi + xl / 2^15)
(about 30 bits).  This module
re-applies exactly that rounding to GEMV inputs inside a float64 decode built
from the oracle's dequantised weights and attention, so a test can tell how
much of a decode's deviation from the exact oracle the documented format
explains on a given (possibly ill-conditioned) random model.
"""
import numpy as np

XQ_MAX = 16383.0


def group_round(v, planes: int):
    v = np.asarray(v, np.float64).reshape(-1, 32)
    amax = np.abs(v).max(axis=1, keepdims=True)
    s = amax / XQ_MAX
    safe = np.where(s > 0, s, 1.0)
    t = np.where(s > 0, v / safe, 0.0)
    xi = np.rint(t)
    out = xi
    if planes == 2:
        out = xi + np.rint((t - xi) * 32768.0) / 32768.0
    return (out * s).reshape(-1)


def _rms(x, g, eps):
    x = np.asarray(x, np.float64)
    return x / np.sqrt((x * x).mean() + eps) * np.asarray(g, np.float64)


def dequantised(orc, m):
    def deq(W, fmt, rows, K):
        return (orc.dequant_q4k(W) if fmt == 1 else orc.dequant_q6k(W)).reshape(rows, K)

    qdim = m.n_q_heads * m.head_dim
    return {
        "qkv": [deq(w, 1, m.qkv_rows, m.hidden) for w in m.wqkv],
        "o": [deq(w, 1, m.hidden, qdim) for w in m.wo],
        "gate": [deq(w, 1, m.ffn, m.hidden) for w in m.wgate],
        "up": [deq(w, 1, m.ffn, m.hidden) for w in m.wup],
        "down": [deq(w, f, m.hidden, m.ffn) for w, f in zip(m.wdown, m.down_fmt)],
        "vocab": deq(m.wvocab, 2, m.vocab, m.hidden),
    }


def decode(orc, m, Wd, x_in, pos, kv, o_planes: int = 2):
    """One token with the CUDA path's activation rounding; updates kv (fp16 bits) in place.
    ``o_planes``: the O projection's activation planes (the fused token kernel uses 1)."""
    hd, nq, nkv = m.head_dim, m.n_q_heads, m.n_kv_heads
    qdim, kvdim = nq * hd, nkv * hd
    kvf = kv.view(np.float16)
    x = np.asarray(x_in, np.float64)
    for l in range(m.n_layers):
        qkv = Wd["qkv"][l] @ group_round(_rms(x, m.attn_norm[l], m.eps), 2)
        if getattr(m, "q_norm", None):  # Qwen3 attention inputs, exact (fp64) as in the oracle
            for h in range(nq):
                qkv[h * hd:(h + 1) * hd] = orc.rope(orc.head_rmsnorm(qkv[h * hd:(h + 1) * hd], m.q_norm[l], m.eps),
                                                    pos, m.rope_theta)
            for g in range(nkv):
                sl = slice(qdim + g * hd, qdim + (g + 1) * hd)
                qkv[sl] = orc.rope(orc.head_rmsnorm(qkv[sl], m.k_norm[l], m.eps), pos, m.rope_theta)
        kvf[l, 0, :, pos, :] = qkv[qdim:qdim + kvdim].reshape(nkv, hd).astype(np.float16)
        kvf[l, 1, :, pos, :] = qkv[qdim + kvdim:].reshape(nkv, hd).astype(np.float16)
        att = orc.attention(qkv[:qdim].reshape(nq, hd), kv[l, 0], kv[l, 1], pos + 1).reshape(-1)
        x = x + Wd["o"][l] @ group_round(att, o_planes)
        h = group_round(_rms(x, m.ffn_norm[l], m.eps), 1)
        g, u = Wd["gate"][l] @ h, Wd["up"][l] @ h
        x = x + Wd["down"][l] @ group_round(g / (1.0 + np.exp(-g)) * u, 1)
    return Wd["vocab"] @ group_round(_rms(x, m.out_norm, m.eps), 1)
