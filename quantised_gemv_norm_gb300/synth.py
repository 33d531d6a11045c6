"""Seeded synthetic inputs for the decode hot path.

This module only draws random numbers and places them in the storage formats:
it holds none of the method's arithmetic (no dequantisation, no products, no
norms).  It is the one module that both the CUDA path's tests/bench and the CPU
oracle's tests are fed from; neither side imports the other.

Recipes (all numpy PCG64 ``default_rng``; every tensor has its own stream keyed
by (seed, layer, role) so tensors can be drawn independently and reproducibly):

* norm rows: x ~ N(0, 1), gamma ~ N(1, 0.1), beta ~ N(0, 0.1), float32;
* bf16 matrices: W ~ N(0, 0.02), vectors ~ N(0, 1), drawn in float32 and rounded
  to nearest-even bfloat16 (torch's conversion);
* Q4_K blocks: every bit uniform, then the two binary16 fields forced into a
  binade: d in [2^-13, 2^-12), dmin in [2^-10, 2^-9) (mantissa bits stay
  uniform).  Scales, mins and codes are therefore uniform over their widths;
* Q6_K blocks: every bit uniform, d forced into [2^-14, 2^-13);
* activations x ~ N(0, 1) float32; the fp16 KV cache ~ N(0, 1) for positions
  already filled, zero elsewhere.

With those binades every dequantised weight is exactly representable in fp32
(see the block-format notes in the library header), so dequantisation can be
compared bit for bit.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

Q4K_BLOCK_BYTES = 144
Q6K_BLOCK_BYTES = 210
Q2K_BLOCK_BYTES = 84
FMT_BF16, FMT_Q4K, FMT_Q6K, FMT_Q2K = 0, 1, 2, 3

# Role ids keep every tensor on its own random stream.
_ROLES = {"x": 1, "gamma": 2, "beta": 3, "w": 4, "wqkv": 10, "wo": 11, "wgate": 12, "wup": 13,
          "wdown": 14, "attn_norm": 15, "ffn_norm": 16, "out_norm": 17, "wvocab": 18, "kv": 19,
          "xin": 20, "q_norm": 21, "k_norm": 22}


def rng_for(seed: int, *key: int) -> np.random.Generator:
    return np.random.default_rng([int(seed)] + [int(k) for k in key])


def _role(name: str) -> int:
    return _ROLES[name]


def random_bytes(rng: np.random.Generator, n: int) -> np.ndarray:
    words = (n + 7) // 8
    u = rng.integers(0, np.iinfo(np.uint64).max, size=words, dtype=np.uint64, endpoint=True)
    return u.view(np.uint8)[:n].copy() if words * 8 != n else u.view(np.uint8)


def normal_f32(rng: np.random.Generator, shape, mean: float = 0.0, std: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    return x


def to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even (torch)."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def norm_inputs(seed: int, rows: int, n: int):
    """(x, gamma, beta) for the norm configs."""
    x = normal_f32(rng_for(seed, _role("x")), (rows, n))
    gamma = normal_f32(rng_for(seed, _role("gamma")), (n,), 1.0, 0.1)
    beta = normal_f32(rng_for(seed, _role("beta")), (n,), 0.0, 0.1)
    return x, gamma, beta


def bf16_gemv_inputs(seed: int, rows: int, K: int):
    """(W bits [rows, K], x bits [K]) with W ~ N(0, 0.02), x ~ N(0, 1)."""
    W = to_bf16_bits(normal_f32(rng_for(seed, _role("w")), (rows, K), 0.0, 0.02))
    x = to_bf16_bits(normal_f32(rng_for(seed, _role("x")), (K,)))
    return W, x


def q4k_blocks(rng: np.random.Generator, nblocks: int) -> np.ndarray:
    b = random_bytes(rng, nblocks * Q4K_BLOCK_BYTES).reshape(nblocks, Q4K_BLOCK_BYTES)
    # d: binary16 exponent field 2 (sign 0) -> [2^-13, 2^-12); byte 1 = s|eeeee|mm
    b[:, 1] = (b[:, 1] & 0x03) | (2 << 2)
    # dmin: exponent field 5 -> [2^-10, 2^-9)
    b[:, 3] = (b[:, 3] & 0x03) | (5 << 2)
    return b


def q6k_blocks(rng: np.random.Generator, nblocks: int) -> np.ndarray:
    b = random_bytes(rng, nblocks * Q6K_BLOCK_BYTES).reshape(nblocks, Q6K_BLOCK_BYTES)
    # d at bytes 208..209: exponent field 1 -> [2^-14, 2^-13)
    b[:, 209] = (b[:, 209] & 0x03) | (1 << 2)
    return b


def q2k_blocks(rng: np.random.Generator, nblocks: int) -> np.ndarray:
    # d and dmin in Q4_K's binades: d sc q (< 2^17 units of 2^-23) minus dmin m
    # (< 2^18 units) is an fp32 number
    b = random_bytes(rng, nblocks * Q2K_BLOCK_BYTES).reshape(nblocks, Q2K_BLOCK_BYTES)
    b[:, 1] = (b[:, 1] & 0x03) | (2 << 2)
    b[:, 3] = (b[:, 3] & 0x03) | (5 << 2)
    return b


def quant_matrix(seed: int, fmt: int, rows: int, K: int, *key: int) -> np.ndarray:
    """A [rows, K] matrix in Q4_K, Q6_K or Q2_K blocks, as uint8 [rows, row_bytes]."""
    assert K % 256 == 0
    rng = rng_for(seed, _role("w"), fmt, rows, K, *key)
    nb = rows * (K // 256)
    if fmt == FMT_Q4K:
        return q4k_blocks(rng, nb).reshape(rows, -1)
    if fmt == FMT_Q6K:
        return q6k_blocks(rng, nb).reshape(rows, -1)
    if fmt == FMT_Q2K:
        return q2k_blocks(rng, nb).reshape(rows, -1)
    raise ValueError(fmt)


def activation(seed: int, K: int, *key: int) -> np.ndarray:
    return normal_f32(rng_for(seed, _role("x"), K, *key), (K,))


def row_bytes(fmt: int, K: int) -> int:
    if fmt == FMT_BF16:
        return 2 * K
    return (K // 256) * {FMT_Q4K: Q4K_BLOCK_BYTES, FMT_Q6K: Q6K_BLOCK_BYTES, FMT_Q2K: Q2K_BLOCK_BYTES}[fmt]


# ----------------------------------------------------------------- models

QWEN3_8B = dict(n_layers=36, hidden=4096, ffn=12288, n_q_heads=32, n_kv_heads=8, head_dim=128,
                vocab=151936)


@dataclass
class SyntheticModel:
    """Random-init weights of a Qwen3-8B-shaped decoder (host numpy arrays).

    wqkv rows are q (n_q*hd) | k (n_kv*hd) | v (n_kv*hd); all projections are
    Q4_K except the down projection (Q6_K in odd layers, Q4_K in even layers)
    and the vocabulary table (Q6_K).
    """
    n_layers: int
    hidden: int
    ffn: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    vocab: int
    max_ctx: int
    eps: float = 1e-6
    attn_norm: list = field(default_factory=list)
    wqkv: list = field(default_factory=list)
    wo: list = field(default_factory=list)
    ffn_norm: list = field(default_factory=list)
    wgate: list = field(default_factory=list)
    wup: list = field(default_factory=list)
    wdown: list = field(default_factory=list)
    down_fmt: list = field(default_factory=list)
    out_norm: np.ndarray = None
    wvocab: np.ndarray = None
    # Qwen3 attention inputs (empty: plain attention on the projections)
    q_norm: list = field(default_factory=list)
    k_norm: list = field(default_factory=list)
    rope_theta: float = 0.0

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim

    def weight_bytes(self) -> int:
        n = 0
        for l in range(self.n_layers):
            n += self.wqkv[l].nbytes + self.wo[l].nbytes + self.wgate[l].nbytes
            n += self.wup[l].nbytes + self.wdown[l].nbytes
        return n + self.wvocab.nbytes


QWEN3_ROPE_THETA = 1.0e6


def make_model(seed: int, n_layers: int, hidden: int, ffn: int, n_q_heads: int, n_kv_heads: int,
               head_dim: int, vocab: int, max_ctx: int, eps: float = 1e-6,
               qwen3_attention: bool = False) -> SyntheticModel:
    """``qwen3_attention`` adds per-layer q/k head-norm weights ~ N(1, 0.1) and the
    rotary base 1e6 (Qwen3's); the other tensors do not depend on it."""
    m = SyntheticModel(n_layers, hidden, ffn, n_q_heads, n_kv_heads, head_dim, vocab, max_ctx, eps)
    qdim = n_q_heads * head_dim
    for l in range(n_layers):
        m.attn_norm.append(normal_f32(rng_for(seed, _role("attn_norm"), l), (hidden,), 1.0, 0.1))
        m.ffn_norm.append(normal_f32(rng_for(seed, _role("ffn_norm"), l), (hidden,), 1.0, 0.1))
        m.wqkv.append(q4k_blocks(rng_for(seed, _role("wqkv"), l), m.qkv_rows * hidden // 256).reshape(m.qkv_rows, -1))
        m.wo.append(q4k_blocks(rng_for(seed, _role("wo"), l), hidden * qdim // 256).reshape(hidden, -1))
        m.wgate.append(q4k_blocks(rng_for(seed, _role("wgate"), l), ffn * hidden // 256).reshape(ffn, -1))
        m.wup.append(q4k_blocks(rng_for(seed, _role("wup"), l), ffn * hidden // 256).reshape(ffn, -1))
        fmt = FMT_Q6K if l % 2 == 1 else FMT_Q4K
        m.down_fmt.append(fmt)
        gen = q6k_blocks if fmt == FMT_Q6K else q4k_blocks
        m.wdown.append(gen(rng_for(seed, _role("wdown"), l), hidden * ffn // 256).reshape(hidden, -1))
    if qwen3_attention:
        for l in range(n_layers):
            m.q_norm.append(normal_f32(rng_for(seed, _role("q_norm"), l), (head_dim,), 1.0, 0.1))
            m.k_norm.append(normal_f32(rng_for(seed, _role("k_norm"), l), (head_dim,), 1.0, 0.1))
        m.rope_theta = QWEN3_ROPE_THETA
    m.out_norm = normal_f32(rng_for(seed, _role("out_norm")), (hidden,), 1.0, 0.1)
    m.wvocab = q6k_blocks(rng_for(seed, _role("wvocab")), vocab * hidden // 256).reshape(vocab, -1)
    return m


def make_kv_cache(seed: int, m: SyntheticModel, filled: int) -> np.ndarray:
    """fp16 bits [L, 2, n_kv, max_ctx, hd]; positions < filled ~ N(0, 1), rest 0."""
    kv = np.zeros((m.n_layers, 2, m.n_kv_heads, m.max_ctx, m.head_dim), np.uint16)
    if filled > 0:
        rng = rng_for(seed, _role("kv"))
        vals = rng.standard_normal(size=(m.n_layers, 2, m.n_kv_heads, filled, m.head_dim),
                                   dtype=np.float32).astype(np.float16)
        kv[:, :, :, :filled, :] = vals.view(np.uint16)
    return kv


def decode_input(seed: int, hidden: int, token: int = 0) -> np.ndarray:
    return normal_f32(rng_for(seed, _role("xin"), token), (hidden,))
