"""Byte and roofline arithmetic for the decode step.

Everything here is bookkeeping on layouts and measured rates, used to report
bandwidth; none of it runs the method.  The relations follow "The roofline
holds on a second GPU" (research.arkey.ai), section "The Math": one token reads
every weight once, so tokens/s <= BW / B, and the memory/compute crossover is
M* = (w / 16) * (R / BW) for w bits per weight and an arithmetic rate R that
counts two operations (a multiply and an add) per weight per token.
"""
from __future__ import annotations

Q4K_BLOCK_BYTES = 144
Q6K_BLOCK_BYTES = 210
WEIGHTS_PER_BLOCK = 256
FMT_BF16, FMT_Q4K, FMT_Q6K = 0, 1, 2


def bits_per_weight(fmt: int) -> float:
    if fmt == FMT_BF16:
        return 16.0
    return 8.0 * (Q4K_BLOCK_BYTES if fmt == FMT_Q4K else Q6K_BLOCK_BYTES) / WEIGHTS_PER_BLOCK


def matrix_bytes(fmt: int, rows: int, K: int) -> int:
    if fmt == FMT_BF16:
        return 2 * rows * K
    assert K % WEIGHTS_PER_BLOCK == 0
    bpb = Q4K_BLOCK_BYTES if fmt == FMT_Q4K else Q6K_BLOCK_BYTES
    return rows * (K // WEIGHTS_PER_BLOCK) * bpb


def layer_tensors(hidden: int, ffn: int, n_q: int, n_kv: int, hd: int, down_fmt: int):
    """(role, fmt, rows, K) of one decoder layer's weight tables."""
    return [
        ("wqkv", FMT_Q4K, (n_q + 2 * n_kv) * hd, hidden),
        ("wo", FMT_Q4K, hidden, n_q * hd),
        ("wgate", FMT_Q4K, ffn, hidden),
        ("wup", FMT_Q4K, ffn, hidden),
        ("wdown", down_fmt, hidden, ffn),
    ]


def model_weight_bytes(n_layers: int, hidden: int, ffn: int, n_q: int, n_kv: int, hd: int,
                       vocab: int, down_fmts=None) -> int:
    """Bytes of every weight table, read once per token (the roofline's B)."""
    if down_fmts is None:
        down_fmts = [FMT_Q6K if l % 2 == 1 else FMT_Q4K for l in range(n_layers)]
    total = 0
    for l in range(n_layers):
        for _, fmt, rows, K in layer_tensors(hidden, ffn, n_q, n_kv, hd, down_fmts[l]):
            total += matrix_bytes(fmt, rows, K)
    return total + matrix_bytes(FMT_Q6K, vocab, hidden)


def norm_bytes(n_layers: int, hidden: int) -> int:
    """fp32 gamma vectors: two per layer plus the final norm."""
    return 4 * hidden * (2 * n_layers + 1)


def kv_read_bytes(n_layers: int, n_kv: int, hd: int, n_keys: int, elem_bytes: int = 2) -> int:
    """K and V bytes read by one token's attention over n_keys positions."""
    return n_layers * 2 * n_kv * hd * n_keys * elem_bytes


def token_bytes(n_layers: int, hidden: int, ffn: int, n_q: int, n_kv: int, hd: int, vocab: int,
                ctx: int = 0) -> int:
    """Algorithmic bytes of one decode token at `ctx` cached positions:
    weights + norm gammas + the K/V already in the cache (the new key and value
    are written and read once more; activations are negligible and not counted)."""
    return (model_weight_bytes(n_layers, hidden, ffn, n_q, n_kv, hd, vocab)
            + norm_bytes(n_layers, hidden) + kv_read_bytes(n_layers, n_kv, hd, ctx))


def tokens_per_s_limit(bw_bytes_per_s: float, bytes_per_token: float) -> float:
    return bw_bytes_per_s / bytes_per_token


def floor_seconds(nbytes: float, bw_bytes_per_s: float) -> float:
    return nbytes / bw_bytes_per_s


def sums_per_byte(bits_per_w: float, m_tokens: int = 1) -> float:
    """Two operations (multiply, add) per weight per token over w/8 bytes."""
    return 2.0 * m_tokens / (bits_per_w / 8.0)


def m_star(bits_per_w: float, rate_ops_per_s: float, bw_bytes_per_s: float) -> float:
    """Crossover token count: (w / 16) * (R / BW)."""
    return bits_per_w / 16.0 * rate_ops_per_s / bw_bytes_per_s


def bytes_in_flight(bw_bytes_per_s: float, latency_s: float) -> float:
    """Little's law: what must be outstanding to keep the memory busy."""
    return bw_bytes_per_s * latency_s


QWEN3_8B_SHAPE = dict(n_layers=36, hidden=4096, ffn=12288, n_q=32, n_kv=8, hd=128, vocab=151936)
