"""The byte/roofline ledger against the numbers the pages print (tests/golden/pages_ledger.txt)."""
import os

import pytest

from quantised_gemv_norm_gb300 import ledger as L

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_ledger.txt")
S = L.QWEN3_8B_SHAPE


def _golden():
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, value, tol, _src = [f.strip() for f in line.split("|", 3)]
        out[name] = (float(value), float(tol))
    return out


def _computed():
    B_pages = 4.68e9  # the pages' own per-token bytes, used where they divide by it
    vocab = L.matrix_bytes(L.FMT_Q6K, S["vocab"], S["hidden"])
    kv512 = L.kv_read_bytes(S["n_layers"], S["n_kv"], S["hd"], 512)
    return {
        "q4k_bits_per_weight": L.bits_per_weight(L.FMT_Q4K),
        "q6k_bits_per_weight": L.bits_per_weight(L.FMT_Q6K),
        "q4k_block_bytes": L.Q4K_BLOCK_BYTES,
        "q6k_block_bytes": L.Q6K_BLOCK_BYTES,
        "vocab_table_MB": vocab / 1e6,
        "vocab_floor_us_1700GBps": L.floor_seconds(vocab, 1700e9) * 1e6,
        "kv_512_MB": kv512 / 1e6,
        "token_GB": L.model_weight_bytes(**S) / 1e9,
        "sums_per_byte_4p5": L.sums_per_byte(4.5),
        "m4_mstar_numerator": L.m_star(4.5, 3.78e12, 1.0) / 1e9,  # M* * BW with BW in GB/s
        "m3_limit_tok_s": L.tokens_per_s_limit(89.9e9, B_pages),
        "m3_limit_512_tok_s": L.tokens_per_s_limit(89.9e9, B_pages + kv512),
        "rtx5090_floor_ms": L.floor_seconds(B_pages, 1700e9) * 1e3,
        "m3_floor_ms": L.floor_seconds(B_pages, 89.9e9) * 1e3,
        "rtx5090_sums_per_byte": 255.4e12 / 1700e9,
        "m3_sums_per_byte": 3.152e12 / 89.9e9,
        "prefill_sums_per_byte": L.sums_per_byte(4.5, 512),
        "little_5090_MB_per_us": L.bytes_in_flight(1700e9, 1e-6) / 1e6,
        "little_m3_KB_per_us": L.bytes_in_flight(89.9e9, 1e-6) / 1e3,
        "tinygrad_ms_per_token": 1e3 / 237.8,
    }


@pytest.mark.parametrize("name", sorted(_golden()))
def test_ledger_matches_pages(name):
    value, tol = _golden()[name]
    got = _computed()[name]
    assert abs(got - value) <= max(tol * abs(value), 1e-12), (name, got, value)


def test_exact_layout_bytes():
    # Our exact per-token weight bytes (O projection included); 0.6% under the pages' 4.68 GB.
    assert L.model_weight_bytes(**S) == 4_651_069_440
    assert L.kv_read_bytes(36, 8, 128, 512) == 75_497_472
    assert L.matrix_bytes(L.FMT_Q4K, 12288, 4096) == 28_311_552
    assert L.matrix_bytes(L.FMT_Q6K, 4096, 12288) == 41_287_680
    assert L.matrix_bytes(L.FMT_BF16, 151936, 4096) == 1_244_659_712
