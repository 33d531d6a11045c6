"""Mutation check of the oracle's pins.  Each entry below plants one plausible
slip in a copy of oracle/dq_oracle.c -- a dropped term, a wrong sign, index, bit
position, operand or rounding rule -- builds that copy, and runs the pin suite
(tests/test_oracle_pins.py) against it: the suite must fail.  The oracle itself
is never modified.  A control build of the unchanged source must pass, so each
failure is the planted slip being seen.  No GPU needed."""
import concurrent.futures
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "dq_oracle.c")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# name -> (text of the oracle, its slipped replacement); each text occurs once
MUTANTS = {
    # number formats
    "half_subnormal_scale": ("v = ldexp((double)m, -24);", "v = ldexp((double)m, -25);"),
    "half_exponent_bias": ("v = ldexp((double)(1024 + m), e - 25);", "v = ldexp((double)(1024 + m), e - 24);"),
    "half_ties_away_from_zero": ("double n = nearbyint(ldexp(a, 10 - E));", "double n = round(ldexp(a, 10 - E));"),
    "bf16_low_half": ("uint32_t u = (uint32_t)b << 16;", "uint32_t u = (uint32_t)b;"),
    "half_subnormal_threshold": ("if (E < -14)", "if (E < -15)"),
    "half_sign_dropped": ("return sign ? -v : v;", "return v;"),
    "fields_big_endian": ("return (uint16_t)(p[0] | (p[1] << 8));", "return (uint16_t)(p[1] | (p[0] << 8));"),
    # Q4_K
    "q4k_min_sign": ("w[n] = d * sc[j] * q[n] - dmin * m[j];", "w[n] = d * sc[j] * q[n] + dmin * m[j];"),
    "q4k_nibbles_swapped": ("q[32 * j + i] = byte & 15;\n            q[32 * j + 16 + i] = byte >> 4;",
                            "q[32 * j + i] = byte >> 4;\n            q[32 * j + 16 + i] = byte & 15;"),
    "q4k_scales_interleaved": ("sc[j] = field6(blk + 4, 6 * j);\n        m[j] = field6(blk + 4, 48 + 6 * j);",
                               "sc[j] = field6(blk + 4, 12 * j);\n        m[j] = field6(blk + 4, 12 * j + 6);"),
    "q4k_field_msb_first": ("v |= bit_at(bits, first_bit + k) << k;", "v |= bit_at(bits, first_bit + k) << (5 - k);"),
    "q4k_scale_of_wrong_subblock": ("int j = n / 32;\n        w[n]", "int j = n / 32 % 7;\n        w[n]"),
    "q4k_d_and_dmin_swapped": ("*d = oracle_half_to_double(rd16(blk + 0));\n    *dmin = oracle_half_to_double(rd16(blk + 2));\n"
                               "    for (int j = 0; j < 8; j++) {",
                               "*d = oracle_half_to_double(rd16(blk + 2));\n    *dmin = oracle_half_to_double(rd16(blk + 0));\n"
                               "    for (int j = 0; j < 8; j++) {"),
    # Q6_K
    "q4k_packer_nibbles_swapped": ("(uint8_t)((q[32 * j + i] & 15) | ((q[32 * j + 16 + i] & 15) << 4));",
                                   "(uint8_t)((q[32 * j + 16 + i] & 15) | ((q[32 * j + i] & 15) << 4));"),
    "q6k_centre": ("w[n] = d * sc[n / 16] * (q[n] - 32);", "w[n] = d * sc[n / 16] * (q[n] - 31);"),
    "q6k_scale_index": ("w[n] = d * sc[n / 16] * (q[n] - 32);", "w[n] = d * sc[n % 16] * (q[n] - 32);"),
    "q6k_high_bits_order": ("q[32 * g + 16 * h + 4 * t + e] |= hi << 4;", "q[32 * g + 16 * h + 4 * e + t] |= hi << 4;"),
    "q6k_scale_unsigned": ("sc[s] = (int)(int8_t)blk[192 + s];", "sc[s] = (int)blk[192 + s];"),
    "q6k_d_offset": ("*d = oracle_half_to_double(rd16(blk + 208));", "*d = oracle_half_to_double(rd16(blk + 192));"),
    # Q2_K
    "q2k_code_position": ("q[16 * j + 4 * k + b] = (blk[20 + 4 * j + b] >> (2 * k)) & 3;",
                          "q[16 * j + 4 * b + k] = (blk[20 + 4 * j + b] >> (2 * k)) & 3;"),
    "q2k_scale_min_swapped": ("sc[j] = blk[4 + j] & 15;\n        m[j] = blk[4 + j] >> 4;",
                              "sc[j] = blk[4 + j] >> 4;\n        m[j] = blk[4 + j] & 15;"),
    "q2k_min_dropped": ("w[n] = d * sc[n / 16] * q[n] - dmin * m[n / 16];", "w[n] = d * sc[n / 16] * q[n];"),
    "q2k_d_and_dmin_swapped": ("*d = oracle_half_to_double(rd16(blk + 0));\n    *dmin = oracle_half_to_double(rd16(blk + 2));\n"
                               "    for (int j = 0; j < 16; j++) {",
                               "*d = oracle_half_to_double(rd16(blk + 2));\n    *dmin = oracle_half_to_double(rd16(blk + 0));\n"
                               "    for (int j = 0; j < 16; j++) {"),
    # GEMV and the M-sweep product
    "gemv_block_offset_dropped": ("acc += w[n] * x[256 * b + n];", "acc += w[n] * x[n];"),
    "gemv_last_block_dropped": ("for (int b = 0; b < K / 256; b++) {", "for (int b = 0; b < K / 256 - 1; b++) {"),
    "gemv_bf16_activation_as_fp16": ("xd[k] = oracle_bf16_to_double(x[k]);", "xd[k] = oracle_half_to_double(x[k]);"),
    "gemv_bf16_transposed": ("acc += oracle_bf16_to_double(rd16(row + 2 * (size_t)k)) * x[k];",
                             "acc += oracle_bf16_to_double(rd16(W + 2 * ((size_t)k * rows + r))) * x[k];"),
    "matmul_tokens_transposed": ("xd[k] = X[(size_t)m * K + k];", "xd[k] = X[(size_t)k * M + m];"),
    # norms
    "rmsnorm_eps_outside_root": ("double inv = 1.0 / sqrt(ss / n + eps);", "double inv = 1.0 / (sqrt(ss / n) + eps);"),
    "rmsnorm_sum_not_mean": ("double inv = 1.0 / sqrt(ss / n + eps);", "double inv = 1.0 / sqrt(ss + eps);"),
    "rmsnorm_gamma_dropped": ("y[i] = x[i] * inv * (double)gamma[i];", "y[i] = x[i] * inv;"),
    "rmsnorm_eps_dropped": ("double inv = 1.0 / sqrt(ss / n + eps);", "double inv = 1.0 / sqrt(ss / n);"),
    "layernorm_eps_dropped": ("double inv = 1.0 / sqrt(v / n + eps);", "double inv = 1.0 / sqrt(v / n);"),
    "layernorm_sample_variance": ("double inv = 1.0 / sqrt(v / n + eps);", "double inv = 1.0 / sqrt(v / (n - 1) + eps);"),
    "layernorm_uncentred_moment": ("v += (xr[i] - mean) * (xr[i] - mean);", "v += xr[i] * xr[i];"),
    "layernorm_beta_dropped": ("* (double)gamma[i] + (double)beta[i];", "* (double)gamma[i];"),
    "layernorm_gamma_dropped": ("inv * (double)gamma[i] + (double)beta[i];", "inv + (double)beta[i];"),
    # attention
    "attention_scale_by_hd": ("double scale = 1.0 / sqrt((double)hd);", "double scale = 1.0 / (double)hd;"),
    "attention_heads_interleaved": ("int g = h / group;", "int g = h % n_kv;"),
    "attention_not_normalised": ("out[h * hd + dd] = o / l;", "out[h * hd + dd] = o;"),
    "attention_query_of_kv_head": ("dot += q[h * hd + dd]", "dot += q[g * hd + dd]"),
    "attention_values_from_key_plane": ("o += s[j] * oracle_half_to_double(vc[",
                                        "o += s[j] * oracle_half_to_double(kc["),
    "silu_sign": ("return z / (1.0 + exp(-z));", "return z / (1.0 + exp(z));"),
    "silu_is_sigmoid": ("return z / (1.0 + exp(-z));", "return 1.0 / (1.0 + exp(-z));"),
    # Qwen3 attention inputs
    "head_norm_weight_dropped": ("v[i] = v[i] * r * (double)w[i];", "v[i] = v[i] * r;"),
    "head_norm_eps_outside_root": ("double r = 1.0 / sqrt(ss / hd + eps);", "double r = 1.0 / (sqrt(ss / hd) + eps);"),
    "head_norm_divisor": ("double r = 1.0 / sqrt(ss / hd + eps);", "double r = 1.0 / sqrt(ss / (hd - 1) + eps);"),
    "rope_position_off_by_one": ("double ang = (double)pos * pow(", "double ang = (double)(pos + 1) * pow("),
    "rope_rotation_sign": ("v[i] = a * c - b * sn;\n        v[i + half] = b * c + a * sn;",
                           "v[i] = a * c + b * sn;\n        v[i + half] = b * c - a * sn;"),
    "rope_frequency": ("pow(theta, -2.0 * i / hd)", "pow(theta, -1.0 * i / hd)"),
    "rope_adjacent_pairs": ("double a = v[i], b = v[i + half];\n        v[i] = a * c - b * sn;\n"
                            "        v[i + half] = b * c + a * sn;",
                            "double a = v[2 * i], b = v[2 * i + 1];\n        v[2 * i] = a * c - b * sn;\n"
                            "        v[2 * i + 1] = b * c + a * sn;"),
    # decode step
    "decode_k_and_v_swapped": ("kc[at] = oracle_double_to_half(qkv[qdim + kvh * hd + dd]);\n"
                               "                vc[at] = oracle_double_to_half(qkv[qdim + kvdim + kvh * hd + dd]);",
                               "kc[at] = oracle_double_to_half(qkv[qdim + kvdim + kvh * hd + dd]);\n"
                               "                vc[at] = oracle_double_to_half(qkv[qdim + kvh * hd + dd]);"),
    "decode_current_key_excluded": ("hd, mdl->max_ctx, pos + 1);", "hd, mdl->max_ctx, pos > 0 ? pos : 1);"),
    "decode_attention_residual_dropped": ("att, y, H, qdim);\n        for (int i = 0; i < H; i++)\n"
                                          "            x[i] += y[i];",
                                          "att, y, H, qdim);\n        for (int i = 0; i < H; i++)\n"
                                          "            x[i] = y[i];"),
    "decode_swiglu_operands_swapped": ("g[i] = oracle_silu(g[i]) * u[i];", "g[i] = g[i] * oracle_silu(u[i]);"),
    "decode_value_plane_is_key_plane": ("uint16_t *vc = kc + plane;", "uint16_t *vc = kc;"),
    "decode_ffn_uses_attention_norm": ("rmsnorm_row(x, mdl->ffn_norm[l], h, H, mdl->eps);",
                                       "rmsnorm_row(x, mdl->attn_norm[l], h, H, mdl->eps);"),
    "decode_final_norm_dropped": ("rmsnorm_row(x, mdl->out_norm, h, H, mdl->eps);",
                                  "for (int i = 0; i < H; i++)\n        h[i] = x[i];"),
    "decode_rope_before_q_norm": ("oracle_head_rmsnorm(qkv + hh * hd, mdl->q_norm[l], hd, mdl->eps);\n"
                                  "                oracle_rope(qkv + hh * hd, hd, pos, mdl->rope_theta);",
                                  "oracle_rope(qkv + hh * hd, hd, pos, mdl->rope_theta);\n"
                                  "                oracle_head_rmsnorm(qkv + hh * hd, mdl->q_norm[l], hd, mdl->eps);"),
    "decode_key_not_rotated": ("oracle_rope(qkv + qdim + kvh * hd, hd, pos, mdl->rope_theta);", ";"),
    "decode_query_norm_on_kv_head_count": ("for (int hh = 0; hh < nq; hh++) {", "for (int hh = 0; hh < nkv; hh++) {"),
    "decode_vocab_as_q4k": ("gemv_any(FMT_Q6K, mdl->wvocab, h, logits, mdl->vocab, H);",
                            "gemv_any(FMT_Q4K, mdl->wvocab, h, logits, mdl->vocab, H);"),
    "decode_key_uses_query_norm": ("oracle_head_rmsnorm(qkv + qdim + kvh * hd, mdl->k_norm[l], hd, mdl->eps);",
                                   "oracle_head_rmsnorm(qkv + qdim + kvh * hd, mdl->q_norm[l], hd, mdl->eps);"),
}


def _build(text: str, lib: str) -> None:
    src = lib[:-3] + ".c"
    with open(src, "w") as f:
        f.write(text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", src, "-o", lib, "-lm"], check=True,
                   capture_output=True)


def _pins_exit_code(lib: str) -> int:
    env = dict(os.environ, DQ_ORACLE_MUTANT=lib, OMP_NUM_THREADS="1")
    run = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu"],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    return run.returncode


def test_pins_reject_every_planted_slip(tmp_path):
    with open(SRC) as f:
        src = f.read()
    builds = {"control": src}
    for name, (old, new) in MUTANTS.items():
        assert src.count(old) == 1, f"{name}: the text to mutate must occur exactly once"
        builds[name] = src.replace(old, new)

    def run(item):
        name, text = item
        lib = str(tmp_path / f"lib_{name}.so")
        _build(text, lib)
        return name, _pins_exit_code(lib)

    with concurrent.futures.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        codes = dict(ex.map(run, builds.items()))
    assert codes.pop("control") == 0, "the unchanged oracle must pass its pins"
    # exit code 1: tests ran and at least one failed (not a crash or a collection error)
    survivors = {name: code for name, code in codes.items() if code != 1}
    assert not survivors, f"planted slips the pins did not reject (name: pytest exit code): {survivors}"
