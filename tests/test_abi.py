"""The C-ABI library: builds, loads and exports every symbol include/dq.h declares;
argument checks that return before any CUDA call.  No GPU needed."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dq.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"DQ_API\s+[\w\s\*]+?\b(dq_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from quantised_gemv_norm_gb300 import build

    build.build()
    from quantised_gemv_norm_gb300 import dq

    return dq.load()


def test_header_declares_the_hot_path():
    names = declared_symbols()
    for required in ("dq_rmsnorm", "dq_layernorm", "dq_gemv_bf16", "dq_gemv_q4k", "dq_gemv_q6k",
                     "dq_dequant_q4k", "dq_dequant_q6k", "dq_attention_decode", "dq_matmul_q4k",
                     "dq_model_create", "dq_decode_step", "dq_model_destroy"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def test_binding_covers_every_declared_symbol():
    from quantised_gemv_norm_gb300 import dq

    assert sorted(dq.SIGNATURES) == declared_symbols()


def test_status_strings(lib):
    for code in range(0, -8, -1):
        s = lib.dq_status_string(code)
        assert s and s != b"unknown status"
    assert lib.dq_status_string(-99) == b"unknown status"


def test_argument_errors_return_before_launch(lib):
    P = ctypes.c_void_p
    fake = P(16)  # never dereferenced: checks fail first
    assert lib.dq_gemv_q4k(None, fake, fake, 4, 256, None) == -1
    assert lib.dq_gemv_q4k(P(17), fake, fake, 4, 256, None) == -3          # misaligned W
    assert lib.dq_gemv_q4k(fake, fake, fake, 4, 16640, None) == -4        # K too large
    assert lib.dq_gemv_q6k(fake, fake, fake, 4, 40000, None) == -4
    assert lib.dq_gemv_bf16(fake, fake, fake, 4, 30000, None) == -4
    assert lib.dq_rmsnorm(None, fake, fake, 1, 8, 1e-6, None) == -1
    assert lib.dq_rmsnorm(fake, fake, fake, 0, 8, 1e-6, None) == -2
    assert lib.dq_rmsnorm_threads(fake, fake, fake, 1, 8, 1e-6, 3, None) == -2  # not a power of two
    assert lib.dq_layernorm(fake, fake, None, fake, 1, 8, 1e-6, None) == -1
    assert lib.dq_dequant_q4k(fake, fake, 0, None) == -2
    assert lib.dq_dequant_q2k(fake, fake, 0, None) == -2
    assert lib.dq_gemv_q2k(fake, fake, fake, 4, 1536, None) == -3         # 84-byte blocks: K % 1024
    assert lib.dq_gemv_q2k(fake, fake, fake, 4, 17408, None) == -4
    assert lib.dq_gemv_ex(4, fake, fake, fake, 4, 256, 0, None) == -2      # no such format
    assert lib.dq_gemv_ex(1, fake, fake, fake, 4, 256, 2, None) == -2      # unknown flag
    assert lib.dq_gemv_ex(1, None, fake, fake, 4, 256, 1, None) == -1
    assert lib.dq_gemv_ex(1, fake, fake, fake, 4, 16640, 1, None) == -4
    assert lib.dq_gemv_ex(0, fake, fake, fake, 4, 30000, 0, None) == -4
    assert lib.dq_attention_decode(fake, fake, fake, fake, 32, 8, 64, 16, 1, fake, 1 << 20, None) == -4
    assert lib.dq_attention_decode(fake, fake, fake, fake, 32, 8, 128, 16, 17, fake, 1 << 20, None) == -2
    assert lib.dq_attention_decode(fake, fake, fake, fake, 32, 8, 128, 16, 4, fake, 8, None) == -2
    assert lib.dq_matmul_q4k(fake, fake, fake, 65, 4, 256, None) == -2
    assert lib.dq_matmul_q4k(fake, fake, fake, 2, 4, 300, None) == -2         # K not a multiple of 256
    assert lib.dq_matmul_q4k_path(fake, fake, fake, 2, 4, 256, 3, None) == -2  # no such path
    assert lib.dq_matmul_q4k_path(P(17), fake, fake, 2, 4, 256, 2, None) == -3
    assert lib.dq_matmul_q4k_path(fake, fake, fake, 2, 4, 32768, 1, None) == -4
    assert lib.dq_matmul_q4k_split(fake, fake, fake, 2, 4, 256, None, 1 << 20, None) == -1
    assert lib.dq_matmul_q4k_split(fake, fake, fake, 65, 4, 256, fake, 1 << 20, None) == -2
    assert lib.dq_matmul_q4k_split(fake, fake, fake, 2, 4, 300, fake, 1 << 20, None) == -2
    assert lib.dq_matmul_q4k_split(fake, fake, fake, 2, 4, 256, P(24), 1 << 20, None) == -3  # misaligned workspace
    assert lib.dq_matmul_q4k_split_workspace_bytes(0, 4, 256) == -2
    assert lib.dq_matmul_q4k_split_workspace_bytes(2, 4, 300) == -2
    assert lib.dq_matmul_q4k_split_workspace_bytes(2, 524289, 256) == -4
    assert lib.dq_matmul_q4k_split(fake, fake, fake, 2, 524289, 256, fake, 1 << 40, None) == -4
    assert lib.dq_rope_table(None, 16, 128, 1e6, None) == -1
    assert lib.dq_rope_table(fake, 16, 127, 1e6, None) == -2              # odd head_dim
    assert lib.dq_rope_table(fake, 16, 128, 1.0, None) == -2              # theta must exceed 1
    assert lib.dq_rope_table(P(24), 16, 128, 1e6, None) == -3
    r = lib.dq_attention_decode_rope
    assert r(fake, None, fake, fake, fake, fake, fake, fake, 1e-6, 32, 8, 128, 16, 1, fake, 1 << 20, None) == -1
    assert r(fake, fake, fake, fake, fake, fake, fake, fake, 1e-6, 32, 8, 64, 16, 1, fake, 1 << 20, None) == -4
    assert r(fake, fake, fake, fake, fake, fake, fake, fake, 1e-6, 32, 8, 128, 16, 0, fake, 1 << 20, None) == -2
    assert r(fake, fake, fake, fake, fake, fake, fake, P(24), 1e-6, 32, 8, 128, 16, 1, fake, 1 << 20, None) == -3
    # a norm epsilon must be finite and >= 0
    for eps in (-1e-6, float("nan"), float("inf")):
        assert lib.dq_rmsnorm(fake, fake, fake, 1, 8, eps, None) == -2
        assert lib.dq_layernorm_threads(fake, fake, fake, fake, 1, 8, eps, 64, None) == -2
        assert r(fake, fake, fake, fake, fake, fake, fake, fake, eps, 32, 8, 128, 16, 1, fake, 1 << 20, None) == -2
    assert lib.dq_rmsnorm(fake, P(24), fake, 1, 8, 1e-6, None) == -3  # gamma read as float4
    assert lib.dq_decode_step(None, fake, 0, fake, None) == -1
    assert lib.dq_decode_step_host(None, fake, 0, fake, None) == -1
    h = P()
    assert lib.dq_model_create(None, ctypes.byref(h)) == -1
    assert lib.dq_model_destroy(None) == 0


def test_attention_workspace_size(lib):
    assert lib.dq_attention_workspace_bytes(32, 8) == 256 + 32 * 32 * 132 * 4
    assert lib.dq_attention_workspace_bytes(0, 8) == 0


def test_model_create_checks_qwen3_inputs_before_allocating(lib):
    # q_norm set: k_norm, every layer's weights and the rotary base are checked first
    from quantised_gemv_norm_gb300 import dq

    L = 2
    fake = [16 * (i + 1) for i in range(L)]

    def arr(vals):
        a = (ctypes.c_void_p * L)(*vals)
        keep.append(a)
        return ctypes.cast(a, ctypes.c_void_p)

    keep = []
    fmts = (ctypes.c_int * L)(1, 2)

    def desc(q_norm, k_norm, theta):
        d = dq._Desc(L, 2048, 4096, 8, 2, 128, 1000, 64, 1e-6, arr(fake), arr(fake), arr(fake), arr(fake),
                     arr(fake), arr(fake), arr(fake), ctypes.cast(fmts, ctypes.c_void_p), 16, 16, 16, 0, 0)
        d.q_norm = q_norm
        d.k_norm = k_norm
        d.rope_theta = theta
        return d

    h = ctypes.c_void_p()
    assert lib.dq_model_create(ctypes.byref(desc(arr(fake), None, 1e6)), ctypes.byref(h)) == -1
    assert lib.dq_model_create(ctypes.byref(desc(arr(fake), arr(fake), 0.5)), ctypes.byref(h)) == -2
    assert lib.dq_model_create(ctypes.byref(desc(arr(fake), arr([16, 0]), 1e6)), ctypes.byref(h)) == -1
    assert lib.dq_model_create(ctypes.byref(desc(arr(fake), arr([16, 40]), 1e6)), ctypes.byref(h)) == -3
    for eps in (-1.0, float("nan"), float("inf")):
        d = desc(arr(fake), arr(fake), 1e6)
        d.eps = eps
        assert lib.dq_model_create(ctypes.byref(d), ctypes.byref(h)) == -2
    assert h.value is None


def test_binding_struct_and_constants_match_the_header(tmp_path):
    # the header compiled by a C compiler reports the descriptor's layout and the
    # constants; the ctypes binding must agree field by field
    import subprocess

    from quantised_gemv_norm_gb300 import dq, synth

    fields = [name for name, _ in dq._Desc._fields_]
    consts = ["DQ_OK", "DQ_ERR_NULL", "DQ_ERR_SHAPE", "DQ_ERR_ALIGN", "DQ_ERR_UNSUPPORTED", "DQ_ERR_CUDA",
              "DQ_ERR_TIMEOUT", "DQ_ERR_ALLOC", "DQ_FMT_BF16", "DQ_FMT_Q4K", "DQ_FMT_Q6K", "DQ_FMT_Q2K",
              "DQ_MODEL_NO_PDL", "DQ_MODEL_FUSED", "DQ_MATMUL_AUTO", "DQ_MATMUL_CUDA_CORE", "DQ_MATMUL_TENSOR"]
    src = ["#include <stdio.h>", "#include <stddef.h>", '#include "dq.h"', "int main(void) {",
           '  printf("size %zu\\n", sizeof(dq_model_desc));']
    src += ['  printf("%s %%zu\\n", offsetof(dq_model_desc, %s));' % (f, f) for f in fields]
    src += ['  printf("%s %%d\\n", (int)(%s));' % (c, c) for c in consts]
    src += ["  return 0;", "}"]
    c = tmp_path / "layout.c"
    c.write_text("\n".join(src) + "\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c11", "-I", os.path.join(ROOT, "include"), str(c), "-o", str(exe)], check=True)
    got = dict(line.split() for line in subprocess.run([str(exe)], check=True, capture_output=True,
                                                           text=True).stdout.splitlines())
    assert int(got["size"]) == ctypes.sizeof(dq._Desc)
    for f in fields:
        assert int(got[f]) == getattr(dq._Desc, f).offset, f
    assert [int(got[c]) for c in consts[:8]] == [0, -1, -2, -3, -4, -5, -6, -7]
    assert [int(got[c]) for c in consts[8:12]] == [synth.FMT_BF16, synth.FMT_Q4K, synth.FMT_Q6K, synth.FMT_Q2K]
    assert [int(got[c]) for c in consts[12:14]] == [dq.MODEL_NO_PDL, dq.MODEL_FUSED]
    assert [int(got[c]) for c in consts[14:]] == [dq.MATMUL_AUTO, dq.MATMUL_CUDA_CORE, dq.MATMUL_TENSOR]
