"""The bench's reference arm (the CPU oracle) on this host: its JSON line keeps the
contract's keys and the requested step counts, and ranks other than 0 print nothing."""
import json
import types

import pytest


@pytest.fixture
def bench_mod(monkeypatch):
    import bench

    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    return bench


def test_reference_line_with_sampled_steps(bench_mod, monkeypatch, capsys):
    monkeypatch.setattr(bench_mod, "REFERENCE_BUDGET_S", 1e-3)  # forces the smallest sample
    bench_mod.run_reference(types.SimpleNamespace(steps=2, warmup=3))
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True and line["value"] > 0
    assert line["metric"] == bench_mod.METRIC and line["config"]["workload"] == bench_mod.WORKLOAD
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert "first 1 of 36 layers" in cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_sample_model_keeps_layer_shapes(bench_mod):
    from quantised_gemv_norm_gb300 import synth

    m = synth.make_model(2, n_layers=4, hidden=256, ffn=512, n_q_heads=4, n_kv_heads=2, head_dim=64, vocab=300,
                         max_ctx=8, qwen3_attention=True)
    s = bench_mod.sample_model(m, 3, 100)
    assert s.n_layers == 3 and s.vocab == 100 and s.wvocab.shape == (100, m.wvocab.shape[1])
    for name in ("attn_norm", "wqkv", "wo", "ffn_norm", "wgate", "wup", "wdown", "down_fmt", "q_norm", "k_norm"):
        assert len(getattr(s, name)) == 3 and all(a is b for a, b in zip(getattr(s, name), getattr(m, name)))
    assert m.n_layers == 4 and m.vocab == 300  # the full model is untouched


def test_reference_other_ranks_print_nothing(bench_mod, monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench_mod.run_reference(types.SimpleNamespace(steps=2, warmup=3))
    assert capsys.readouterr().out == ""
