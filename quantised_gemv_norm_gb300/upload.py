"""Move a synthetic host model (numpy) to the GPU as torch tensors for dq.Model."""
from __future__ import annotations

import numpy as np
import torch


def to_device(m, kv_cache: np.ndarray, device="cuda") -> dict:
    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a)).to(device, non_blocking=False)

    w = {
        "attn_norm": [t(a) for a in m.attn_norm],
        "ffn_norm": [t(a) for a in m.ffn_norm],
        "wqkv": [t(a) for a in m.wqkv],
        "wo": [t(a) for a in m.wo],
        "wgate": [t(a) for a in m.wgate],
        "wup": [t(a) for a in m.wup],
        "wdown": [t(a) for a in m.wdown],
        "down_fmt": list(m.down_fmt),
        "out_norm": t(m.out_norm),
        "wvocab": t(m.wvocab),
        "kv_cache": torch.from_numpy(kv_cache.view(np.int16)).to(device),
    }
    if getattr(m, "q_norm", None):
        w["q_norm"] = [t(a) for a in m.q_norm]
        w["k_norm"] = [t(a) for a in m.k_norm]
    return w


def model_kwargs(m) -> dict:
    return dict(n_layers=m.n_layers, hidden=m.hidden, ffn=m.ffn, n_q_heads=m.n_q_heads, n_kv_heads=m.n_kv_heads,
                head_dim=m.head_dim, vocab=m.vocab, max_ctx=m.max_ctx, eps=m.eps,
                rope_theta=float(getattr(m, "rope_theta", 0.0) or 0.0))
