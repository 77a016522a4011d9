"""Synthetic model, KV histories and token batches, all from seeded streams.

The shapes are those of a 36-layer GQA decoder (hidden 4096, 32 query / 8 KV
heads of 128, SwiGLU FFN 14336, tied 151,936-row embedding); weights are
N(0, 0.02^2) quantized to canonical Q4_K, norm gains 1 + 0.1*N(0,1) (not all
ones, so that a dropped gain shows), KV history N(0,1) rounded to fp16 and
treated as already rotated.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

from . import kv_stream, normal_f16, normal_f32, q4k_matrix, stream_id, uniform_int


@dataclass(frozen=True)
class ModelDesc:
    n_layers: int = 36
    hidden: int = 4096
    n_q_heads: int = 32
    n_kv_heads: int = 8
    head_dim: int = 128
    ffn: int = 14336
    vocab: int = 151936
    rope_theta: float = 1e6
    rms_eps: float = 1e-6

    def with_(self, **kw) -> "ModelDesc":
        return replace(self, **kw)

    def astuple(self):
        return (self.n_layers, self.hidden, self.n_q_heads, self.n_kv_heads, self.head_dim,
                self.ffn, self.vocab, self.rope_theta, self.rms_eps)


FULL = ModelDesc()
WEIGHT_STD = 0.02
GAIN_STD = 0.1


def make_model(desc: ModelDesc, seed: int) -> dict:
    """Canonical Q4_K weights: dict of uint8 [rows, cols/256*144] matrices
    (per-layer tensors as lists) plus fp32 norm gains."""
    H, F = desc.hidden, desc.ffn
    qd, kvd = desc.n_q_heads * desc.head_dim, desc.n_kv_heads * desc.head_dim
    w = {"embed": q4k_matrix(seed, stream_id("embed"), desc.vocab, H, WEIGHT_STD)}
    gain = lambda stream: normal_f32(seed, stream, H, std=GAIN_STD, mean=1.0)
    w["final_norm"] = gain(10)
    shapes = {"wq": (qd, H), "wk": (kvd, H), "wv": (kvd, H), "wo": (H, qd),
              "w_gate": (F, H), "w_up": (F, H), "w_down": (H, F)}
    for name in shapes:
        w[name] = []
    w["attn_norm"], w["ffn_norm"] = [], []
    for l in range(desc.n_layers):
        for name, (r, c) in shapes.items():
            w[name].append(q4k_matrix(seed, stream_id(name, l), r, c, WEIGHT_STD))
        w["attn_norm"].append(gain(20 + 2 * l))
        w["ffn_norm"].append(gain(21 + 2 * l))
    return w


def make_kv_history(desc: ModelDesc, seed: int, seq: int, L: int):
    """fp16 (uint16 bits) K and V of L cached tokens: [n_layers][L][n_kv][hd]."""
    n = L * desc.n_kv_heads * desc.head_dim
    shape = (desc.n_layers, L, desc.n_kv_heads, desc.head_dim)
    k = np.empty(shape, dtype=np.uint16)
    v = np.empty(shape, dtype=np.uint16)
    for l in range(desc.n_layers):
        k[l] = normal_f16(seed, kv_stream(seq, l, 0), n).reshape(shape[1:])
        v[l] = normal_f16(seed, kv_stream(seq, l, 1), n).reshape(shape[1:])
    return k, v


def make_tokens(desc: ModelDesc, seed: int, B: int) -> np.ndarray:
    return uniform_int(seed, stream_id("tokens"), B, desc.vocab)
