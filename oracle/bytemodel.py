"""Closed-form byte model of a batched decode step (TEST INFRASTRUCTURE ONLY).

From "Batched swarm: the KV read does not amortize", section "The two halves
of a decode-step memory bill": a step that advances B sequences, each holding
L cached tokens, moves the shared weight stream W once plus B*L*k bytes of
private KV, where k is the KV bytes per token.  Per generated token that is
W/B + L*k.  Section "Where the private read overtakes the shared one" gives
the B-sequence speedup over one sequence, B*(W + L*k)/(W + B*L*k), and the
crossover context where the private read equals the shared one, L* = W/(B*k)
("Q8 KV cache pushes an RDNA4 swarm crossover...", section "The crossover is
just a byte count", states the same equality).
"""
from __future__ import annotations


def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, kv: str = "f16") -> int:
    """KV bytes one token adds to one sequence's cache, K and V over all layers.

    f16: 2 bytes per element.  q8_0: 32-element blocks of int8 codes plus one
    fp16 scale, i.e. 34 bytes per 32 elements.  fp8: one e4m3 byte per element,
    no scale.  A (k, v) pair of kinds gives each tensor its own type."""
    if isinstance(kv, tuple):
        k, v = kv
        return (kv_bytes_per_token(n_layers, n_kv_heads, head_dim, k) +
                kv_bytes_per_token(n_layers, n_kv_heads, head_dim, v)) // 2
    elems = 2 * n_layers * n_kv_heads * head_dim
    if kv == "f16":
        return 2 * elems
    if kv == "q8_0":
        assert head_dim % 32 == 0
        return elems // 32 * 34
    if kv == "fp8":
        return elems
    raise ValueError(kv)


def q4k_bytes(rows: int, cols: int) -> int:
    """Canonical Q4_K bytes of a rows x cols matrix: 144 bytes per 256 weights."""
    assert cols % 256 == 0
    return rows * cols // 256 * 144


def weight_bytes(n_layers=36, hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128,
                 ffn=14336, vocab=151936, with_norms=True) -> int:
    """Bytes of the shared weight stream of one step: every layer's Q4_K
    matrices, the tied embedding / LM head, and (optionally) the fp32 norm gains."""
    q = n_q_heads * head_dim
    kvd = n_kv_heads * head_dim
    per_layer = (q4k_bytes(q, hidden) + 2 * q4k_bytes(kvd, hidden) + q4k_bytes(hidden, q)
                 + 2 * q4k_bytes(ffn, hidden) + q4k_bytes(hidden, ffn))
    total = n_layers * per_layer + q4k_bytes(vocab, hidden)
    if with_norms:
        total += (2 * n_layers + 1) * hidden * 4
    return total


def step_bytes(W: float, B: int, L: float, k: float) -> float:
    """Bytes one decode step moves: shared weights once plus B private KV reads."""
    return W + B * L * k


def per_token_bytes(W: float, B: int, L: float, k: float) -> float:
    return W / B + L * k


def speedup(W: float, B: int, L: float, k: float) -> float:
    """Aggregate-throughput gain of one B-sequence step over B single steps."""
    return B * (W + L * k) / (W + B * L * k)


def crossover(W: float, B: int, k: float) -> float:
    """Context per sequence where the private KV read equals the shared weight read."""
    return W / (B * k)


def time_model_ms(B: int, ctx: float, base_ms: float = 16.9, per_seq_ms: float = 1.1,
                  k_ms_per_token: float = 4.1e-4) -> float:
    """The RX 9070 XT step-time fit t(B, C) = 16.9 + B*(1.1 + k*C) ms from the
    crossover page's figure caption; k is fitted, not printed."""
    return base_ms + B * (per_seq_ms + k_ms_per_token * ctx)
