"""Parity at the sweep's published configurations: full-width layers (hidden
4096, 32/8 heads of 128, SwiGLU 14336, the full 151,936-row tied LM head) at
the batch sizes and contexts the benchmark grid reports, fp16 and Q8_0
caches, through the C ABI against the CPU oracle.

Two layers keep the oracle to seconds per sequence; the projection kernels,
their K splits and the attention's split are chosen by batch size and
context alone, so these are the same launches the 36-layer sweep times.
Contexts follow the pages' swarm ("Batched swarm: the KV read does not
amortize", section "Where the private read overtakes the shared one":
contexts from a few thousand to tens of thousands of tokens per agent)."""
import numpy as np
import pytest

from synth.model import ModelDesc, make_tokens
from tests.helpers import cached_model, gpu, needs_cuda
from tests.test_gpu_step import check_step, setup_pair

pytestmark = [gpu, needs_cuda, pytest.mark.slow]

torch = pytest.importorskip("torch")

WIDE2 = ModelDesc(n_layers=2)   # full width and vocabulary, two layers


def _run(seed, lengths, kv_dtype, n_steps, tag):
    w = cached_model(WIDE2, seed)
    dec, om, kvs = setup_pair(WIDE2, w, seed, lengths, kv_dtype, max(lengths) + n_steps + 1)
    pos = np.array(lengths, np.int32)
    for s in range(n_steps):
        check_step(dec, om, kvs, make_tokens(WIDE2, seed * 100 + s, len(lengths)), pos,
                   f"{tag} kv{kv_dtype} step {s}")
        pos += 1
    assert [dec.seq_len(b) for b in range(len(lengths))] == list(pos)
    dec.close()


@pytest.mark.parametrize("kv_dtype", [0, 1])
def test_b32_ragged_contexts(kv_dtype):
    """B = 32 (the one-CTA-per-SM projection kernels, NT = 8) over ragged
    contexts from 64 to 2048, two steps.  (A row with no history attends
    only to its own new token, whose quantized V then reaches the output
    undiluted; the quantized caches' empty-history case is checked on the
    small model, where its bound is stated.)"""
    lengths = [64 + (97 * b + 41 * (b % 5)) % 1985 for b in range(32)]
    lengths[0], lengths[31] = 2048, 64
    _run(21, lengths, kv_dtype, 2, "B=32 ragged<=2048")


@pytest.mark.parametrize("kv_dtype", [0, 1])
def test_b16_l16384(kv_dtype):
    """B = 16 (NT = 4 projections) at 16k tokens per sequence."""
    _run(22, [16384] * 15 + [16000], kv_dtype, 1, "B=16 L=16384")


@pytest.mark.parametrize("kv_dtype", [0, 1])
def test_b2_l32768(kv_dtype):
    """Two sequences at 32k tokens: the longest context of the grid."""
    _run(23, [32768, 32700], kv_dtype, 1, "B=2 L=32768")
