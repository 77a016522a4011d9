"""The paged KV pool and slot indirection through the C ABI against the CPU
oracle: rows of a step mapped to any slots, slots of very different lengths
sharing one page pool, a slot freed and its pages re-admitted to a new
sequence mid-run, and a pool that runs out of pages refusing cleanly.

The pages' swarm is the source of the shapes: agents hold 800 to 30,000
tokens and the KV budget, not the arithmetic, bounds how many run ("Eight
concurrent agents pull 5.6x more tokens from one RX 9070 XT", sections
"Where it stops, and the argument I got wrong in May" and "What I am
building next")."""
import numpy as np
import pytest

import oracle
from synth.model import ModelDesc, make_kv_history, make_tokens
from tests.helpers import cached_model, gpu, needs_cuda
from tests.test_gpu_step import SMALL, check_step, odesc

pytestmark = [gpu, needs_cuda]

torch = pytest.importorskip("torch")
import quantized_decode_step_02_gb300 as z  # noqa: E402

WIDE2 = ModelDesc(n_layers=2)   # full width and vocabulary, two layers


def _history(dec, d, seed, slot, seq_id, L, kv_dtype, max_L):
    """The seeded history of sequence seq_id into `slot` and into a new oracle cache."""
    kv = oracle.KV(odesc(d), max_L, kv_dtype)
    if L:
        k, v = make_kv_history(d, seed, seq_id, L)
        dec.append_kv(slot, k, v)
        kv.append(k, v)
    return kv


class _Slots:
    """check_step over rows mapped to slots (the decoder runs step_host with slots)."""

    def __init__(self, dec, slots):
        self.dec, self.slots = dec, slots
        self.desc = dec.desc

    def step_capture_hidden(self, tokens, positions, logits=None, ids=None):
        B = len(tokens)
        hid = np.empty((B, self.desc.n_layers + 1, self.desc.hidden), np.float32)
        self.dec._check(self.dec.lib.zdec_debug_capture_hidden(self.dec.h, hid.ctypes.data))
        logits, ids = self.dec.step_host(tokens, positions, logits, ids, slots=self.slots)
        return logits, ids, hid


@pytest.mark.parametrize("kv_dtype", [0, 1])
def test_rows_mapped_to_any_slots(kv_dtype):
    """Three rows in slots 3, 0 and 2 of four (slot 1 idle), two steps, then the
    same slots in another row order: every step matches the oracle, each slot
    grows by one per step, the idle slot is untouched."""
    d = SMALL
    w = cached_model(d, 131)
    dec = z.Decoder(d, w, kv_dtype, max_B=4, max_L=300)
    om = oracle.Model(odesc(d), w)
    L = {3: 70, 0: 5, 2: 200, 1: 33}
    kvs = {s: _history(dec, d, 131, s, s, L[s], kv_dtype, 300) for s in L}
    for step, slots in enumerate([[3, 0, 2], [3, 0, 2], [2, 3, 0]]):
        pos = np.array([dec.seq_len(s) for s in slots], np.int32)
        check_step(_Slots(dec, slots), om, [kvs[s] for s in slots], make_tokens(d, 1310 + step, 3), pos,
                   f"slots {slots} kv{kv_dtype} step {step}")
    assert [dec.seq_len(s) for s in range(4)] == [8, 33, 203, 73]
    dec.close()


def test_pool_runs_out_and_reset_returns_pages():
    """A pool of four pages: filling it refuses further appends and steps with
    ZDEC_ERR_CAPACITY and changes nothing; resetting a slot returns its pages,
    which the next sequence takes."""
    d = SMALL
    w = cached_model(d, 132)
    dec = z.Decoder(d, w, z.KV_F16, max_B=2, max_L=512, pool_tokens=4 * z.PAGE_TOKENS)
    om = oracle.Model(odesc(d), w)
    assert dec.info()["pool_pages"] == 4 and dec.info()["free_pages"] == 4
    kv0 = _history(dec, d, 132, 0, 0, 250, 0, 512)   # four pages (tokens 0..255)
    assert dec.info()["free_pages"] == 0
    k, v = make_kv_history(d, 132, 1, 1)
    with pytest.raises(z.ZdecError) as e:
        dec.append_kv(1, k, v)
    assert e.value.status == -3 and dec.seq_len(1) == 0
    pos = np.array([250], np.int32)
    for s in range(6):   # tokens 250..255 still fit the fourth page
        check_step(dec, om, [kv0], make_tokens(d, 1320 + s, 1), pos, f"full pool step {s}")
        pos += 1
    with pytest.raises(z.ZdecError) as e:   # token 256 needs a fifth page
        dec.step_host(make_tokens(d, 1330, 1), pos)
    assert e.value.status == -3 and dec.seq_len(0) == 256 and dec.info()["free_pages"] == 0
    table0 = dec.block_table(0)
    dec.reset_seq(0)
    assert dec.info()["free_pages"] == 4 and (dec.block_table(0) < 0).all()
    kv1 = _history(dec, d, 132, 1, 7, 100, 0, 512)   # a new sequence takes two freed pages
    t1 = dec.block_table(1)
    assert set(t1[:2]) <= set(table0[:4]) and (t1[2:] < 0).all()
    check_step(_Slots(dec, [1]), om, [kv1], make_tokens(d, 1331, 1), np.array([100], np.int32), "re-admitted")
    dec.close()


@pytest.mark.slow
@pytest.mark.parametrize("kv_dtype", [0, 1])
def test_ragged_swarm_with_readmission(kv_dtype):
    """Two full-width layers, four agents of 800 to 30,000 tokens in a pool too
    small for four full slots: two steps, then the 5,000-token agent retires
    and a new 3,000-token one is admitted into its slot (its freed pages),
    and two more steps run with the rows in another order."""
    d = WIDE2
    w = cached_model(d, 24)
    max_L = 30100
    lengths = {0: 800, 1: 5000, 2: 30000, 3: 12000}
    pool = sum(lengths.values()) + 4 * 2 * z.PAGE_TOKENS + 3000
    dec = z.Decoder(d, w, kv_dtype, max_B=4, max_L=max_L, pool_tokens=pool)
    om = oracle.Model(odesc(d), w)
    kvs = {s: _history(dec, d, 24, s, s, lengths[s], kv_dtype, max_L) for s in lengths}
    for step in range(2):
        slots = [0, 1, 2, 3]
        pos = np.array([dec.seq_len(s) for s in slots], np.int32)
        check_step(_Slots(dec, slots), om, [kvs[s] for s in slots], make_tokens(d, 240 + step, 4), pos,
                   f"swarm kv{kv_dtype} step {step}")
    free_before = dec.info()["free_pages"]
    dec.reset_seq(1)
    assert dec.info()["free_pages"] == free_before + (5002 + 63) // 64
    kvs[1] = _history(dec, d, 24, 1, 9, 3000, kv_dtype, max_L)
    for step in range(2):
        slots = [2, 1, 3, 0]
        pos = np.array([dec.seq_len(s) for s in slots], np.int32)
        check_step(_Slots(dec, slots), om, [kvs[s] for s in slots], make_tokens(d, 250 + step, 4), pos,
                   f"swarm re-admitted kv{kv_dtype} step {step}")
    assert [dec.seq_len(s) for s in range(4)] == [804, 3002, 30004, 12004]
    dec.close()
