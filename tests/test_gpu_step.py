"""Full decode-step parity on the GPU through the C ABI against the CPU oracle:
small models over several steps with ragged lengths, fp16, Q8_0 and FP8
caches (one type for K and V, or one each), per-layer hidden states, logits
and ids; batch-B vs B independent steps; graph replay vs eager launches;
device-side input checks."""
import numpy as np
import pytest

import oracle
from synth.model import ModelDesc, make_kv_history, make_tokens
from tests.helpers import GAP, TOL, cached_model, gpu, needs_cuda, normwise, record_margin, top2_gap

pytestmark = [gpu, needs_cuda]

torch = pytest.importorskip("torch")
import quantized_decode_step_02_gb300 as z  # noqa: E402

SMALL = ModelDesc(n_layers=3, hidden=1024, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn=2048,
                  vocab=3000)


def odesc(d):
    return oracle.Desc(*d.astuple())


def setup_pair(d, w, seed, lengths, kv_dtype, max_L):
    """A GPU decoder and oracle caches holding the same seeded history."""
    B = len(lengths)
    dec = z.Decoder(d, w, kv_dtype, max_B=B, max_L=max_L)
    om = oracle.Model(odesc(d), w)
    kvs = []
    for b, L in enumerate(lengths):
        kv = oracle.KV(odesc(d), max_L, kv_dtype)
        if L:
            k, v = make_kv_history(d, seed, b, L)
            dec.append_kv(b, k, v)
            kv.append(k, v)
        kvs.append(kv)
    return dec, om, kvs


def check_step(dec, om, kvs, tokens, positions, tag=""):
    """One host-I/O step through the C ABI against the oracle's step: every
    row's residual after the embedding and after each layer and its logits
    within TOL (normwise), ids equal where the oracle's top-2 gap exceeds GAP.
    The worst errors go to record_margin (printed, and kept in a file when
    ZDEC_MARGINS_FILE is set)."""
    B = len(tokens)
    logits = np.empty((B, dec.desc.vocab), np.float32)
    _, ids, hid = dec.step_capture_hidden(tokens, positions, logits)
    rl, rid, rhid = oracle.decode_step(om, kvs, tokens, positions, capture_hidden=True)
    gaps = top2_gap(rl)
    worst_h = worst_l = 0.0
    n_ids = 0
    for b in range(B):
        for l in range(hid.shape[1]):
            err = normwise(hid[b, l], rhid[b, l])
            worst_h = max(worst_h, err)
            assert err <= TOL, f"{tag} row {b} layer {l}: hidden error {err:.3g}"
        err = normwise(logits[b], rl[b])
        worst_l = max(worst_l, err)
        assert err <= TOL, f"{tag} row {b}: logits error {err:.3g}"
        if gaps[b] > GAP:
            n_ids += 1
            assert ids[b] == rid[b], f"{tag} row {b}: id {ids[b]} != oracle {rid[b]} (gap {gaps[b]:.3g})"
    record_margin(tag, worst_h, worst_l, n_ids, B)
    return logits, ids, rl, rid


@pytest.mark.parametrize("kv_dtype", [0, 1])
def test_small_model_multi_step_ragged(kv_dtype):
    d = SMALL
    w = cached_model(d, 101)
    lengths = [0, 63, 130]
    dec, om, kvs = setup_pair(d, w, 101, lengths, kv_dtype, 160)
    pos = np.array(lengths, np.int32)
    for step in range(3):
        toks = make_tokens(d, 200 + step, 3)
        check_step(dec, om, kvs, toks, pos, f"kv{kv_dtype} step {step}")
        pos += 1
    # the appended tokens agree with the oracle's cache up to the rounding of
    # the projected values (fp16 ulp / one Q8 code)
    for b in range(3):
        n = int(pos[b])
        got = dec.read_kv(b, 1, 0, n)
        if kv_dtype == 0:
            gk = got[0].view(np.float16).astype(np.float64)
            rk = kvs[b].k16[1, :n].view(np.float16).astype(np.float64)
            assert np.allclose(gk, rk, rtol=2e-3, atol=2e-3)
        else:
            assert np.abs(got[0].astype(int) - kvs[b].kq[1, :n].astype(int)).max() <= 1
            assert np.abs(got[1].astype(int) - kvs[b].vq[1, :n].astype(int)).max() <= 1
    assert [dec.seq_len(b) for b in range(3)] == [3, 66, 133]
    dec.close()


@pytest.mark.parametrize("kv_dtype", [0, 1])
def test_batch_of_eight_across_chunk_boundaries(kv_dtype):
    """Eight sequences whose new tokens fall on and next to 64-token chunk
    boundaries, over two steps: the attention's split over a cluster gives
    the rank that appends the new token one chunk less, and that token is
    rotated, quantized and inserted at its own chunk; the appended tokens
    must land in the arena."""
    d = SMALL
    w = cached_model(d, 103)
    lengths = [1, 63, 64, 127, 128, 191, 256, 319]
    dec, om, kvs = setup_pair(d, w, 103, lengths, kv_dtype, 330)
    pos = np.array(lengths, np.int32)
    for step in range(2):
        toks = make_tokens(d, 300 + step, len(lengths))
        check_step(dec, om, kvs, toks, pos, f"kv{kv_dtype} step {step}")
        pos += 1
    for b in (2, 4, 7):
        n = int(pos[b])
        got = dec.read_kv(b, 2, 0, n)
        if kv_dtype == 0:
            gk = got[0].view(np.float16).astype(np.float64)
            rk = kvs[b].k16[2, :n].view(np.float16).astype(np.float64)
            assert np.allclose(gk, rk, rtol=2e-3, atol=2e-3)
        else:
            assert np.abs(got[0].astype(int) - kvs[b].kq[2, :n].astype(int)).max() <= 1
            assert np.abs(got[1].astype(int) - kvs[b].vq[2, :n].astype(int)).max() <= 1
    assert [dec.seq_len(b) for b in range(8)] == [L + 2 for L in lengths]
    dec.close()


def _codes_close(got, ref, kind):
    """Stored codes of tokens the step appended: the GPU's projection differs
    from the oracle's by rounding, so a code may sit one step off."""
    got, ref = np.asarray(got), np.asarray(ref)
    if kind == z.KV_F16:
        a = got.view(np.float16).astype(np.float64)
        b = ref.view(np.float16).astype(np.float64)
        return np.allclose(a, b, rtol=2e-3, atol=2e-3)
    if kind == z.KV_Q8_0:
        return np.abs(got.astype(int) - ref.astype(int)).max() <= 1
    ga = got.astype(np.uint8).astype(int)
    ra = ref.astype(np.uint8).astype(int)
    same_sign = (ga & 0x80) == (ra & 0x80)
    near_zero = ((ga & 0x7F) <= 1) & ((ra & 0x7F) <= 1)
    return bool(np.all((same_sign & (np.abs((ga & 0x7F) - (ra & 0x7F)) <= 1)) | near_zero))


def _oracle_rows(kv, which, layer, t0, n):
    kind = kv.k_type if which == 0 else kv.v_type
    arr = {z.KV_F16: kv.k16 if which == 0 else kv.v16, z.KV_Q8_0: kv.kq if which == 0 else kv.vq,
           z.KV_FP8: kv.k8 if which == 0 else kv.v8}[kind]
    return arr[layer, t0:t0 + n], kind


@pytest.mark.parametrize("types", [(1, 0), (0, 1), (2, 2), (2, 0), (0, 2), (1, 2), (2, 1)])
def test_separate_k_and_v_cache_types(types):
    """K and V each in its own format (fp16, Q8_0 or FP8): two full steps
    against the oracle holding the same per-tensor types, and the appended
    tokens within one code of the oracle's.  Histories are at least one page
    (64 tokens): with a shorter one the new token's own re-quantized V (or
    K) weighs so much in the output that a one-code difference between two
    correct projections can exceed the float tolerance."""
    d = SMALL
    w = cached_model(d, 112)
    lengths = [64, 129, 200]
    dec, om, kvs = setup_pair(d, w, 112, lengths, types, 260)
    pos = np.array(lengths, np.int32)
    for step in range(2):
        check_step(dec, om, kvs, make_tokens(d, 1120 + step, 3), pos, f"types {types} step {step}")
        pos += 1
    for b in range(3):
        got = dec.read_kv(b, 1, lengths[b], 2)
        for which in (0, 1):
            ref, kind = _oracle_rows(kvs[b], which, 1, lengths[b], 2)
            assert _codes_close(got[which], ref, kind), (types, b, which)
    info = dec.info()
    assert (info["k_type"], info["v_type"]) == tuple(types)
    dec.close()


@pytest.mark.parametrize("impl", [1, 2, 3])
def test_matvec_and_mma_paths_both_match(impl):
    d = SMALL
    w = cached_model(d, 102)
    lengths = [40, 9]
    dec, om, kvs = setup_pair(d, w, 102, lengths, 0, 64)
    dec.set_gemm_impl(impl)
    check_step(dec, om, kvs, make_tokens(d, 300, 2), np.array(lengths, np.int32), f"impl {impl}")
    dec.close()
    # batch of one (impl 3 runs its own kernel only there)
    dec, om, kvs = setup_pair(d, w, 102, lengths[:1], 0, 64)
    dec.set_gemm_impl(impl)
    check_step(dec, om, kvs, make_tokens(d, 301, 1), np.array(lengths[:1], np.int32), f"impl {impl} B=1")
    dec.close()


def test_batch_equals_independent_steps():
    d = SMALL
    w = cached_model(d, 103)
    lengths = [17, 0, 90, 64]
    toks = make_tokens(d, 103, 4)
    dec, _, _ = setup_pair(d, w, 103, lengths, 1, 128)
    lg = np.empty((4, d.vocab), np.float32)
    _, ids = dec.step_host(toks, np.array(lengths, np.int32), lg)
    dec.close()
    for b in range(4):
        dec1 = z.Decoder(d, w, z.KV_Q8_0, max_B=1, max_L=128)
        if lengths[b]:
            k, v = make_kv_history(d, 103, b, lengths[b])
            dec1.append_kv(0, k, v)
        lg1 = np.empty((1, d.vocab), np.float32)
        _, id1 = dec1.step_host(toks[b:b + 1], np.array([lengths[b]], np.int32), lg1)
        assert id1[0] == ids[b]
        assert normwise(lg[b], lg1[0]) < 1e-4
        dec1.close()


def test_graph_replay_equals_eager():
    d = SMALL
    w = cached_model(d, 104)
    lengths = [33, 70]
    toks = make_tokens(d, 104, 2)
    out = []
    for eager in (False, True):
        dec, _, _ = setup_pair(d, w, 104, lengths, 0, 128)
        pos = np.array(lengths, np.int32)
        res = []
        for step in range(3):
            lg = np.empty((2, d.vocab), np.float32)
            _, ids = dec.step_host(toks, pos + step, lg, eager=eager)
            res.append((lg.copy(), ids.copy()))
        out.append(res)
        dec.close()
    for (la, ia), (lb, ib) in zip(*out):
        assert np.array_equal(la, lb) and np.array_equal(ia, ib)


def test_device_io_step_and_position_checks():
    d = SMALL
    w = cached_model(d, 105)
    dec, om, kvs = setup_pair(d, w, 105, [12, 3], 0, 32)
    dev = torch.device("cuda")
    toks = torch.from_numpy(make_tokens(d, 105, 2)).to(dev)
    pos = torch.tensor([12, 3], dtype=torch.int32, device=dev)
    logits = torch.empty((2, d.vocab), dtype=torch.float32, device=dev)
    ids = torch.empty(2, dtype=torch.int32, device=dev)
    dec.step(toks, pos, logits, ids)
    dec.sync()
    rl, rid, _ = oracle.decode_step(om, kvs, toks.cpu().numpy(), [12, 3])
    for b in range(2):
        assert normwise(logits[b].cpu().numpy(), rl[b]) <= TOL
    # host I/O: a wrong position is refused before anything runs
    with pytest.raises(z.ZdecError) as e:
        dec.step_host(np.array([1, 2], np.int32), np.array([13, 5], np.int32))
    assert e.value.status == -4
    assert dec.seq_len(0) == 13 and dec.seq_len(1) == 4
    # device inputs: the first kernel checks positions (row 1 is wrong but in
    # range), the step writes no KV row and advances no length, and
    # zdec_sync reports it
    before = [dec.read_kv(b, l, 0, 32) for b in range(2) for l in range(d.n_layers)]
    bad = torch.tensor([13, 9], dtype=torch.int32, device=dev)
    dec.step(toks, bad, logits, ids)
    with pytest.raises(z.ZdecError) as e:
        dec.sync()
    assert e.value.status == -8
    dec.sync()   # the status was cleared
    assert dec.seq_len(0) == 13 and dec.seq_len(1) == 4
    after = [dec.read_kv(b, l, 0, 32) for b in range(2) for l in range(d.n_layers)]
    for x, y in zip(before, after):
        assert all(np.array_equal(u, v) for u, v in zip(x, y))
    # the next correct step is the oracle's step at the unchanged lengths
    check_step(dec, om, kvs, make_tokens(d, 1051, 2), np.array([13, 4], np.int32), "after a flagged step")
    with pytest.raises(z.ZdecError) as e:
        dec.step_host(np.array([d.vocab], np.int32), np.array([14], np.int32))
    assert e.value.status == -1
    dec.close()


def test_wait_that_runs_out_reports_timeout_and_changes_nothing():
    """Every projection's first stage wait gives up at once (the debug bound
    -1): the kernels record the timeout, wait for their own copies in flight
    and return; the step writes no KV row and advances no length; sync
    reports ZDEC_ERR_TIMEOUT; with the default bound back, the next step
    matches the oracle."""
    d = SMALL
    w = cached_model(d, 111)
    lengths = [40, 7]
    dec, om, kvs = setup_pair(d, w, 111, lengths, 1, 64)
    before = [dec.read_kv(b, l, 0, 64) for b in range(2) for l in range(d.n_layers)]
    dec.set_wait_limit(-1)
    for eager in (True, False):   # launched directly and from a captured graph
        with pytest.raises(z.ZdecError) as e:
            dec.step_host(make_tokens(d, 1110, 2), np.array(lengths, np.int32), eager=eager)
        assert e.value.status == -7
        assert [dec.seq_len(b) for b in range(2)] == lengths
    after = [dec.read_kv(b, l, 0, 64) for b in range(2) for l in range(d.n_layers)]
    for x, y in zip(before, after):
        assert all(np.array_equal(u, v) for u, v in zip(x, y))
    dec.set_wait_limit(0)
    check_step(dec, om, kvs, make_tokens(d, 1111, 2), np.array(lengths, np.int32), "after a timeout")
    dec.close()


def test_profile_step_reports_every_launch():
    d = SMALL
    w = cached_model(d, 106)
    dec, _, _ = setup_pair(d, w, 106, [5], 0, 16)
    dev = torch.device("cuda")
    toks = torch.from_numpy(make_tokens(d, 106, 1)).to(dev)
    ids = torch.empty(1, dtype=torch.int32, device=dev)
    rec = dec.profile_step(toks, torch.tensor([5], dtype=torch.int32, device=dev), None, ids)
    kinds = [k for k, _ in rec]
    assert len(rec) == dec.info()["kernels_per_step"] == 3 + 5 * d.n_layers
    assert kinds.count("attention") == d.n_layers and kinds[-1] == "argmax"
    assert all(ms > 0 for _, ms in rec)
    assert dec.seq_len(0) == 6
    dec.close()


# ------------------------------------------------------------ full-size configs
FULL = ModelDesc()


def _full_config(seed, B, lengths, kv_dtype, n_steps=1, max_L=None):
    w = cached_model(FULL, seed)
    max_L = max_L or max(lengths) + n_steps + 1
    dec, om, kvs = setup_pair(FULL, w, seed, lengths, kv_dtype, max_L)
    pos = np.array(lengths, np.int32)
    for s in range(n_steps):
        check_step(dec, om, kvs, make_tokens(FULL, seed * 100 + s, B), pos, f"seed {seed} step {s}")
        pos += 1
    dec.close()


@pytest.mark.slow
def test_full_step_b1_l2048_fp16():
    _full_config(1, 1, [2048], 0, n_steps=2)


@pytest.mark.slow
def test_full_step_b8_l2400_fp16_and_batch_invariance():
    lengths = [2400] * 8
    _full_config(2, 8, lengths, 0)
    # batch-8 ids equal 8 independent batch-1 steps
    w = cached_model(FULL, 2)
    toks = make_tokens(FULL, 200, 8)
    dec, _, _ = setup_pair(FULL, w, 2, lengths, 0, 2402)
    _, ids8 = dec.step_host(toks, np.array(lengths, np.int32))
    dec.close()
    for b in (0, 5):
        d1 = z.Decoder(FULL, w, z.KV_F16, max_B=1, max_L=2402)
        k, v = make_kv_history(FULL, 2, b, 2400)
        d1.append_kv(0, k, v)
        _, id1 = d1.step_host(toks[b:b + 1], np.array([2400], np.int32))
        assert id1[0] == ids8[b]
        d1.close()


@pytest.mark.slow
def test_full_step_b1_l8192_q8_0():
    """The 36-layer model at B = 1 over an 8k Q8_0 cache (the sub-block-column
    projection kernel and the batch-of-one attention split)."""
    _full_config(4, 1, [8192], 1, n_steps=2)


@pytest.mark.slow
@pytest.mark.parametrize("kv_dtype", [0, 1])
def test_full_step_b8_long_context(kv_dtype):
    _full_config(3, 8, [6900, 8192, 6900, 8192, 7000, 8000, 6900, 8192], kv_dtype)


def test_trace_timeline():
    """Tracing records every launch (start <= release from the dependency
    wait <= end, each release after the previous launch's end); traced steps
    still match the oracle."""
    d = SMALL
    w = cached_model(d, 110)
    dec, om, kvs = setup_pair(d, w, 110, [20, 7], 0, 64)
    dec.set_trace(True)
    check_step(dec, om, kvs, make_tokens(d, 1100, 2), np.array([20, 7], np.int32), "traced kernels")
    tr = dec.step_trace().astype(np.int64)
    assert tr.shape == (3 + 5 * d.n_layers, 8)
    kinds = [z.KERNEL_KINDS[k] for k in tr[:, 3]]
    assert kinds[0] == "embed" and kinds[-2] == "gemm_lmhead" and kinds[-1] == "argmax"
    assert kinds.count("attention") == d.n_layers
    assert np.all(tr[:, 0] <= tr[:, 1]) and np.all(tr[:, 1] <= tr[:, 2])
    assert np.all(tr[1:, 1] >= tr[:-1, 2])
    dec.set_trace(False)
    assert dec.step_trace().size == 0
    dec.close()
