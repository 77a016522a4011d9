"""CPU pins of the oracle's attention and full decode step: special cases with
known answers, torch CPU library routines (scaled_dot_product_attention with
grouped-query heads, rms_norm, silu) composed independently, and the pages'
batch invariant (a batch of B equals B independent single steps)."""
import numpy as np
import pytest

import oracle
import synth
from synth.model import ModelDesc, make_kv_history, make_model, make_tokens

torch = pytest.importorskip("torch")
F = torch.nn.functional

TINY = ModelDesc(n_layers=2, hidden=512, n_q_heads=4, n_kv_heads=2, head_dim=128,
                 ffn=768, vocab=300)


def odesc(d: ModelDesc) -> oracle.Desc:
    return oracle.Desc(*d.astuple())


def _kv_with_history(d, seed, seq, L, max_L, kv_dtype):
    kv = oracle.KV(odesc(d), max_L, kv_dtype)
    if L:
        k, v = make_kv_history(d, seed, seq, L)
        kv.append(k, v)
    return kv


def _stored_tensor(kind, x16, xq, xs, x8, layer, n):
    """One stored tensor of one layer, dequantized by library routines and
    numpy: fp16 bits through numpy, Q8_0 codes times their fp16 scales, e4m3
    codes through torch's float8_e4m3fn."""
    if kind == oracle.KV_F16:
        return x16[layer, :n].view(np.float16).astype(np.float64)
    if kind == oracle.KV_Q8_0:
        s = xs[layer, :n].view(np.float16).astype(np.float64)
        return xq[layer, :n].astype(np.float64) * np.repeat(s, 32, axis=-1)
    return torch.from_numpy(np.ascontiguousarray(x8[layer, :n])).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _stored_kv(kv, layer, n):
    """Dequantized stored K, V of one layer: [n_kv, n, hd] float64."""
    k = _stored_tensor(kv.k_type, kv.k16, kv.kq, kv.ks, kv.k8, layer, n)
    v = _stored_tensor(kv.v_type, kv.v16, kv.vq, kv.vs, kv.v8, layer, n)
    return np.transpose(k, (1, 0, 2)), np.transpose(v, (1, 0, 2))


# ------------------------------------------------------------------ attention
@pytest.mark.parametrize("kv_dtype", [0, 1])
def test_attention_matches_torch_sdpa_gqa(kv_dtype):
    d = TINY
    L = 77
    kv = _kv_with_history(d, 5, 0, L, 128, kv_dtype)
    q = np.random.default_rng(2).standard_normal(d.n_q_heads * d.head_dim) * 1.3
    o = oracle.attention(odesc(d), kv, 1, L - 1, q)
    k, v = _stored_kv(kv, 1, L)
    ref = F.scaled_dot_product_attention(
        torch.from_numpy(q.reshape(1, d.n_q_heads, 1, d.head_dim)),
        torch.from_numpy(k[None]), torch.from_numpy(v[None]), enable_gqa=True)
    assert np.allclose(o, ref.numpy().reshape(-1), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("k_type", [0, 1, 2])
@pytest.mark.parametrize("v_type", [0, 1, 2])
def test_attention_with_separate_k_and_v_types(k_type, v_type):
    """Separate K and V cache types (fp16, Q8_0, FP8 e4m3 each): the oracle's
    attention equals torch's grouped-query SDPA over the stored tensors, each
    dequantized by its own type; a tensor read with the other's type, or an
    e4m3 code read as anything else, fails."""
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    d = TINY
    L = 45
    kv = _kv_with_history(d, 8, 0, L, 64, (k_type, v_type))
    q = np.random.default_rng(4).standard_normal(d.n_q_heads * d.head_dim) * 1.3
    o = oracle.attention(odesc(d), kv, 0, L - 1, q)
    k, v = _stored_kv(kv, 0, L)
    ref = F.scaled_dot_product_attention(
        torch.from_numpy(q.reshape(1, d.n_q_heads, 1, d.head_dim)),
        torch.from_numpy(k[None]), torch.from_numpy(v[None]), enable_gqa=True)
    assert np.allclose(o, ref.numpy().reshape(-1), rtol=1e-10, atol=1e-12)
    # the types really differ: an fp16 K read back as stored equals the history
    # only for the fp16 type
    kh, _ = make_kv_history(d, 8, 0, L)
    exact = np.array_equal(k, np.transpose(kh[0].view(np.float16).astype(np.float64), (1, 0, 2)))
    assert exact == (k_type == oracle.KV_F16)


@pytest.mark.parametrize("types", [(2, 2), (1, 0), (0, 2)])
def test_separate_cache_types_in_a_full_decode_step(types):
    """Decode steps over FP8 and mixed-type caches: a batch of two equals two
    single steps, bit for bit in the logits and in every stored array; the
    appended token sits where the step put it (position pos) and nowhere else."""
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    d = TINY
    w = make_model(d, 31)
    m = oracle.Model(odesc(d), w)
    toks = make_tokens(d, 32, 2)
    kvs = [_kv_with_history(d, 9, b, L, 48, types) for b, L in enumerate((5, 20))]
    pos = np.array([5, 20], np.int32)
    before = [{k: getattr(kv, k).copy() for k in ("k16", "v16", "kq", "vq", "ks", "vs", "k8", "v8")
               if getattr(kv, k) is not None} for kv in kvs]
    logits, ids, _ = oracle.decode_step(m, kvs, toks, pos)
    one = [_kv_with_history(d, 9, b, L, 48, types) for b, L in enumerate((5, 20))]
    for b in range(2):
        lb, ib, _ = oracle.decode_step(m, [one[b]], toks[b:b + 1], pos[b:b + 1])
        assert np.array_equal(lb[0], logits[b]) and ib[0] == ids[b]
        for name, old in before[b].items():
            new = getattr(kvs[b], name)
            assert np.array_equal(new, getattr(one[b], name)), name
            changed = np.nonzero(np.any((new != old).reshape(new.shape[0], new.shape[1], -1), axis=-1))[1]
            assert set(changed.tolist()) <= {int(pos[b])}, name
    assert np.isfinite(logits).all()


def test_attention_single_token_returns_v():
    d = TINY
    kv = _kv_with_history(d, 7, 0, 1, 16, 0)
    q = np.random.default_rng(3).standard_normal(d.n_q_heads * d.head_dim)
    o = oracle.attention(odesc(d), kv, 0, 0, q).reshape(d.n_q_heads, d.head_dim)
    v = kv.v16[0, 0].view(np.float16).astype(np.float64)      # [n_kv, hd]
    group = d.n_q_heads // d.n_kv_heads
    for h in range(d.n_q_heads):
        assert np.array_equal(o[h], v[h // group])


def test_attention_identical_keys_average_values():
    d = TINY
    L = 10
    kv = oracle.KV(odesc(d), 16, 0)
    k = np.tile(np.float16(0.25), (d.n_layers, L, d.n_kv_heads, d.head_dim)).view(np.uint16)
    vv = np.random.default_rng(4).standard_normal((d.n_layers, L, d.n_kv_heads, d.head_dim))
    v = vv.astype(np.float16).view(np.uint16)
    kv.append(k, v)
    q = np.random.default_rng(5).standard_normal(d.n_q_heads * d.head_dim)
    o = oracle.attention(odesc(d), kv, 1, L - 1, q).reshape(d.n_q_heads, d.head_dim)
    vmean = v[1].view(np.float16).astype(np.float64).mean(axis=0)   # [n_kv, hd]
    for h in range(d.n_q_heads):
        assert np.allclose(o[h], vmean[h // 2], rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------------ full step
def _dense(mat, rows, cols):
    return torch.from_numpy(oracle.q4k_dequant(mat).reshape(rows, cols).astype(np.float64))


def _rope_t(x, pos, theta):
    hd = x.shape[-1]
    half = hd // 2
    i = torch.arange(half, dtype=torch.float64)
    ang = pos * theta ** (-2.0 * i / hd)
    c, s = torch.cos(ang), torch.sin(ang)
    x0, x1 = x[..., :half], x[..., half:]
    return torch.cat([x0 * c - x1 * s, x1 * c + x0 * s], dim=-1)


def _f16_round(t):
    return t.to(torch.float16).to(torch.float64)


def _q8_round(t):
    """Round rows to fp16 and then through the (pinned) oracle Q8_0 quantizer."""
    bits = t.to(torch.float16).numpy().view(np.uint16).reshape(-1)
    sc, q = oracle.q8_0_quantize(bits)
    vals = q.astype(np.float64) * np.repeat(sc.view(np.float16).astype(np.float64), 32)
    return torch.from_numpy(vals.reshape(t.shape))


def torch_reference_step(d, w, kv, token, pos):
    """Independent torch CPU float64 composition of one decode step."""
    H, hd, nq, nkv = d.hidden, d.head_dim, d.n_q_heads, d.n_kv_heads
    E = _dense(w["embed"], d.vocab, H)
    x = E[token].to(torch.float32)
    rnd = _f16_round if kv.kv_dtype == 0 else _q8_round
    for l in range(d.n_layers):
        g1 = torch.from_numpy(w["attn_norm"][l].astype(np.float64))
        h = F.rms_norm(x.to(torch.float64), (H,), g1, eps=d.rms_eps)
        q = (_dense(w["wq"][l], nq * hd, H) @ h).to(torch.float32).to(torch.float64)
        k = (_dense(w["wk"][l], nkv * hd, H) @ h).to(torch.float32).to(torch.float64)
        v = (_dense(w["wv"][l], nkv * hd, H) @ h).to(torch.float32).to(torch.float64)
        q = _rope_t(q.view(nq, hd), pos, d.rope_theta)
        k = rnd(_rope_t(k.view(nkv, hd), pos, d.rope_theta))
        v = rnd(v.view(nkv, hd))
        kh, vh = _stored_kv(kv, l, pos)
        K = torch.cat([torch.from_numpy(kh), k[:, None]], dim=1)
        V = torch.cat([torch.from_numpy(vh), v[:, None]], dim=1)
        o = F.scaled_dot_product_attention(q[None, :, None], K[None], V[None], enable_gqa=True)
        y = (_dense(w["wo"][l], H, nq * hd) @ o.reshape(-1)).to(torch.float32)
        x = x + y
        g2 = torch.from_numpy(w["ffn_norm"][l].astype(np.float64))
        h = F.rms_norm(x.to(torch.float64), (H,), g2, eps=d.rms_eps)
        gt = (_dense(w["w_gate"][l], d.ffn, H) @ h).to(torch.float32).to(torch.float64)
        up = (_dense(w["w_up"][l], d.ffn, H) @ h).to(torch.float32).to(torch.float64)
        a = F.silu(gt) * up
        y = (_dense(w["w_down"][l], H, d.ffn) @ a).to(torch.float32)
        x = x + y
    gf = torch.from_numpy(w["final_norm"].astype(np.float64))
    h = F.rms_norm(x.to(torch.float64), (H,), gf, eps=d.rms_eps)
    return (E @ h).to(torch.float32).numpy(), x.numpy()


@pytest.mark.parametrize("kv_dtype", [0, 1])
def test_decode_step_matches_torch_composition(kv_dtype):
    d = TINY
    w = make_model(d, seed=11)
    model = oracle.Model(odesc(d), w)
    L = [37, 5]
    kvs = [_kv_with_history(d, 11, b, L[b], 64, kv_dtype) for b in range(2)]
    toks = make_tokens(d, 11, 2)
    refs = [torch_reference_step(d, w, kvs[b], int(toks[b]), L[b]) for b in range(2)]
    logits, ids, hidden = oracle.decode_step(model, kvs, toks, L, capture_hidden=True)
    for b in range(2):
        ref_logits, ref_x = refs[b]
        scale = np.abs(ref_logits).max()
        assert np.abs(logits[b] - ref_logits).max() <= 1e-5 * scale
        assert np.abs(hidden[b, -1] - ref_x).max() <= 1e-5 * np.abs(ref_x).max()
        assert ids[b] == int(np.argmax(ref_logits))


def test_decode_step_batch_equals_independent_steps():
    d = TINY
    w = make_model(d, seed=12)
    model = oracle.Model(odesc(d), w)
    L = [9, 30, 0]
    toks = make_tokens(d, 12, 3)
    kvs = [_kv_with_history(d, 12, b, L[b], 64, 1) for b in range(3)]
    lg, ids, hid = oracle.decode_step(model, kvs, toks, L, capture_hidden=True)
    for b in range(3):
        kv1 = _kv_with_history(d, 12, b, L[b], 64, 1)
        lg1, ids1, hid1 = oracle.decode_step(model, [kv1], toks[b:b + 1], L[b:b + 1],
                                             capture_hidden=True)
        assert np.array_equal(lg[b], lg1[0]) and ids[b] == ids1[0]
        assert np.array_equal(hid[b], hid1[0])
        assert np.array_equal(kvs[b].kq, kv1.kq) and np.array_equal(kvs[b].vs, kv1.vs)


def test_decode_step_appends_new_token():
    d = TINY
    w = make_model(d, seed=13)
    model = oracle.Model(odesc(d), w)
    kv = _kv_with_history(d, 13, 0, 4, 16, 0)
    before = kv.k16.copy()
    oracle.decode_step(model, [kv], make_tokens(d, 13, 1), [4])
    assert kv.len == 5
    assert np.array_equal(kv.k16[:, :4], before[:, :4])
    assert kv.k16[:, 4].any() and not kv.k16[:, 5:].any()
