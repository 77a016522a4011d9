"""CPU pins of the oracle's building blocks against things other than itself:
library conversions (numpy float16), hand-built Q4_K / Q8_0 blocks with known
fields, closed forms, invariants and brute force on tiny shapes."""
import math

import numpy as np
import pytest

import oracle
import synth

RNG = np.random.default_rng(1234)


# ------------------------------------------------------------------ fp16
def test_half_to_float_all_patterns():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float32)
    got = np.array([oracle.half_to_float(int(p)) for p in pats], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _edge_values():
    tiny = [2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25,
            65504.0, 65519.99, 65520.0, 1e6, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,
            0.0, 1e-30, 2049.0, 2051.0, 0.1, 1 / 3]
    return np.array(tiny + [-v for v in tiny], dtype=np.float64)


def test_double_to_half_matches_numpy():
    xs = np.concatenate([_edge_values(), RNG.standard_normal(20000) * 10.0,
                         RNG.standard_normal(2000) * 1e-5, RNG.standard_normal(2000) * 3e4])
    ref = xs.astype(np.float16).view(np.uint16)
    got = np.array([oracle.double_to_half(float(v)) for v in xs], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_synth_f32_to_f16_matches_numpy():
    xs = np.concatenate([_edge_values().astype(np.float32),
                         RNG.standard_normal(5000).astype(np.float32) * 4,
                         (RNG.standard_normal(500) * 1e-6).astype(np.float32)])
    ref = xs.astype(np.float16).view(np.uint16)
    assert np.array_equal(synth.f32_to_f16_bits(xs), ref)


# ------------------------------------------------------------------ Q4_K
def _block(d_bits, dmin_bits, field_bytes, codes):
    b = np.zeros(144, np.uint8)
    b[0], b[1] = d_bits & 0xFF, d_bits >> 8
    b[2], b[3] = dmin_bits & 0xFF, dmin_bits >> 8
    b[4:16] = field_bytes
    b[16:] = codes
    return b


def test_q4k_unpack_hand_built_fields():
    # bytes 4..15 all ones -> every 6-bit field is 63
    d, dm, sc, mn, q = oracle.q4k_unpack(_block(0x3C00, 0x3800, [0xFF] * 12, [0] * 128))
    assert d == 1.0 and dm == 0.5
    assert list(sc) == [63] * 8 and list(mn) == [63] * 8
    # byte 4 = 0x3F: field 0 (sc_0) is bits 0..5 -> 63, nothing else
    fb = [0x3F] + [0] * 11
    _, _, sc, mn, _ = oracle.q4k_unpack(_block(0, 0, fb, [0] * 128))
    assert list(sc) == [63, 0, 0, 0, 0, 0, 0, 0] and list(mn) == [0] * 8
    # bits 6..11 (top 2 bits of byte 4, low nibble of byte 5) -> field 1 = sc_1
    fb = [0xC0, 0x0F] + [0] * 10
    _, _, sc, mn, _ = oracle.q4k_unpack(_block(0, 0, fb, [0] * 128))
    assert list(sc) == [0, 63, 0, 0, 0, 0, 0, 0]
    # field 8 = m_0 sits at bits 48..53 = byte 10 bits 0..5
    fb = [0] * 6 + [0x05] + [0] * 5
    _, _, sc, mn, _ = oracle.q4k_unpack(_block(0, 0, fb, [0] * 128))
    assert list(mn) == [5, 0, 0, 0, 0, 0, 0, 0] and list(sc) == [0] * 8
    # field 15 = m_7: bits 90..95 = byte 15 bits 2..7
    fb = [0] * 11 + [0xFC]
    _, _, sc, mn, _ = oracle.q4k_unpack(_block(0, 0, fb, [0] * 128))
    assert list(mn) == [0] * 7 + [63]
    # codes: byte t holds element 2t (low nibble) and 2t+1 (high nibble)
    codes = [0x21] + [0xF0] + [0] * 126
    _, _, _, _, q = oracle.q4k_unpack(_block(0, 0, [0] * 12, codes))
    assert list(q[:4]) == [1, 2, 0, 15] and not q[4:].any()


def _pack_fields(sc, mn):
    word = 0
    for i, v in enumerate(list(sc) + list(mn)):
        word |= (int(v) & 63) << (6 * i)
    return list(word.to_bytes(12, "little"))


def test_q4k_dequant_exact_small_integers():
    # d = 1, dmin = 0.5, sc_j = j+1, m_j = 2j, q_i = i % 16:
    # w_i = (j+1)*q_i - 0.5*2j = (j+1)*q_i - j, all exact in fp32
    sc = [j + 1 for j in range(8)]
    mn = [2 * j for j in range(8)]
    q = [i % 16 for i in range(256)]
    codes = [q[2 * t] | (q[2 * t + 1] << 4) for t in range(128)]
    blk = _block(0x3C00, 0x3800, _pack_fields(sc, mn), codes)
    w = oracle.q4k_dequant(blk)
    ref = np.array([(i // 32 + 1) * (i % 16) - (i // 32) for i in range(256)], np.float32)
    assert np.array_equal(w, ref)


def test_q4k_quantizer_roundtrip_error_bound():
    x = (RNG.standard_normal(256 * 64) * 0.02).astype(np.float32)
    blocks = synth.q4k_quantize(x).reshape(-1, 144)
    w = oracle.q4k_dequant(blocks)
    for b in range(blocks.shape[0]):
        d, dm, sc, mn, q = oracle.q4k_unpack(blocks[b])
        assert (q >= 0).all() and (q <= 15).all() and (sc <= 63).all() and (mn <= 63).all()
        for j in range(8):
            seg = slice(256 * b + 32 * j, 256 * b + 32 * j + 32)
            step = d * sc[j]
            # rounding to the grid costs at most half a step, plus the 6-bit
            # scale/min rounding which can stretch the grid by < 1/2 of a
            # scale unit per end: bound by one full step plus d and dmin
            err = np.abs(w[seg] - x[seg]).max()
            assert err <= step + d * 8 + dm * 1.0 + 1e-6, (b, j, err, step)
    rel = np.linalg.norm(w - x) / np.linalg.norm(x)
    assert rel < 0.12   # 4-bit quantization of Gaussian data


def test_q4k_matvec_against_numpy_dense():
    N, K = 16, 512
    W = synth.q4k_quantize((RNG.standard_normal(N * K) * 0.02).astype(np.float32))
    x = RNG.standard_normal(K)
    dense = oracle.q4k_dequant(W).reshape(N, K).astype(np.float64)
    y = oracle.q4k_matvec(W, N, K, x)
    assert np.allclose(y, dense @ x, rtol=1e-12, atol=1e-15)


def test_q4k_matvec_integer_matrix():
    # d=1, sc=1, dmin=0 -> W[n][k] = q (known integers); y = row sums of q * x
    N, K = 4, 256
    rows = []
    qs = []
    for n in range(N):
        q = [(n + 3 * i) % 16 for i in range(256)]
        qs.append(q)
        codes = [q[2 * t] | (q[2 * t + 1] << 4) for t in range(128)]
        rows.append(_block(0x3C00, 0x0000, _pack_fields([1] * 8, [0] * 8), codes))
    W = np.concatenate(rows)
    x = np.arange(256, dtype=np.float64) * 0.25
    y = oracle.q4k_matvec(W, N, K, x)
    for n in range(N):
        assert y[n] == sum(qs[n][i] * x[i] for i in range(256))


# ------------------------------------------------------------------ Q8_0
def f16(vals):
    return np.asarray(vals, dtype=np.float16).view(np.uint16)


def test_q8_0_integers_with_unit_scale():
    vals = np.arange(-127, 128, 8).tolist()
    vals = (vals + [127, -127] * 32)[:32]
    vals[0] = 127                               # amax = 127 -> d = 1
    sc, q = oracle.q8_0_quantize(f16(vals))
    assert sc[0] == 0x3C00
    assert list(q) == vals


def test_q8_0_ties_to_even_and_clamp():
    vals = [127.0, 0.5, 1.5, 2.5, -0.5, -1.5, -2.5, 3.5, -127.0] + [0.0] * 23
    sc, q = oracle.q8_0_quantize(f16(vals))
    assert list(q[:9]) == [127, 0, 2, 2, 0, -2, -2, 4, -127]
    assert q.min() >= -127


def test_q8_0_zero_block():
    sc, q = oracle.q8_0_quantize(np.zeros(32, np.uint16))
    assert sc[0] == 0 and not q.any()
    # negative zero is zero too
    sc, q = oracle.q8_0_quantize(np.full(32, 0x8000, np.uint16))
    assert sc[0] == 0 and not q.any()


def test_q8_0_multiples_of_scale_roundtrip():
    # amax = 63.5 -> d = 0.5 exactly; x = k*0.5 must come back as k
    ks = list(range(-127, 128, 8))[:31] + [127]
    sc, q = oracle.q8_0_quantize(f16([k * 0.5 for k in ks]))
    assert sc[0] == f16([0.5])[0]
    assert list(q) == ks
    assert all(oracle.q8_0_value(int(sc[0]), int(c)) == k * 0.5 for c, k in zip(q, ks))


def test_q8_0_codes_use_fp32_scale_not_fp16():
    # amax = 1 -> d32 = 1/127 (fp32) whose fp16 rounding differs; find a value
    # where dividing by d32 and by the fp16 scale round differently and check
    # the oracle follows the fp32 divisor.
    d32 = np.float32(1.0) / np.float32(127.0)
    d16 = np.float32(np.float16(d32))
    assert d16 != d32
    cands = np.arange(-1.0, 1.0, 2 ** -11, dtype=np.float32).astype(np.float16).astype(np.float32)
    by32 = np.rint(cands / d32)
    by16 = np.rint(cands / d16)
    diff = np.nonzero(by32 != by16)[0]
    assert diff.size > 0
    v = float(cands[diff[0]])
    sc, q = oracle.q8_0_quantize(f16([1.0, v] + [0.0] * 30))
    assert q[1] == by32[diff[0]] and q[0] == 127


# ------------------------------------------------------------------ norms, RoPE, silu
def test_rmsnorm_against_torch_and_constant_vector():
    torch = pytest.importorskip("torch")
    x = RNG.standard_normal(4096) * 3.0
    g = (1.0 + 0.1 * RNG.standard_normal(4096)).astype(np.float32)
    y = oracle.rmsnorm(x, g, 1e-6)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (4096,),
                                       torch.from_numpy(g.astype(np.float64)), eps=1e-6)
    assert np.allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)
    c = np.full(256, 2.0)
    y = oracle.rmsnorm(c, np.ones(256, np.float32), 0.0)
    assert np.allclose(y, 1.0, rtol=0, atol=1e-15)


def test_rope_pairs_and_angles():
    hd = 128
    for i in (0, 1, 17, 63):
        e = np.zeros(hd)
        e[i] = 1.0
        p = 37
        r = oracle.rope(e, p, 1e6)
        ang = p * 1e6 ** (-2.0 * i / hd)
        # rotate-half: component i goes to (i, i+64) as (cos, sin)
        assert math.isclose(r[i], math.cos(ang), abs_tol=1e-14)
        assert math.isclose(r[i + 64], math.sin(ang), abs_tol=1e-14)
        others = np.delete(r, [i, i + 64])
        assert not others.any()
    v = RNG.standard_normal(hd)
    assert np.array_equal(oracle.rope(v, 0, 1e6), v)
    assert math.isclose(np.linalg.norm(oracle.rope(v, 12345, 1e6)), np.linalg.norm(v), rel_tol=1e-13)


def test_rope_relative_position_invariant():
    q, k = RNG.standard_normal(128), RNG.standard_normal(128)
    a = np.dot(oracle.rope(q, 900, 1e6), oracle.rope(k, 700, 1e6))
    b = np.dot(oracle.rope(q, 200, 1e6), oracle.rope(k, 0, 1e6))
    assert math.isclose(a, b, rel_tol=1e-10, abs_tol=1e-12)


def test_silu_against_torch():
    torch = pytest.importorskip("torch")
    xs = np.linspace(-30, 30, 601)
    ref = torch.nn.functional.silu(torch.from_numpy(xs)).numpy()
    got = np.array([oracle.silu(v) for v in xs])
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-300)
    assert oracle.silu(0.0) == 0.0


def test_argmax_ties_lowest_index():
    x = np.zeros(1000, np.float32)
    x[[17, 400, 999]] = 5.0
    assert oracle.argmax(x) == 17
    x[3] = 5.0000005
    assert oracle.argmax(x) == 3


# ------------------------------------------------------------------ FP8 e4m3
def test_e4m3_worked_values():
    """The e4m3 format: bias 7, 3 mantissa bits, largest finite 448 (code 0x7E),
    smallest normal 2^-6 (0x08), smallest subnormal 2^-9 (0x01); nearest value,
    ties to the even code; magnitudes beyond 448 saturate (the hardware's
    satfinite conversion, the reading taken for an FP8 cache)."""
    h = oracle.double_to_half
    cases = {1.0: 0x38, -1.0: 0xB8, 448.0: 0x7E, 1000.0: 0x7E, -60000.0: 0xFE, 2.0 ** -6: 0x08,
             2.0 ** -9: 0x01, 2.0 ** -10: 0x00, 3 * 2.0 ** -10: 0x02, 1.0625: 0x38, 1.1875: 0x3A,
             0.0: 0x00, 240.0: 0x77, 0.5: 0x30}
    for v, code in cases.items():
        assert oracle.e4m3_from_half(h(v)) == code, (v, hex(code))
    assert oracle.e4m3_from_half(0x8000) == 0x80            # -0
    assert oracle.e4m3_from_half(0x7C00) == 0x7E            # +inf saturates
    assert oracle.e4m3_from_half(0x7E00) & 0x7F == 0x7F     # NaN stays NaN
    assert oracle.e4m3_value(0x7E) == 448.0 and oracle.e4m3_value(0x01) == 2.0 ** -9
    assert math.isnan(oracle.e4m3_value(0x7F)) and math.isnan(oracle.e4m3_value(0xFF))


def test_e4m3_matches_torch_on_every_in_range_half():
    """Every finite fp16 value below the rounding boundary to 480 (|x| < 464)
    converts as PyTorch's float8_e4m3fn cast does (nearest, ties to even); the
    decoded codes equal PyTorch's decode.  (Above it PyTorch returns NaN where
    the cache saturates.)"""
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16).astype(np.float32)
    keep = np.isfinite(vals) & (np.abs(vals) < 464.0)
    ref = torch.from_numpy(vals[keep]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.e4m3_from_half(int(b)) for b in bits[keep]], dtype=np.uint8)
    assert np.array_equal(got, ref)
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    dec = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle.e4m3_value(int(c)) for c in codes])
    assert np.array_equal(mine, dec)


def test_fp8_cache_bytes():
    from oracle.bytemodel import kv_bytes_per_token
    assert kv_bytes_per_token(36, 8, 128, "fp8") == 73_728 == kv_bytes_per_token(36, 8, 128, "f16") // 2
    assert kv_bytes_per_token(36, 8, 128, ("q8_0", "f16")) == (78_336 + 147_456) // 2
