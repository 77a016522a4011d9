"""Kernel-level parity on the GPU through the C ABI against the CPU oracle:
Q4_K repack/unpack (bit-exact), dequantization (bit-exact), the dense Q4_K
projection (matvec and mma.sync GEMM), the split-K attention over fp16, Q8_0
and FP8 caches (also K and V of different types), and encode-on-append
(bit-exact Q8_0 codes and scales, e4m3 codes)."""
import numpy as np
import pytest

import oracle
import synth
from synth.model import ModelDesc, make_kv_history, make_model
from tests.helpers import TOL, cached_model, gpu, needs_cuda, normwise

pytestmark = [gpu, needs_cuda]

torch = pytest.importorskip("torch")
import quantized_decode_step_02_gb300 as z  # noqa: E402

SMALL = ModelDesc(n_layers=2, hidden=512, n_q_heads=4, n_kv_heads=1, head_dim=128, ffn=1024,
                  vocab=1000)


def odesc(d):
    return oracle.Desc(*d.astuple())


@pytest.fixture(scope="module")
def small_dec():
    w = cached_model(SMALL, 21)
    dec = z.Decoder(SMALL, w, z.KV_F16, max_B=4, max_L=256)
    yield dec, w
    dec.close()


# ------------------------------------------------------------ repack/unpack
@pytest.mark.parametrize("which,name", [(z.T_EMBED, "embed"), (z.T_WQ, "wq"), (z.T_WK, "wk"),
                                        (z.T_WV, "wv"), (z.T_WO, "wo"), (z.T_GATE, "w_gate"),
                                        (z.T_UP, "w_up"), (z.T_DOWN, "w_down")])
def test_repack_roundtrip_bit_exact(small_dec, which, name):
    dec, w = small_dec
    for layer in range(SMALL.n_layers):
        src = w[name] if which == z.T_EMBED else w[name][layer]
        got = dec.export_q4k(which, layer, 0, src.shape[0])
        assert np.array_equal(got, src), (name, layer)
        if which == z.T_EMBED:
            break


@pytest.mark.parametrize("which,name", [(z.T_EMBED, "embed"), (z.T_WQ, "wq"), (z.T_GATE, "w_gate"),
                                        (z.T_UP, "w_up"), (z.T_DOWN, "w_down")])
def test_dequant_bit_exact_against_oracle(small_dec, which, name):
    dec, w = small_dec
    src = w[name] if which == z.T_EMBED else w[name][1]
    rows = [0, 1, 7, 8, 15, 16, src.shape[0] - 1]
    for r in rows:
        got = dec.dequant(which, 1, r, 1)[0]
        ref = oracle.q4k_dequant(src[r])
        assert np.array_equal(got.view(np.uint32), ref.view(np.uint32)), (name, r)


# ------------------------------------------------------------ dense Q4_K projection
def _gemm_case(N, K, B, impl, seed):
    W = synth.q4k_matrix(seed, 500, N, K, 0.02)
    x = synth.normal_f32(seed, 501, B * K).reshape(B, K)
    dev = torch.device("cuda")
    Wc = torch.from_numpy(W.reshape(-1)).to(dev)
    Wr = torch.empty(z.q4k_repacked_bytes(N, K), dtype=torch.uint8, device=dev)
    z.q4k_repack(Wc, N, K, Wr)
    xd = torch.from_numpy(x).to(dev)
    y = torch.full((B, N), float("nan"), dtype=torch.float32, device=dev)
    ws = torch.empty(z.q4k_gemm_workspace_bytes(K, B), dtype=torch.uint8, device=dev)
    z.q4k_gemm(Wr, N, K, xd, y, impl, ws)
    torch.cuda.synchronize()
    got = y.cpu().numpy()
    for b in range(B):
        ref = oracle.q4k_matvec(W, N, K, x[b].astype(np.float64))
        err = normwise(got[b], ref)
        assert err <= TOL, (N, K, B, impl, b, err)
    return got


def test_gemm_4096_square_batch1_all_kernels():
    # single-layer tiny step: Q4_K GEMV 4096 x 4096, N(0, 0.02) weights, x ~ N(0,1), seed 0
    a = _gemm_case(4096, 4096, 1, 2, 0)
    b = _gemm_case(4096, 4096, 1, 1, 0)
    c = _gemm_case(4096, 4096, 1, 3, 0)
    assert normwise(a, b) < 1e-4 and normwise(a, c) < 1e-4


@pytest.mark.parametrize("N,K", [(16, 512), (48, 1024), (4096, 14336), (151936 // 16 * 16, 512), (2048, 4096)])
def test_gemm_subblock_column_matvec_batch1(N, K):
    """impl 3 (raw codes as fp16 subnormal mma operands, one column per
    sub-block): ragged row tiles, long K, a split-K cluster and a grid of
    thousands of CTAs."""
    _gemm_case(N, K, 1, 3, N + K)


@pytest.mark.parametrize("N,K,B", [(16, 512, 1), (48, 1024, 3), (4096, 14336, 2), (6144, 4096, 8),
                                   (1024, 4096, 13), (512, 512, 32), (2048, 4096, 17)])
def test_gemm_mma_shapes_and_ragged_batch(N, K, B):
    _gemm_case(N, K, B, 2, N + K + B)


@pytest.mark.parametrize("B", [1, 2, 3, 4])
def test_gemm_matvec_batches(B):
    _gemm_case(2048, 2048, B, 1, 40 + B)


# ------------------------------------------------------------ attention
ATT = ModelDesc(n_layers=1, hidden=4096, n_q_heads=32, n_kv_heads=8, head_dim=128, ffn=512,
                vocab=256)


@pytest.mark.parametrize("kv_dtype", [0, 1, 2, (1, 0), (0, 2), (2, 1)])
@pytest.mark.parametrize("lengths", [[256], [1, 65, 700], [64, 128, 5000, 33]])
def test_attention_matches_oracle(kv_dtype, lengths):
    """GQA 32q/8kv, head_dim 128, over fp16, Q8_0 and FP8 caches (one type, or
    one for K and one for V); lengths are cached tokens per sequence and the
    query attends over all of them (positions = length - 1)."""
    B = len(lengths)
    w = cached_model(ATT, 3)
    max_L = max(lengths) + 1
    dec = z.Decoder(ATT, w, kv_dtype, max_B=B, max_L=max_L)
    seed = 30 + (kv_dtype if isinstance(kv_dtype, int) else 3 * kv_dtype[0] + kv_dtype[1])
    kvs = []
    for b, L in enumerate(lengths):
        k, v = make_kv_history(ATT, seed, b, L)
        dec.append_kv(b, k, v)
        kv = oracle.KV(odesc(ATT), max_L, kv_dtype)
        kv.append(k, v)
        kvs.append(kv)
    q = synth.normal_f32(9, 77, B * ATT.n_q_heads * ATT.head_dim, std=1.3).reshape(B, ATT.n_q_heads, 128)
    pos = np.array(lengths, np.int32) - 1
    o = dec.attention(0, q, pos)
    for b in range(B):
        ref = oracle.attention(odesc(ATT), kvs[b], 0, int(pos[b]), q[b].reshape(-1).astype(np.float64))
        ref = ref.reshape(ATT.n_q_heads, 128)
        for h in range(ATT.n_q_heads):
            err = normwise(o[b, h], ref[h])
            assert err <= TOL, (lengths, b, h, err)
    dec.close()


# ------------------------------------------------------------ KV append
def _special_fp16_rows(n_layers, n, nkv):
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((n_layers, n, nkv, 128)) * 2).astype(np.float16)
    x[0, 0, 0, :32] = 0.0                                       # all-zero block
    x[0, 0, 0, 32:64] = np.arange(-16, 16) * 0.5                # ties after scaling
    x[0, 1, 0, :32] = 127.0
    x[0, 1, 0, 0] = -127.0                                      # amax 127 -> d = 1
    x[0, 1, 0, 1:32] = np.arange(1, 32) + 0.5                   # ties to even at d = 1
    x[0, 2, 0, :32] = np.float16(6e-8)                          # fp16 subnormals
    x[0, 2, 0, 32:64] = -65504.0                                # fp16 extreme
    x[0, 2, 0, 40] = 1.0
    return x.view(np.uint16)


def _check_encoded(x16, codes, scales, kind):
    """Stored codes (and Q8_0 scales) of fp16 rows [t][g][128] against the oracle's encoders."""
    for t in range(x16.shape[0]):
        for g in range(x16.shape[1]):
            if kind == z.KV_F16:
                assert np.array_equal(codes[t, g], x16[t, g]), (t, g)
            elif kind == z.KV_Q8_0:
                rs, rq = oracle.q8_0_quantize(x16[t, g])
                assert np.array_equal(scales[t, g], rs) and np.array_equal(codes[t, g], rq), (t, g)
            else:
                ref = np.array([oracle.e4m3_from_half(int(h)) for h in x16[t, g]], np.uint8)
                assert np.array_equal(codes[t, g], ref), (t, g)


@pytest.mark.parametrize("types", [(1, 1), (2, 2), (1, 2), (2, 0), (0, 1)])
def test_append_encodes_bit_exact(types):
    """Bulk append through the C ABI encodes each tensor by its own type,
    bit-exact against the oracle's Q8_0 quantizer and e4m3 conversion (ties,
    all-zero blocks, subnormals, +-65504 saturating to +-448 in e4m3), across
    a page boundary."""
    d = SMALL
    w = cached_model(d, 21)
    dec = z.Decoder(d, w, types, max_B=2, max_L=160)
    k = _special_fp16_rows(d.n_layers, 70, d.n_kv_heads)
    v = np.flip(k, axis=-1).copy()
    dec.append_kv(1, k[:, :3], v[:, :3])
    dec.append_kv(1, k[:, 3:], v[:, 3:])   # the second call crosses into the second page
    for layer in range(d.n_layers):
        got = dec.read_kv(1, layer, 0, 70)
        ks = got[2] if len(got) == 4 else None
        vs = got[3] if len(got) == 4 else None
        _check_encoded(k[layer], got[0], ks, types[0])
        _check_encoded(v[layer], got[1], vs, types[1])
    assert dec.seq_len(1) == 70 and dec.seq_len(0) == 0
    assert (dec.block_table(1)[:2] >= 0).all() and (dec.block_table(1)[2:] < 0).all()
    assert (dec.block_table(0) < 0).all()
    dec.close()


def test_fp16_append_is_exact_and_capacity_is_enforced():
    d = SMALL
    dec = z.Decoder(d, cached_model(d, 21), z.KV_F16, max_B=1, max_L=10)
    k = _special_fp16_rows(d.n_layers, 10, d.n_kv_heads)
    dec.append_kv(0, k[:, :4], k[:, :4])
    dec.append_kv(0, k[:, 4:], k[:, 4:])
    kk, vv = dec.read_kv(0, 1, 0, 10)
    assert np.array_equal(kk, k[1]) and np.array_equal(vv, k[1])
    with pytest.raises(z.ZdecError) as e:
        dec.append_kv(0, k[:, :1], k[:, :1])
    assert e.value.status == -3
    with pytest.raises(z.ZdecError) as e:   # a full sequence cannot take a decode step
        dec.step_host(np.array([1], np.int32), np.array([10], np.int32))
    assert e.value.status == -3
    assert dec.seq_len(0) == 10
    dec.close()
