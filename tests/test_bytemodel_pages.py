"""The byte model of a batched decode step against the numbers the pages print
(tests/golden/byte_model_pages.json, each value cited to its page)."""
import json
import os

import pytest

from oracle import bytemodel as bm

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "byte_model_pages.json")))


def test_kv_bytes_per_token_exact_and_q8_ratio():
    g = GOLD["kv_bytes_per_token_exact"]
    f16 = bm.kv_bytes_per_token(g["n_layers"], g["n_kv_heads"], g["head_dim"], "f16")
    q8 = bm.kv_bytes_per_token(g["n_layers"], g["n_kv_heads"], g["head_dim"], "q8_0")
    assert f16 == g["f16"] == 147456
    assert q8 == g["q8_0"] == 78336
    assert q8 / f16 == 34 / 64          # Q8_0 "halves" KV up to its fp16 scale per 32
    assert abs(f16 - GOLD["kv_bytes_per_token_f16"]["value"]) / f16 < 0.01


def test_crossover_b8_page2():
    W, k = GOLD["weights_bytes"]["value"], GOLD["kv_bytes_per_token_f16"]["value"]
    g = GOLD["crossover_b8_f16"]
    assert abs(bm.crossover(W, 8, k) - g["value"]) <= g["tolerance"]
    # at the crossover the private KV read equals the shared weight read
    L = bm.crossover(W, 8, k)
    assert abs(8 * L * k - W) / W < 1e-12


def test_speedup_table_page2():
    W, k = GOLD["weights_bytes"]["value"], GOLD["kv_bytes_per_token_f16"]["value"]
    for L, printed in GOLD["speedup_b8_table"]["rows"]:
        s = bm.speedup(W, 8, L, k)
        assert abs(s - printed) <= GOLD["speedup_b8_table"]["tolerance"], (L, s, printed)
    assert bm.speedup(W, 8, 0, k) == 8.0


def test_crossover_page3_fp16_and_q8():
    g = GOLD["crossover_b8_f16_p3"]
    W = g["weights_mb"] * 1e6
    k = g["kv_mb_per_token"] * 1e6
    assert abs(bm.crossover(W, 8, k) - g["value"]) <= g["tolerance"]
    q8 = GOLD["crossover_b8_q8_p3"]
    assert abs(bm.crossover(W, 8, k / 2) - q8["value"]) / q8["value"] <= q8["relative_tolerance"]


def test_fig1_time_model_page1():
    g = GOLD["fig1_step_ms"]
    for B, t, agg, per in zip(g["batch"], g["step_ms"], g["aggregate_tok_s"],
                              g["per_sequence_tok_s"]):
        model_t = bm.time_model_ms(B, 0, per_seq_ms=1.1, k_ms_per_token=0.0)
        assert abs(model_t - t) < 1e-9
        assert abs(1000.0 * B / model_t - agg) < 0.6
        assert abs(1000.0 / model_t - per) < 0.06


def test_ceiling_table_page3():
    rows = GOLD["ceiling_b8_table"]["rows_ctx_f16_q8"]
    # fit the per-token KV time k from the first printed point, check the rest
    ctx0, f16_0, _ = rows[0]
    t0 = 8000.0 / f16_0
    k = ((t0 - 16.9) / 8 - 1.1) / ctx0
    for ctx, f16, q8 in rows:
        if f16 is not None:
            assert abs(8000.0 / bm.time_model_ms(8, ctx, k_ms_per_token=k) - f16) < 1.5
        assert abs(8000.0 / bm.time_model_ms(8, ctx, k_ms_per_token=k / 2) - q8) < 1.5


def test_weight_bytes_of_synthetic_model():
    W = bm.weight_bytes()
    assert W == 4_767_858_688
    assert bm.weight_bytes(with_norms=False) == 4_766_662_656
    # step bytes are linear in B and L, and the weight term is independent of B
    k = 147456
    assert bm.step_bytes(W, 8, 2048, k) - bm.step_bytes(W, 4, 2048, k) == 4 * 2048 * k
    assert bm.step_bytes(W, 1, 0, k) == W


def test_time_model_fit_recovers_its_coefficients():
    """bench.py fits the pages' time model t(B, L) = a + B (b + k L) to a sweep;
    on points generated from known coefficients (the pages' 16.9 ms and 1.1 ms,
    with a per-token k) the fit returns them, and a perturbed point shows up
    as the largest relative residual."""
    import bench
    a, b, k = 16.9, 1.1, 2.0e-4
    pts = [(B, L, a + B * (b + k * L)) for B in (1, 4, 8, 16, 32) for L in (2048, 8192, 16384, 32768)]
    fit = bench.fit_time_model(pts)
    assert abs(fit["a_ms"] - a) < 1e-9 * a and abs(fit["b_ms"] - b) < 1e-9 and abs(fit["k_ms_per_token"] - k) < 1e-13
    assert fit["max_rel_residual"] < 1e-12 and fit["points"] == 20
    B0, L0, t0 = pts[7]
    pts[7] = (B0, L0, t0 * 1.1)
    assert bench.fit_time_model(pts)["max_rel_residual"] > 0.05


def test_bench_byte_accounting_matches_the_byte_model():
    """The roofline numerators bench.py reports come from the same closed forms
    the pages state: its weight stream is the byte model's W (4,767,858,688 B
    for the 36-layer model), its KV bytes per token are 147,456 (fp16) and
    78,336 (Q8_0), the five projection launches of a step add up to the Q4_K
    part of W, and a step's bytes are the model's W + B L k plus the token the
    step appends and reads, the embedding rows and the logits."""
    import bench
    from synth.model import FULL as d
    W = bm.weight_bytes()
    assert bench.weight_bytes(d) == W == 4_767_858_688
    for kv, k in (("f16", 147_456), ("q8_0", 78_336)):
        assert bench.kv_bytes_per_token(d, kv) == k == bm.kv_bytes_per_token(36, 8, 128, kv)
    per_layer = sum(bench.kernel_bytes(d, kind, 0, 0, "f16")
                    for kind in ("gemm_qkv", "gemm_o", "gemm_gateup", "gemm_down"))
    lm = bench.kernel_bytes(d, "gemm_lmhead", 0, 0, "f16")
    assert d.n_layers * per_layer + lm == bm.weight_bytes(with_norms=False)
    for B, L in ((1, 2048), (8, 2400), (32, 32768)):
        k = bm.kv_bytes_per_token(36, 8, 128, "f16")
        extra = B * k + B * (d.hidden // 256 * 144 + 4 * d.vocab)
        assert bench.step_bytes(d, B, L, "f16") == bm.step_bytes(W, B, L + 1, k) + extra
    # per layer, the attention launch moves 1/36 of the step's KV bytes
    att = bench.kernel_bytes(d, "attention", 8, 2400, "q8_0")
    assert att - 8 * (2 * 4096 + 2 * 1024) * 4 == pytest.approx(8 * 2402 * 78_336 / 36)


def test_traffic_table_matches_its_captures():
    """Every ncu traffic entry bench.py may report names a committed capture
    summary under profiles/, and its DRAM bytes lie between what must come from
    HBM (the weights, or the KV pages read) and the kernel's algorithmic bytes
    plus 1 % (more would mean re-reads; less, an entry of another launch).
    Activations and outputs may stay in L2, so they only bound from above."""
    import bench
    from synth.model import FULL as d
    root = os.path.dirname(os.path.dirname(__file__))
    tab = json.load(open(os.path.join(root, "profiles", "ncu_traffic.json")))["kernels"]
    assert tab, "no traffic entries"
    for key, ent in tab.items():
        kind, bclass, tail = key.split("/")
        assert os.path.exists(os.path.join(root, ent["source"])), ent["source"]
        B = int(bclass[1:])
        if kind == "attention":
            # one layer's KV in whole 64-token pages: the captures ran at
            # L = 2048 (B = 1) and L = 8192 (B = 8), in their second step
            L = 2048 if B == 1 else 8192
            pages = -(-(L + 2) // 64)
            lo = B * pages * 64 * bench.kv_bytes_per_token(d, tail) / d.n_layers
            hi = 1.01 * lo + B * 16 * 1024 * 4 + 4e6
        else:
            lo = bench.kernel_bytes(d, kind, 0, 0, "f16")   # the matrix alone
            hi = 1.01 * bench.kernel_bytes(d, kind, B, 0, "f16")
            assert bench.ncu_traffic(kind, B, "f16", int(tail[4:])) == ent["bytes"]
        assert lo <= ent["bytes"] <= hi, (key, ent["bytes"], lo, hi)
