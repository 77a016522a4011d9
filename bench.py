#!/usr/bin/env python
"""Benchmark of the batched Q4_K decode step (aggregate decode tok/s).

Default workload: the full synthetic 36-layer GQA model (hidden 4096, 32/8
heads of 128, SwiGLU 14336, tied 151,936-row LM head, all weights Q4_K from
N(0, 0.02), ~4.77 GB), B = 1 sequence holding L = 2048 cached fp16 tokens,
seed 1.  A step is one full decode step (every layer + LM head + argmax).

value: B * steps / device time of K back-to-back CUDA-graph steps, inputs
resident in HBM.  Every step streams ~5 GB (weights + KV), far more than the
129 MB L2, so no explicit flush is needed.
e2e: the same metric through the C ABI with host buffers (token ids and
positions copied in, argmax ids copied out, every step).
roofline: the dominant kernel kind (largest total time in one profiled
eager step): its algorithmic bytes per launch over its mean CUDA-event
launch time, against the measured HBM copy bandwidth in MEASURED_PEAKS.json.
cpu_baseline: the CPU oracle (plain C, fp64, OpenMP) on a bounded sample.

--impl reference times that oracle, as it stands, on the same workload.
Multi-GPU (torchrun): replicas only; each rank decodes its own batch.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from synth.model import FULL, ModelDesc, make_kv_history, make_model, make_tokens  # noqa: E402

METRIC = "aggregate decode tok/s"
KV_BYTES_PER_ELEM = {"f16": 2.0, "q8_0": 34.0 / 32.0, "fp8": 1.0}
KV_CODE = {"f16": 0, "q8_0": 1, "fp8": 2}


def kv_types(kv: str):
    """'t' (both tensors) or 'k_type:v_type' -> (k, v) type names."""
    parts = kv.split(":")
    k, v = (parts[0], parts[0]) if len(parts) == 1 else (parts[0], parts[1])
    if k not in KV_CODE or v not in KV_CODE:
        raise ValueError(f"bad KV type {kv!r}: use f16, q8_0, fp8 or K:V")
    return k, v


def kv_codes(kv: str):
    k, v = kv_types(kv)
    return KV_CODE[k], KV_CODE[v]


def args_parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--B", type=int, default=1)
    p.add_argument("--L", type=int, default=2048)
    p.add_argument("--kv", default="f16", help="cache type of K and V (f16, q8_0, fp8) or K:V, e.g. q8_0:f16")
    p.add_argument("--lengths", default=None,
                   help="comma-separated cached tokens per row (a ragged batch; overrides --B and --L)")
    p.add_argument("--seed", type=int, default=1)
    p.add_argument("--gemm-impl", type=int, default=0, help="0 auto, 1 matvec, 2 mma")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-targets", action="store_true",
                   help="skip the B {1,8} x L {2048,8192} x {f16,q8_0} target grid of the default line")
    p.add_argument("--sweep", action="store_true", help="B x L x kv grid, one JSON line per point")
    p.add_argument("--device-history", action="store_true",
                   help="one seeded device-side N(0,1) KV history shared by the sequences (fast setup)")
    p.add_argument("--layers", type=int, default=None, help="smaller model (profiling runs only)")
    p.add_argument("--trace", default=None, help="save the launch timeline of one step (.npy)")
    return p.parse_args()


def max_over_ranks(x: float, world: int, device) -> float:
    """The job's time is its slowest rank's: all-reduce MAX over the ranks."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def aggregate_tok_s(B: int, world: int, ms_per_step: float) -> float:
    """Replicas: every rank decodes its own batch of B, so the job advances
    B * world sequences per step of the slowest rank."""
    return B * world * 1000.0 / ms_per_step


def fit_time_model(points):
    """Least-squares fit of the pages' decode time model t(B, L) = a + B (b + k L)
    to measured (B, L, ms) points: features 1, B and B L.  Returns a, b and k in
    ms, ms and ms per token, and the largest relative residual."""
    import numpy as np
    P = np.asarray(points, dtype=np.float64)
    B, L, t = P[:, 0], P[:, 1], P[:, 2]
    A = np.stack([np.ones_like(B), B, B * L], axis=1)
    coef, *_ = np.linalg.lstsq(A, t, rcond=None)
    resid = np.abs(A @ coef - t) / t
    return {"a_ms": float(coef[0]), "b_ms": float(coef[1]), "k_ms_per_token": float(coef[2]),
            "max_rel_residual": float(resid.max()), "points": int(len(t))}


def ncu_traffic(kind: str, B: int, kv: str, impl: int):
    """DRAM bytes per launch of a kernel kind from a committed ncu capture
    (profiles/ncu_traffic.json), or None when no capture matches."""
    try:
        tab = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))["kernels"]
    except Exception:
        return None
    key = f"{kind}/B{B}/" + (kv if kind == "attention" else f"impl{impl}")
    return tab.get(key, {}).get("bytes")


def peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


def kv_bytes_per_token(d: ModelDesc, kv: str) -> float:
    k, v = kv_types(kv)
    return d.n_layers * d.n_kv_heads * d.head_dim * (KV_BYTES_PER_ELEM[k] + KV_BYTES_PER_ELEM[v])


def q4k_bytes(rows, cols):
    return rows * cols // 256 * 144


def weight_bytes(d: ModelDesc) -> int:
    qd, kvd = d.n_q_heads * d.head_dim, d.n_kv_heads * d.head_dim
    per = q4k_bytes(qd + 2 * kvd, d.hidden) + q4k_bytes(d.hidden, qd) + 2 * q4k_bytes(d.ffn, d.hidden) \
        + q4k_bytes(d.hidden, d.ffn)
    return d.n_layers * per + q4k_bytes(d.vocab, d.hidden) + (2 * d.n_layers + 1) * d.hidden * 4


def step_bytes(d: ModelDesc, B: int, L: float, kv: str) -> float:
    """Algorithmic HBM bytes of one step: weights once, each sequence's KV read
    over L+1 tokens and one token written, embedding rows and logits.  L is
    the mean cached length of the B rows."""
    k = kv_bytes_per_token(d, kv)
    return weight_bytes(d) + B * (L + 2) * k + B * (d.hidden // 256 * 144 + 4 * d.vocab)


def kernel_bytes(d: ModelDesc, kind: str, B: int, L: float, kv: str) -> float:
    """Algorithmic bytes of one launch of a kernel kind (weights or KV it must
    read, activations in, results out)."""
    H, F, qd, kvd = d.hidden, d.ffn, d.n_q_heads * d.head_dim, d.n_kv_heads * d.head_dim
    act = lambda k_in, n_out: B * (2 * k_in + k_in // 32 * 4 + 4 * n_out)
    if kind == "gemm_qkv":
        return q4k_bytes(qd + 2 * kvd, H) + act(H, qd + 2 * kvd)
    if kind == "gemm_o":
        return q4k_bytes(H, qd) + act(qd, 2 * H)
    if kind == "gemm_gateup":
        return 2 * q4k_bytes(F, H) + act(H, F)
    if kind == "gemm_down":
        return q4k_bytes(H, F) + act(F, 2 * H)
    if kind == "gemm_lmhead":
        return q4k_bytes(d.vocab, H) + act(H, d.vocab)
    if kind == "attention":
        per_tok_layer = kv_bytes_per_token(d, kv) / d.n_layers
        return B * (L + 2) * per_tok_layer + B * (qd + 2 * kvd + qd) * 4
    return 0.0


class Clocks:
    """nvidia-smi sampler running during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev: int):
        self.dev, self.p = dev, None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                       "-lms", "200", "-i", str(self.dev)], stdout=subprocess.PIPE,
                                      stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.p:
            time.sleep(0.25)
            self.p.terminate()
            try:
                self.out, _ = self.p.communicate(timeout=5)
            except Exception:
                self.p.kill()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def workload_config(a, desc, world):
    """The `config` object both arms print (identical keys and values)."""
    shape = f"lengths {a.lengths}" if a.lengths else f"L={a.L}"
    return {"workload": f"decode step B={a.B} {shape} {a.kv} KV, {desc.n_layers}-layer GQA Q4_K synthetic model",
            "B": a.B, "L": a.L, "kv": a.kv, "model_layers": desc.n_layers, "seed": a.seed,
            "lengths": a.lengths,
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": "no flush: every step streams >4.7 GB, far larger than the 129 MB L2"}


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or ''."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        for line in open("/proc/cpuinfo"):
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return ""


def oracle_step_sample(desc, w, seed, B, L, kv, budget_s=20.0, max_steps=None):
    """Time the CPU oracle on up to B of the workload's sequences for about
    budget_s seconds; returns (tok/s, threads, description)."""
    import oracle
    od = oracle.Desc(*desc.astuple())
    om = oracle.Model(od, w)
    kvd = kv_codes(kv)
    nb = 1   # one sequence per sampled step: the oracle computes rows independently
    kvs = []
    steps_possible = max_steps or 64
    for b in range(nb):
        kvo = oracle.KV(od, L + steps_possible + 1, kvd)
        k, v = make_kv_history(desc, seed, b, L)
        kvo.append(k, v)
        kvs.append(kvo)
    t0 = time.perf_counter()
    done = 0
    while True:
        toks = make_tokens(desc, seed * 1000 + 500 + done, nb)
        oracle.decode_step(om, kvs, toks, [kvs[0].len])
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_steps and done >= max_steps) or done >= steps_possible:
            break
    threads = int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))
    return done * nb / el, threads, f"{done} oracle step(s) of 1 sequence (B={B}, L={L}, {kv} KV), {el:.1f} s"


def run_reference(a, rank, world):
    desc = FULL if a.layers is None else FULL.with_(n_layers=a.layers)
    if rank != 0:
        return
    w = make_model(desc, a.seed)
    import oracle  # noqa: F401
    # a.warmup untimed steps; each timed step is one oracle step of one sequence
    if a.warmup > 0:
        oracle_step_sample(desc, w, a.seed, a.B, a.L, a.kv, budget_s=0.0, max_steps=a.warmup)
    per_step = []
    for i in range(a.steps):
        v, threads, _ = oracle_step_sample(desc, w, a.seed, a.B, a.L, a.kv, budget_s=0.0, max_steps=1)
        per_step.append(1.0 / v)
    el = sum(per_step)
    value = a.steps / el
    line = {"metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": a.gpus, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": 1000 * el / a.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference", "config": workload_config(a, desc, world),
            "cpu_baseline": {"kind": "oracle", "value": value, "unit": "tok/s", "cores": threads,
                             "cpu": cpu_model(),
                             "sample": f"{a.steps} timed oracle step(s) of one sequence of the workload "
                                       f"after {a.warmup} untimed"},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def time_steps(dec, B, lengths, n_warm, n_timed, stream, world, desc, seed, logits):
    """n_warm untimed then n_timed CUDA-event-timed steps of rows 0..B-1 whose
    caches hold lengths[b] tokens; returns (ms per step, clock summary)."""
    import torch
    n_total = n_warm + n_timed
    toks = [torch.from_numpy(make_tokens(desc, seed * 1000 + i, B)).cuda() for i in range(n_total)]
    pos = [torch.tensor([n + i for n in lengths], dtype=torch.int32, device="cuda") for i in range(n_total)]
    ids = torch.empty(B, dtype=torch.int32, device="cuda")
    for i in range(n_warm):
        dec.step(toks[i], pos[i], logits, ids)
    dec.sync()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with Clocks(torch.cuda.current_device()) as clk:
        ev0.record(stream)
        for i in range(n_warm, n_total):
            dec.step(toks[i], pos[i], logits, ids)
        ev1.record(stream)
        torch.cuda.synchronize()
    dec.sync()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / n_timed, world, "cuda")
    if world > 1:
        torch.distributed.barrier()
    return ms, clk.summary()


def bench_point(a, desc, w, B, L, kv, rank, world, full_report=True, dev_hist=None, lengths=None):
    """One measured configuration: B rows of L cached tokens each (or of
    `lengths` tokens: a ragged batch).  dev_hist: (k, v) fp16 CUDA tensors
    [n_layers][>= max L][n_kv][hd] appended to every sequence instead of the
    seeded host history (timing does not depend on values).  The timed steps
    write logits [B][vocab] and ids, as step_bytes counts."""
    import torch
    import quantized_decode_step_02_gb300 as z
    stream = torch.cuda.Stream()
    lengths = list(lengths) if lengths is not None else [L] * B
    Lmax, Lmean = max(lengths), sum(lengths) / len(lengths)
    extra = a.warmup + a.steps + 4 + (0 if a.no_e2e else a.warmup + a.steps)
    dec = z.Decoder(desc, w, kv_codes(kv), max_B=B, max_L=Lmax + extra + 2, stream=stream.cuda_stream)
    if a.gemm_impl:
        dec.set_gemm_impl(a.gemm_impl)
    if dev_hist is not None:
        torch.cuda.synchronize()
        for b in range(B):   # one contiguous copy each, alive until its append has run
            k, v = dev_hist[0][:, :lengths[b]].contiguous(), dev_hist[1][:, :lengths[b]].contiguous()
            dec.append_kv(b, k, v)
            del k, v
        dec.sync()
    else:
        for b in range(B):
            k, v = make_kv_history(desc, a.seed, b, lengths[b])
            dec.append_kv(b, k, v)
    logits = torch.empty((B, desc.vocab), dtype=torch.float32, device="cuda")
    ms, clocks = time_steps(dec, B, lengths, a.warmup, a.steps, stream, world, desc, a.seed, logits)
    n_total = a.warmup + a.steps
    Lmid = Lmean + a.warmup + a.steps / 2
    res = {"B": B, "L": L if len(set(lengths)) == 1 else lengths, "kv": kv, "ms_per_step": ms,
           "tok_s": aggregate_tok_s(B, world, ms), "step_bytes": step_bytes(desc, B, Lmid, kv),
           "kernels_per_step": dec.info()["kernels_per_step"], "clocks": clocks,
           "attn_cluster": dec.info()["attn_splits"], "attn_segments": dec.info()["attn_segments"]}
    res["step_gbs"] = res["step_bytes"] / (ms * 1e-3) / 1e9
    i = n_total
    toks = [torch.from_numpy(make_tokens(desc, a.seed * 1000 + 400 + j, B)).cuda() for j in range(2)]
    ids = torch.empty(B, dtype=torch.int32, device="cuda")
    at = lambda j: torch.tensor([n + j for n in lengths], dtype=torch.int32, device="cuda")
    if a.trace:   # one traced step (not timed)
        dec.set_trace(True)
        dec.step(toks[0], at(i), logits, ids)
        np.save(a.trace, dec.step_trace())
        dec.set_trace(False)
        i += 1
    # ---- per-launch profile of one eager step (CUDA events on the library stream)
    prof = dec.profile_step(toks[1], at(i), logits, ids)
    by_kind = {}
    for kind, t in prof:
        by_kind.setdefault(kind, []).append(t)
    res["profile_ms"] = {k: {"launches": len(v), "total_ms": sum(v), "avg_ms": sum(v) / len(v)}
                         for k, v in by_kind.items()}
    # ---- end to end through the C ABI with host buffers: token ids and
    # positions in, argmax ids out, every step (the LM head writes no logits
    # buffer on this path: the ids are the step's result)
    if not a.no_e2e:
        base = i + 1
        ht = [make_tokens(desc, a.seed * 1000 + 700 + j, B) for j in range(n_total)]
        hp = [np.array([n + base + j for n in lengths], np.int32) for j in range(n_total)]
        for j in range(a.warmup):
            dec.step_host(ht[j], hp[j])
        t0 = time.perf_counter()
        for j in range(a.warmup, n_total):
            dec.step_host(ht[j], hp[j])
        el = max_over_ranks(time.perf_counter() - t0, world, "cuda")
        res["e2e"] = {"value": aggregate_tok_s(B, world, 1000.0 * el / a.steps), "unit": "tok/s",
                      "h2d_bytes_per_step": 8 * B, "d2h_bytes_per_step": 4 * B}
    dec.close()
    return res


def target_grid(a, desc, w, world, hbm_peak):
    """The target cells B in {1, 8} x L in {2048, 8192} x {f16, q8_0}: one
    decoder per KV type (max_B = 8), a seeded device-side N(0,1) history
    appended to every sequence of a cell, then the same warm-up and timed
    steps as the headline.  Each cell: ms/step, tok/s, the bytes-moved
    fraction of the measured HBM bandwidth, and the clocks of its timed region."""
    import torch
    import quantized_decode_step_02_gb300 as z
    Lmax = 8192
    gen = torch.Generator(device="cuda").manual_seed(10)
    shape = (desc.n_layers, Lmax, desc.n_kv_heads, desc.head_dim)
    hist = (torch.randn(shape, generator=gen, device="cuda", dtype=torch.float16),
            torch.randn(shape, generator=gen, device="cuda", dtype=torch.float16))
    cells = []
    n = a.warmup + a.steps
    for kv in ("f16", "q8_0"):
        stream = torch.cuda.Stream()
        dec = z.Decoder(desc, w, kv_codes(kv), max_B=8, max_L=Lmax + n + 2, stream=stream.cuda_stream)
        for L in (2048, 8192):
            k, v = hist[0][:, :L].contiguous(), hist[1][:, :L].contiguous()
            for B in (1, 8):
                for b in range(8):
                    dec.reset_seq(b)
                torch.cuda.synchronize()
                for b in range(B):
                    dec.append_kv(b, k, v)
                dec.sync()
                logits = torch.empty((B, desc.vocab), dtype=torch.float32, device="cuda")
                ms, clk = time_steps(dec, B, [L] * B, a.warmup, a.steps, stream, world, desc, a.seed, logits)
                sb = step_bytes(desc, B, L + a.warmup + a.steps / 2, kv)
                gbs = sb / (ms * 1e-3) / 1e9
                cells.append({"B": B, "L": L, "kv": kv, "ms_per_step": round(ms, 4),
                              "tok_s": round(aggregate_tok_s(B, world, ms), 1),
                              "step_hbm_gbs": round(gbs, 1), "step_frac_of_measured_hbm": round(gbs / hbm_peak, 4),
                              "step_frac_of_8tbs": round(gbs / 8000.0, 4), "clocks": clk})
            del k, v
        dec.close()
    del hist
    return cells


def main():
    a = args_parse()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    if a.impl == "reference":
        return run_reference(a, rank, world)
    import torch
    torch.cuda.set_device(local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    desc = FULL if a.layers is None else FULL.with_(n_layers=a.layers)
    t0 = time.time()
    w = make_model(desc, a.seed)
    gen_s = time.time() - t0
    def device_history(L):
        import torch
        gen = torch.Generator(device="cuda").manual_seed(10)
        shape = (desc.n_layers, L, desc.n_kv_heads, desc.head_dim)
        return (torch.randn(shape, generator=gen, device="cuda", dtype=torch.float16),
                torch.randn(shape, generator=gen, device="cuda", dtype=torch.float16))

    if a.sweep:
        # B x L x kv grid on a seeded device-side N(0,1) history (one per L,
        # shared by the sequences), then the projection-kernel switch point
        hist = device_history(32768)
        for kv in ("f16", "q8_0", "fp8"):
            pts = []
            for B in (1, 4, 8, 16, 32):
                for L in (2048, 8192, 16384, 32768):
                    r = bench_point(a, desc, w, B, L, kv, rank, world, dev_hist=hist)
                    pts.append((B, L, r["ms_per_step"]))
                    if rank == 0:
                        print(json.dumps({"sweep": True, **{k: v for k, v in r.items() if k != "profile_ms"},
                                          "profile_ms": r["profile_ms"]}), flush=True)
            if rank == 0:   # the pages' time model t(B, L) = a + B (b + k L), fitted to this kv type's grid
                print(json.dumps({"time_model": True, "kv": kv, **fit_time_model(pts)}), flush=True)
        for B in (1, 2, 3, 4):
            for impl in ((1, 2, 3) if B == 1 else (1, 2)):
                a.gemm_impl = impl
                r = bench_point(a, desc, w, B, 2048, "f16", rank, world, dev_hist=hist)
                if rank == 0:
                    print(json.dumps({"switch": True, "impl": impl, **{k: v for k, v in r.items() if k != "profile_ms"},
                                      "profile_ms": r["profile_ms"]}), flush=True)
        a.gemm_impl = 0
        return
    lengths = [int(x) for x in a.lengths.split(",")] if a.lengths else None
    if lengths:
        a.B, a.L = len(lengths), int(round(sum(lengths) / len(lengths)))
    r = bench_point(a, desc, w, a.B, a.L, a.kv, rank, world, lengths=lengths,
                    dev_hist=device_history(max(lengths) if lengths else a.L) if a.device_history else None)
    if rank != 0:
        return
    pk = peaks() or {}
    hbm_peak = pk.get("hbm_gbs", 6800.0)
    peak_src = "measured" if "hbm_gbs" in pk else "fallback"
    prof = r["profile_ms"]
    dom = max((k for k in prof if k.startswith("gemm") or k == "attention"), key=lambda k: prof[k]["total_ms"])
    launch_ms, launches = prof[dom]["avg_ms"], prof[dom]["launches"]
    Lmid = a.L + a.warmup + a.steps + 0.5
    kb = kernel_bytes(desc, dom, a.B, Lmid, a.kv)
    achieved = kb / (launch_ms * 1e-3) / 1e9
    impl = a.gemm_impl or (3 if a.B == 1 else 2)
    roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
            "frac": achieved / hbm_peak, "peak_source": peak_src,
            "traffic": ncu_traffic(dom, a.B, a.kv, impl),
            "bytes_per_launch": kb, "avg_launch_ms": launch_ms, "launches_per_step": launches}
    targets = None
    if not a.no_targets and a.layers is None and world == 1:
        targets = target_grid(a, desc, w, world, hbm_peak)
    cpu = None
    if not a.no_cpu_baseline and world == 1:
        import oracle
        v, threads, sample = oracle_step_sample(desc, w, a.seed, a.B, a.L, a.kv, budget_s=15.0)
        cpu = {"value": v, "unit": "tok/s", "cores": threads, "kind": "oracle", "sample": sample,
               "cpu": cpu_model()}
        # the same oracle on one core: one step (about cores x the time above)
        oracle.set_threads(1)
        v1, _, sample1 = oracle_step_sample(desc, w, a.seed, a.B, a.L, a.kv, budget_s=0.0, max_steps=1)
        oracle.set_threads(threads)
        cpu["single_thread"] = {"value": v1, "unit": "tok/s", "cores": 1, "sample": sample1}
    line = {"metric": METRIC, "value": r["tok_s"], "unit": "tok/s", "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "q4_k weights, f16 activations, f32 accumulate",
            "data": "synthetic (seeded N(0,0.02) weights quantized to Q4_K, N(0,1) fp16 KV history)",
            "config": workload_config(a, desc, world),
            "step": {"bytes": r["step_bytes"], "hbm_gbs": r["step_gbs"],
                     "lengths": lengths, "attn_cluster": r["attn_cluster"], "attn_segments": r["attn_segments"],
                     "frac_of_measured_hbm": r["step_gbs"] / hbm_peak, "frac_of_8tbs": r["step_gbs"] / 8000.0,
                     "bytes_counted": "weights once + per sequence (L+2) KV tokens + embedding row + fp32 logits "
                                      "(the timed steps write logits)",
                     "model_gen_s": round(gen_s, 1)},
            "roofline": roof, "cpu_baseline": cpu, "e2e": r.get("e2e"),
            "gpu_launches": r["kernels_per_step"] * a.steps, "clocks": r["clocks"],
            "targets": targets, "profile_ms": prof}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
