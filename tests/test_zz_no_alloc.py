"""The allocation-free projection zdec_q4k_gemm_static against the workspace
entry point zdec_q4k_gemm: bitwise-equal outputs on two consecutive calls (so
nothing left in the library's static scratch by one call leaks into the
next), both kernels, a ragged batch and the largest K*B the scratch holds;
and the size check, which answers without a GPU.  Named so that it is
collected last: it must pass alone and after every other test."""
import ctypes

import numpy as np
import pytest

import synth
from tests.helpers import gpu, needs_cuda

import quantized_decode_step_02_gb300 as z


def test_static_gemm_rejects_oversize_before_any_cuda_call():
    lib = z.load_library()
    dummy = ctypes.c_void_p(256)
    K, B = 16384, 17                       # K*B = 278528 > 262144
    assert K * B > z.Q4K_GEMM_STATIC_MAX_KB
    assert lib.zdec_q4k_gemm_static(dummy, 4096, K, dummy, B, dummy, 2, None) == -1
    msg = lib.zdec_last_global_error().decode()
    assert "exceeds" in msg and str(z.Q4K_GEMM_STATIC_MAX_KB) in msg
    assert lib.zdec_q4k_gemm_static(None, 4096, 4096, dummy, 1, dummy, 2, None) == -1
    assert lib.zdec_q4k_gemm_static(dummy, 4096, 4096, dummy, 5, dummy, 1, None) == -5
    assert lib.zdec_q4k_gemm_static(dummy, 4096, 4096, dummy, 1, dummy, 4, None) == -1
    assert lib.zdec_q4k_gemm_static(dummy, 4096, 4000, dummy, 1, dummy, 2, None) == -5


def _matrix(N, K, seed, dev, torch):
    W = synth.q4k_matrix(seed, 600, N, K, 0.02)
    Wc = torch.from_numpy(W.reshape(-1)).to(dev)
    Wr = torch.empty(z.q4k_repacked_bytes(N, K), dtype=torch.uint8, device=dev)
    z.q4k_repack(Wc, N, K, Wr)
    return Wr


@gpu
@needs_cuda
@pytest.mark.parametrize("N,K,B,impl", [(4096, 4096, 1, 1), (2048, 4096, 3, 1), (4096, 4096, 1, 2), (4096, 4096, 1, 3),
                                        (1024, 4096, 13, 2), (512, 8192, 32, 2)])
def test_static_gemm_equals_workspace_gemm_on_consecutive_calls(N, K, B, impl):
    torch = pytest.importorskip("torch")
    dev = torch.device("cuda")
    assert K * B <= z.Q4K_GEMM_STATIC_MAX_KB
    Wr = _matrix(N, K, N + B, dev, torch)
    ws = torch.empty(z.q4k_gemm_workspace_bytes(K, B), dtype=torch.uint8, device=dev)
    for call in range(2):                  # two consecutive calls, different inputs
        x = torch.from_numpy(synth.normal_f32(7 + call, 601, B * K).reshape(B, K)).to(dev)
        ref = torch.full((B, N), float("nan"), dtype=torch.float32, device=dev)
        got = torch.full((B, N), float("nan"), dtype=torch.float32, device=dev)
        z.q4k_gemm(Wr, N, K, x, ref, impl, ws)
        z.q4k_gemm_static(Wr, N, K, x, got, impl)
        torch.cuda.synchronize()
        assert torch.isfinite(ref).all()
        assert torch.equal(got.view(torch.int32), ref.view(torch.int32)), (N, K, B, impl, call)


@gpu
@needs_cuda
def test_static_gemm_back_to_back_shapes_on_one_stream():
    """A large call then a small one queued on the same stream without a
    synchronisation between them: the second reads only what its own prep
    wrote, and stream order keeps the two calls apart."""
    torch = pytest.importorskip("torch")
    dev = torch.device("cuda")
    shapes = [(1024, 8192, 32), (2048, 512, 2)]
    outs, refs = [], []
    for i, (N, K, B) in enumerate(shapes):
        Wr = _matrix(N, K, 90 + i, dev, torch)
        x = torch.from_numpy(synth.normal_f32(90 + i, 602, B * K).reshape(B, K)).to(dev)
        y = torch.empty((B, N), dtype=torch.float32, device=dev)
        z.q4k_gemm_static(Wr, N, K, x, y, 2)
        outs.append((Wr, x, y, N, K, B))
    torch.cuda.synchronize()
    for Wr, x, y, N, K, B in outs:
        ws = torch.empty(z.q4k_gemm_workspace_bytes(K, B), dtype=torch.uint8, device=dev)
        ref = torch.empty((B, N), dtype=torch.float32, device=dev)
        z.q4k_gemm(Wr, N, K, x, ref, 2, ws)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int32), ref.view(torch.int32)), (N, K, B)
