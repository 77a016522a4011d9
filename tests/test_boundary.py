"""CPU checks of the C-ABI boundary: the library builds for sm_103a, loads,
exports every symbol include/zdec.h declares, and its host-side argument
validation answers without touching a GPU."""
import ctypes
import os
import re

import pytest

import quantized_decode_step_02_gb300 as z

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    src = open(os.path.join(ROOT, "include", "zdec.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(zdec_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_function():
    lib = z.load_library()
    declared = _header_functions()
    assert len(declared) >= 20
    missing = [f for f in declared if not hasattr(lib, f)]
    assert not missing, missing
    assert sorted(z.EXPORTS) == declared


def test_size_queries():
    assert z.q4k_repacked_bytes(4096, 4096) == 4096 * 16 * 144
    assert z.q4k_repacked_bytes(4095, 4096) == 0          # N must be a multiple of 16
    assert z.q4k_repacked_bytes(4096, 100) == 0
    ws = z.q4k_gemm_workspace_bytes(4096, 1)
    assert ws >= 2 * 1 * 4096 * 2 + 16 * 16 * 2           # hi + lo planes of one row, sums
    assert z.q4k_gemm_workspace_bytes(4096, 33) == 0
    assert z.q4k_repacked_bytes(144, 512) == 128 * 2 * 2 * 144   # rows padded to 128


def _create(desc_kw, max_B=1, max_L=16):
    lib = z.load_library()
    d = z.ModelDesc(**desc_kw)._c()
    w = z._Weights()
    h = ctypes.c_void_p()
    return lib.zdec_create(ctypes.byref(d), ctypes.byref(w), 0, max_B, max_L, None, ctypes.byref(h))


def test_create_rejects_bad_shapes_before_any_cuda_call():
    small = dict(n_layers=1, hidden=512, n_q_heads=4, n_kv_heads=1, head_dim=128, ffn=512, vocab=10)
    assert _create({**small, "head_dim": 64}) == -5          # ZDEC_ERR_UNSUPPORTED
    assert _create({**small, "n_kv_heads": 2}) == -5          # group of four only
    assert _create({**small, "hidden": 384}) == -5
    assert _create({**small, "n_layers": 0}) == -1            # ZDEC_ERR_ARG
    assert _create(small, max_B=0) == -1
    assert _create(small, max_B=33) == -1
    assert _create(small) == -1                               # null weight pointers
    assert b"null weight" in z.load_library().zdec_last_global_error()


def test_create_cache_rejects_bad_cache_descriptions():
    """Bad K/V types, slot counts, lengths and pool sizes fail with
    ZDEC_ERR_ARG before anything is allocated."""
    lib = z.load_library()
    small = z.ModelDesc(n_layers=1, hidden=512, n_q_heads=4, n_kv_heads=1, head_dim=128, ffn=512, vocab=10)._c()
    w = z._Weights()
    h = ctypes.c_void_p()
    cases = [((3, 0, 1, 16, 0), b"type"), ((0, -1, 1, 16, 0), b"type"), ((0, 0, 0, 16, 0), b"max_B"),
             ((0, 0, 33, 16, 0), b"max_B"), ((0, 2, 1, 0, 0), b"max_L"), ((1, 2, 1, 16, -1), b"pool_tokens"),
             ((2, 1, 1, 16, 64), b"null weight")]
    for args, msg in cases:
        c = z._Cache(*args)
        assert lib.zdec_create_cache(ctypes.byref(small), ctypes.byref(w), ctypes.byref(c), None,
                                     ctypes.byref(h)) == -1, args
        assert msg in lib.zdec_last_global_error(), (args, lib.zdec_last_global_error())


def test_null_context_calls_fail_cleanly():
    lib = z.load_library()
    assert lib.zdec_sync(None) == -1
    assert lib.zdec_decode_step(None, 1, None, None, None, None, 0) == -1
    assert lib.zdec_append_kv(None, 0, 1, None, None, 0) == -1
    lib.zdec_destroy(None)


def test_stateless_gemm_validates_arguments():
    lib = z.load_library()
    dummy = ctypes.c_void_p(16)
    assert lib.zdec_q4k_gemm(dummy, 4096, 4096, dummy, 1, dummy, 4, dummy, 1 << 20, None) == -1
    assert lib.zdec_q4k_gemm(dummy, 4096, 4096, dummy, 2, dummy, 3, dummy, 1 << 20, None) == -5
    assert lib.zdec_q4k_gemm(dummy, 4096, 4096, dummy, 5, dummy, 1, dummy, 1 << 20, None) == -5
    assert lib.zdec_q4k_gemm(dummy, 4008, 4096, dummy, 1, dummy, 2, dummy, 1 << 20, None) == -5
    assert lib.zdec_q4k_gemm(dummy, 4096, 4096, dummy, 1, dummy, 2, dummy, 16, None) == -1
