"""Seeded synthetic inputs for the batched Q4_K decode step.

This module only *produces inputs*: Gaussian weights quantized to canonical
Q4_K blocks, fp16 KV histories, token ids.  Both the CPU oracle tests and the
GPU library consume what it writes; it contains none of the decode step's
arithmetic (no dequantization, matmul, attention or KV quantization).

The generator is counter based (splitmix64 finaliser over (seed, stream,
index)), so every tensor of the synthetic model is addressed by a stream id
and can be regenerated piecewise.  Stream ids of the model are fixed by
:func:`stream_id`.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "_synth.so")
_lib = None

QK_K = 256            # weights per Q4_K super-block
Q4K_BLOCK_BYTES = 144  # canonical bytes per super-block


def build(force: bool = False) -> str:
    """Compile synth.c into _synth.so (plain gcc, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=_HERE)
    os.close(fd)
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    u64, i64, u32, f64, vp = (ctypes.c_uint64, ctypes.c_int64, ctypes.c_uint32,
                              ctypes.c_double, ctypes.c_void_p)
    lib.synth_bits.restype = u64
    lib.synth_bits.argtypes = [u64, u64, u64]
    lib.synth_f32_to_f16.restype = ctypes.c_uint16
    lib.synth_f32_to_f16.argtypes = [ctypes.c_float]
    lib.synth_f16_to_f32.restype = ctypes.c_float
    lib.synth_f16_to_f32.argtypes = [ctypes.c_uint16]
    lib.synth_normal_f32.argtypes = [u64, u64, u64, i64, f64, f64, vp]
    lib.synth_normal_f16.argtypes = [u64, u64, u64, i64, f64, vp]
    lib.synth_uniform_int.argtypes = [u64, u64, i64, u32, vp]
    lib.synth_q4k_quantize_block.argtypes = [vp, vp]
    lib.synth_q4k_quantize.argtypes = [vp, i64, vp]
    lib.synth_q4k_matrix.argtypes = [u64, u64, i64, i64, f64, vp]
    for f in ("synth_normal_f32", "synth_normal_f16", "synth_uniform_int",
              "synth_q4k_quantize_block", "synth_q4k_quantize", "synth_q4k_matrix"):
        getattr(lib, f).restype = None
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


# ----------------------------------------------------------------- streams
# Stream ids of the synthetic model.  Layer tensors: 100 + 16*layer + slot.
_LAYER_SLOTS = {"wq": 0, "wk": 1, "wv": 2, "wo": 3, "w_gate": 4, "w_up": 5, "w_down": 6}


def stream_id(name: str, layer: int = 0) -> int:
    if name == "embed":
        return 1
    if name == "tokens":
        return 2
    if name == "activation":
        return 3
    if name in _LAYER_SLOTS:
        return 100 + 16 * layer + _LAYER_SLOTS[name]
    raise KeyError(name)


def kv_stream(seq: int, layer: int, which: int) -> int:
    """Stream of the KV history of sequence `seq`, layer `layer`; which=0 K, 1 V."""
    return 1_000_000 + 4096 * seq + 2 * layer + which


# ------------------------------------------------------------- primitives
def bits(seed: int, stream: int, index: int) -> int:
    return int(_load().synth_bits(seed, stream, index))


def f32_to_f16_bits(x) -> np.ndarray:
    """Round fp32 values to binary16 (nearest, ties to even); returns uint16 bits."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    lib = _load()
    out = np.empty(x.shape, dtype=np.uint16)
    flat, of = x.reshape(-1), out.reshape(-1)
    for i in range(flat.size):
        of[i] = lib.synth_f32_to_f16(float(flat[i]))
    return out


def normal_f32(seed: int, stream: int, n: int, std: float = 1.0, mean: float = 0.0,
               offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float32)
    _load().synth_normal_f32(seed, stream, offset, n, mean, std, _ptr(out))
    return out


def normal_f16(seed: int, stream: int, n: int, std: float = 1.0, offset: int = 0) -> np.ndarray:
    """n N(0, std^2) draws rounded to fp16; returned as uint16 bit patterns."""
    out = np.empty(n, dtype=np.uint16)
    _load().synth_normal_f16(seed, stream, offset, n, std, _ptr(out))
    return out


def uniform_int(seed: int, stream: int, n: int, hi: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int32)
    _load().synth_uniform_int(seed, stream, n, hi, _ptr(out))
    return out


def q4k_quantize(x: np.ndarray) -> np.ndarray:
    """Quantize fp32 values (length a multiple of 256) to canonical Q4_K bytes."""
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
    assert x.size % QK_K == 0
    nb = x.size // QK_K
    out = np.empty(nb * Q4K_BLOCK_BYTES, dtype=np.uint8)
    _load().synth_q4k_quantize(_ptr(x), nb, _ptr(out))
    return out


def q4k_matrix(seed: int, stream: int, rows: int, cols: int, std: float = 0.02) -> np.ndarray:
    """Gaussian rows x cols matrix quantized to Q4_K: uint8 [rows, cols/256*144]."""
    assert cols % QK_K == 0
    out = np.empty((rows, cols // QK_K * Q4K_BLOCK_BYTES), dtype=np.uint8)
    _load().synth_q4k_matrix(seed, stream, rows, cols, std, _ptr(out))
    return out
