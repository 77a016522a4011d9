"""CPU oracle of the batched Q4_K decode step (TEST INFRASTRUCTURE ONLY).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The library under
``quantized_decode_step_02_gb300`` never does, and shares no code with it.

Every function is a thin ctypes wrapper around ``oracle.c`` (plain C, fp64)
or, for the closed-form byte model, plain Python in :mod:`oracle.bytemodel`.
Parity status: Q4_K unpack/dequant, Q8_0, fp16 rounding, matvec, RMSNorm,
RoPE, attention, SwiGLU and argmax are pinned by the CPU tests; the
full-model logits are pinned only through those parts plus batch
invariance (no page prints a worked model output).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "_oracle.so")
_lib = None


def build(force: bool = False) -> str:
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


class _Desc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("hidden", ctypes.c_int),
                ("n_q_heads", ctypes.c_int), ("n_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int), ("vocab", ctypes.c_int),
                ("rope_theta", ctypes.c_double), ("rms_eps", ctypes.c_double)]


_PP = ctypes.POINTER(ctypes.c_void_p)


class _Weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("attn_norm", _PP), ("ffn_norm", _PP),
                ("wq", _PP), ("wk", _PP), ("wv", _PP), ("wo", _PP),
                ("w_gate", _PP), ("w_up", _PP), ("w_down", _PP)]


class _KV(ctypes.Structure):
    _fields_ = [("kv_dtype", ctypes.c_int), ("max_L", ctypes.c_int64),
                ("k16", ctypes.c_void_p), ("v16", ctypes.c_void_p),
                ("kq", ctypes.c_void_p), ("vq", ctypes.c_void_p),
                ("ks", ctypes.c_void_p), ("vs", ctypes.c_void_p),
                ("k8", ctypes.c_void_p), ("v8", ctypes.c_void_p),
                ("k_type", ctypes.c_int), ("v_type", ctypes.c_int)]

KV_F16, KV_Q8_0, KV_FP8 = 0, 1, 2   # per-tensor cache types


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i64, f64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_double
    sig = {
        "orc_half_to_float": (ctypes.c_float, [ctypes.c_uint16]),
        "orc_double_to_half": (ctypes.c_uint16, [f64]),
        "orc_q4k_unpack": (None, [vp, vp, vp, vp, vp, vp]),
        "orc_q4k_dequant": (None, [vp, vp]),
        "orc_q4k_matvec": (None, [vp, i64, i64, vp, vp]),
        "orc_q8_0_quantize": (None, [vp, vp, vp]),
        "orc_q8_0_value": (f64, [ctypes.c_uint16, ctypes.c_int8]),
        "orc_e4m3_from_half": (ctypes.c_uint8, [ctypes.c_uint16]),
        "orc_e4m3_value": (f64, [ctypes.c_uint8]),
        "orc_rmsnorm": (None, [vp, vp, i64, f64, vp]),
        "orc_rope": (None, [vp, ctypes.c_int, i64, f64]),
        "orc_silu": (f64, [f64]),
        "orc_argmax": (i64, [vp, i64]),
        "orc_attention": (None, [ctypes.POINTER(_Desc), ctypes.POINTER(_KV), ctypes.c_int,
                                 i64, vp, vp]),
        "orc_decode_step": (None, [ctypes.POINTER(_Desc), ctypes.POINTER(_Weights),
                                   ctypes.POINTER(_KV), ctypes.c_int, vp, vp, vp, vp, vp]),
        "orc_kv_append": (None, [ctypes.POINTER(_Desc), ctypes.POINTER(_KV), i64, i64, vp, vp]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def set_threads(n: int) -> None:
    """OpenMP threads the oracle's parallel loops use from now on."""
    lib = _load()
    f = lib.omp_set_num_threads   # libgomp, a dependency of the oracle library
    f.restype = None
    f.argtypes = [ctypes.c_int]
    f(int(n))


def _p(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle wants C-contiguous arrays"
    return a.ctypes.data


# ------------------------------------------------------------ scalars
def half_to_float(bits: int) -> float:
    return float(_load().orc_half_to_float(int(bits)))


def double_to_half(v: float) -> int:
    return int(_load().orc_double_to_half(float(v)))


# ------------------------------------------------------------ Q4_K
def q4k_unpack(block: np.ndarray):
    """Fields of one canonical 144-byte block: (d, dmin, sc[8], m[8], q[256])."""
    block = np.ascontiguousarray(block, dtype=np.uint8)
    assert block.size == 144
    d = np.zeros(1, np.float32)
    dm = np.zeros(1, np.float32)
    sc = np.zeros(8, np.int32)
    mn = np.zeros(8, np.int32)
    q = np.zeros(256, np.int32)
    _load().orc_q4k_unpack(_p(block), _p(d), _p(dm), _p(sc), _p(mn), _p(q))
    return float(d[0]), float(dm[0]), sc, mn, q


def q4k_dequant(blocks: np.ndarray) -> np.ndarray:
    """Dequantize canonical blocks (uint8, 144 bytes each) to fp32 values."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8).reshape(-1, 144)
    out = np.empty((blocks.shape[0], 256), dtype=np.float32)
    lib = _load()
    for i in range(blocks.shape[0]):
        lib.orc_q4k_dequant(_p(blocks[i]), _p(out[i]))
    return out.reshape(-1)


def q4k_matvec(W: np.ndarray, N: int, K: int, x: np.ndarray) -> np.ndarray:
    """y = W x for canonical Q4_K rows W (N x K), summed in double."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    assert W.size == N * (K // 256) * 144
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty(N, dtype=np.float64)
    _load().orc_q4k_matvec(_p(W), N, K, _p(x), _p(y))
    return y


# ------------------------------------------------------------ Q8_0
def q8_0_quantize(x16: np.ndarray):
    """Quantize fp16 values (uint16 bits, length multiple of 32) to Q8_0:
    returns (scales uint16 [n/32], codes int8 [n])."""
    x16 = np.ascontiguousarray(x16, dtype=np.uint16).reshape(-1)
    assert x16.size % 32 == 0
    nb = x16.size // 32
    sc = np.empty(nb, np.uint16)
    q = np.empty(x16.size, np.int8)
    lib = _load()
    for b in range(nb):
        lib.orc_q8_0_quantize(x16[32 * b:].ctypes.data, sc[b:].ctypes.data, q[32 * b:].ctypes.data)
    return sc, q


def q8_0_value(scale_bits: int, code: int) -> float:
    return float(_load().orc_q8_0_value(int(scale_bits), int(code)))


# ------------------------------------------------------------ FP8 e4m3
def e4m3_from_half(bits: int) -> int:
    """e4m3 code of one fp16 value (nearest, ties to even, saturating to +-448)."""
    return int(_load().orc_e4m3_from_half(int(bits)))


def e4m3_value(code: int) -> float:
    return float(_load().orc_e4m3_value(int(code)))


# ------------------------------------------------------------ layer math
def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    g = np.ascontiguousarray(g, dtype=np.float32)
    y = np.empty_like(x)
    _load().orc_rmsnorm(_p(x), _p(g), x.size, eps, _p(y))
    return y


def rope(v: np.ndarray, pos: int, theta: float = 1e6) -> np.ndarray:
    v = np.array(v, dtype=np.float64, copy=True)
    _load().orc_rope(_p(v), v.size, pos, theta)
    return v


def silu(g: float) -> float:
    return float(_load().orc_silu(float(g)))


def argmax(x: np.ndarray) -> int:
    x = np.ascontiguousarray(x, dtype=np.float32)
    return int(_load().orc_argmax(_p(x), x.size))


# ------------------------------------------------------------ model
@dataclass
class Desc:
    n_layers: int = 36
    hidden: int = 4096
    n_q_heads: int = 32
    n_kv_heads: int = 8
    head_dim: int = 128
    ffn: int = 14336
    vocab: int = 151936
    rope_theta: float = 1e6
    rms_eps: float = 1e-6

    def c(self) -> _Desc:
        return _Desc(self.n_layers, self.hidden, self.n_q_heads, self.n_kv_heads,
                     self.head_dim, self.ffn, self.vocab, self.rope_theta, self.rms_eps)


class Model:
    """Canonical Q4_K weights held as numpy arrays (no copies made)."""

    def __init__(self, desc: Desc, weights: dict):
        self.desc = desc
        self.w = weights
        L = desc.n_layers

        def arr(name):
            ptrs = (ctypes.c_void_p * L)(*[_p(weights[name][l]) for l in range(L)])
            return ptrs

        self._keep = {n: arr(n) for n in ("attn_norm", "ffn_norm", "wq", "wk", "wv", "wo",
                                          "w_gate", "w_up", "w_down")}
        k = self._keep
        cast = lambda a: ctypes.cast(a, _PP)
        self.cw = _Weights(_p(weights["embed"]), _p(weights["final_norm"]),
                           cast(k["attn_norm"]), cast(k["ffn_norm"]), cast(k["wq"]),
                           cast(k["wk"]), cast(k["wv"]), cast(k["wo"]), cast(k["w_gate"]),
                           cast(k["w_up"]), cast(k["w_down"]))
        self.cdesc = desc.c()


class KV:
    """One sequence's cache in canonical token-major layout (see oracle.c)."""

    def __init__(self, desc: Desc, max_L: int, kv_dtype):
        """kv_dtype: one type for both tensors (KV_F16, KV_Q8_0, KV_FP8) or a
        (k_type, v_type) pair."""
        self.desc, self.max_L, self.kv_dtype = desc, max_L, kv_dtype
        kt, vt = (kv_dtype, kv_dtype) if isinstance(kv_dtype, int) else tuple(kv_dtype)
        assert kt in (KV_F16, KV_Q8_0, KV_FP8) and vt in (KV_F16, KV_Q8_0, KV_FP8)
        self.k_type, self.v_type = kt, vt
        shape = (desc.n_layers, max_L, desc.n_kv_heads, desc.head_dim)
        sshape = (desc.n_layers, max_L, desc.n_kv_heads, desc.head_dim // 32)
        z = lambda s, t: np.zeros(s, dtype=t)
        self.k16 = z(shape, np.uint16) if kt == KV_F16 else None
        self.v16 = z(shape, np.uint16) if vt == KV_F16 else None
        self.kq, self.ks = (z(shape, np.int8), z(sshape, np.uint16)) if kt == KV_Q8_0 else (None, None)
        self.vq, self.vs = (z(shape, np.int8), z(sshape, np.uint16)) if vt == KV_Q8_0 else (None, None)
        self.k8 = z(shape, np.uint8) if kt == KV_FP8 else None
        self.v8 = z(shape, np.uint8) if vt == KV_FP8 else None
        self.len = 0
        ptr = lambda a: _p(a) if a is not None else None
        self.c = _KV(kt if kt == vt else -1, max_L, ptr(self.k16), ptr(self.v16), ptr(self.kq),
                     ptr(self.vq), ptr(self.ks), ptr(self.vs), ptr(self.k8), ptr(self.v8), kt, vt)

    def append(self, k16: np.ndarray, v16: np.ndarray):
        """Append n tokens of rotated fp16 K/V, arrays [n_layers][n][n_kv][hd] uint16."""
        d = self.desc
        k16 = np.ascontiguousarray(k16, dtype=np.uint16)
        v16 = np.ascontiguousarray(v16, dtype=np.uint16)
        n = k16.shape[1]
        assert self.len + n <= self.max_L
        _load().orc_kv_append(ctypes.byref(d.c()), ctypes.byref(self.c), self.len, n,
                              _p(k16), _p(v16))
        self.len += n


def attention(desc: Desc, kv: KV, layer: int, pos: int, q: np.ndarray) -> np.ndarray:
    """Attention of rotated queries q [n_q*hd] over stored tokens 0..pos."""
    q = np.ascontiguousarray(q, dtype=np.float64)
    o = np.empty(desc.n_q_heads * desc.head_dim, dtype=np.float64)
    _load().orc_attention(ctypes.byref(desc.c()), ctypes.byref(kv.c), layer, pos, _p(q), _p(o))
    return o


def decode_step(model: Model, kvs: list, tokens, positions, capture_hidden: bool = False):
    """One decode step for B = len(kvs) sequences.  Returns (logits [B, vocab]
    fp32, ids [B] int32, hidden [B, n_layers+1, hidden] fp32 or None).  Each
    KV gains the new token at positions[b]."""
    d = model.desc
    B = len(kvs)
    tokens = np.ascontiguousarray(tokens, dtype=np.int32)
    positions = np.ascontiguousarray(positions, dtype=np.int32)
    for b in range(B):
        assert positions[b] == kvs[b].len, "position must equal the cached length"
        assert kvs[b].len + 1 <= kvs[b].max_L
    arr = (_KV * B)(*[kv.c for kv in kvs])
    logits = np.empty((B, d.vocab), dtype=np.float32)
    ids = np.empty(B, dtype=np.int32)
    hidden = np.empty((B, d.n_layers + 1, d.hidden), dtype=np.float32) if capture_hidden else None
    _load().orc_decode_step(ctypes.byref(model.cdesc), ctypes.byref(model.cw), arr, B,
                            _p(tokens), _p(positions), _p(logits), _p(ids),
                            _p(hidden) if hidden is not None else None)
    for kv in kvs:
        kv.len += 1
    return logits, ids, hidden
