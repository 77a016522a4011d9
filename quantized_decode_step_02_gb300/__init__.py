"""Python binding of libzdec, the batched Q4_K decode step for one GB300.

Argument marshalling only: every step of the decode path runs in the CUDA
kernels of ``libzdec.so`` (built from ``csrc/`` for sm_103a).  There is no
CPU or PyTorch fallback; if the library cannot be loaded, every entry point
raises.  PyTorch is used for device buffers and streams.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

from . import _build

__all__ = ["ModelDesc", "Decoder", "ZdecError", "load_library", "q4k_repacked_bytes",
           "q4k_repack", "q4k_gemm", "q4k_gemm_workspace_bytes", "q4k_gemm_static",
           "Q4K_GEMM_STATIC_MAX_KB", "KV_F16", "KV_Q8_0", "KV_FP8", "PAGE_TOKENS",
           "KERNEL_KINDS", "T_EMBED", "T_WQ", "T_WK", "T_WV", "T_WO", "T_GATE", "T_UP", "T_DOWN"]

KV_F16, KV_Q8_0, KV_FP8 = 0, 1, 2   # per-tensor cache types (zdec_kv_dtype)
PAGE_TOKENS = 64                    # tokens per KV pool page
Q4K_GEMM_STATIC_MAX_KB = 262144   # K*B limit of q4k_gemm_static (ZDEC_Q4K_GEMM_STATIC_MAX_KB)
STEP_HOST_IO, STEP_EAGER = 1, 2
T_EMBED, T_WQ, T_WK, T_WV, T_WO, T_GATE, T_UP, T_DOWN = range(8)
KERNEL_KINDS = ["embed", "-", "gemm_qkv", "attention", "gemm_o", "gemm_gateup", "gemm_down",
                "gemm_lmhead", "argmax"]
STATUS = {0: "ok", -1: "bad argument", -2: "out of memory", -3: "capacity", -4: "position",
          -5: "unsupported", -6: "cuda error", -7: "timeout", -8: "device check"}

# Every symbol include/zdec.h declares; load_library() checks they are exported.
EXPORTS = ["zdec_create_cache", "zdec_create", "zdec_destroy", "zdec_append_kv", "zdec_decode_step",
           "zdec_decode_step_slots", "zdec_sync", "zdec_reset_seq", "zdec_seq_len", "zdec_last_error",
           "zdec_last_global_error", "zdec_set_gemm_impl", "zdec_set_trace", "zdec_debug_step_trace",
           "zdec_get_info", "zdec_profile_step", "zdec_debug_export_q4k", "zdec_debug_dequant",
           "zdec_debug_read_kv", "zdec_debug_block_table", "zdec_debug_capture_hidden",
           "zdec_debug_attention", "zdec_debug_set_wait_limit", "zdec_q4k_repacked_bytes", "zdec_q4k_repack",
           "zdec_q4k_gemm_workspace_bytes", "zdec_q4k_gemm", "zdec_q4k_gemm_static"]


class ZdecError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"zdec: {STATUS.get(status, status)}: {msg}")
        self.status = status


class _Desc(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("hidden", ctypes.c_int), ("n_q_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("vocab", ctypes.c_int), ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float)]


_PP = ctypes.POINTER(ctypes.c_void_p)


class _Weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("attn_norm", _PP), ("ffn_norm", _PP), ("wq", _PP), ("wk", _PP), ("wv", _PP),
                ("wo", _PP), ("w_gate", _PP), ("w_up", _PP), ("w_down", _PP)]


class _Cache(ctypes.Structure):
    _fields_ = [("k_type", ctypes.c_int), ("v_type", ctypes.c_int), ("max_B", ctypes.c_int),
                ("max_L", ctypes.c_int), ("pool_tokens", ctypes.c_longlong)]


class _Info(ctypes.Structure):
    _fields_ = [("weight_bytes", ctypes.c_size_t), ("arena_bytes", ctypes.c_size_t),
                ("workspace_bytes", ctypes.c_size_t), ("kv_bytes_per_token", ctypes.c_size_t),
                ("kernels_per_step", ctypes.c_int), ("attn_splits", ctypes.c_int),
                ("matvec_max_B", ctypes.c_int), ("attn_segments", ctypes.c_int),
                ("k_type", ctypes.c_int), ("v_type", ctypes.c_int), ("page_tokens", ctypes.c_int),
                ("pool_pages", ctypes.c_int), ("free_pages", ctypes.c_int)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load_library(build_if_missing: bool = True):
    """Load libzdec.so (building it with nvcc first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(_build.LIB):
        raise ImportError(f"libzdec.so not found at {_build.LIB}; run __graft_entry__.build()")
    lib = ctypes.CDLL(_build.LIB)
    for name in EXPORTS:
        if not hasattr(lib, name):
            raise ImportError(f"libzdec.so does not export {name}")
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    sigs = {
        "zdec_create": (i, [ctypes.POINTER(_Desc), ctypes.POINTER(_Weights), i, i, i, vp,
                            ctypes.POINTER(vp)]),
        "zdec_create_cache": (i, [ctypes.POINTER(_Desc), ctypes.POINTER(_Weights), ctypes.POINTER(_Cache),
                                  vp, ctypes.POINTER(vp)]),
        "zdec_decode_step_slots": (i, [vp, i, vp, vp, vp, vp, vp, i]),
        "zdec_debug_block_table": (i, [vp, i, vp, i, ctypes.POINTER(i)]),
        "zdec_destroy": (None, [vp]),
        "zdec_append_kv": (i, [vp, i, i, vp, vp, i]),
        "zdec_decode_step": (i, [vp, i, vp, vp, vp, vp, i]),
        "zdec_sync": (i, [vp]),
        "zdec_reset_seq": (i, [vp, i]),
        "zdec_seq_len": (i, [vp, i, ctypes.POINTER(i)]),
        "zdec_last_error": (ctypes.c_char_p, [vp]),
        "zdec_last_global_error": (ctypes.c_char_p, []),
        "zdec_set_gemm_impl": (i, [vp, i]),
        "zdec_get_info": (i, [vp, ctypes.POINTER(_Info)]),
        "zdec_set_trace": (i, [vp, i]),
        "zdec_debug_step_trace": (i, [vp, vp, sz, ctypes.POINTER(sz)]),
        "zdec_profile_step": (i, [vp, i, vp, vp, vp, vp, vp, vp, i, ctypes.POINTER(i)]),
        "zdec_debug_export_q4k": (i, [vp, i, i, i, i, vp]),
        "zdec_debug_dequant": (i, [vp, i, i, i, i, vp]),
        "zdec_debug_read_kv": (i, [vp, i, i, i, i, vp, vp, vp, vp]),
        "zdec_debug_capture_hidden": (i, [vp, vp]),
        "zdec_debug_attention": (i, [vp, i, i, vp, vp, vp]),
        "zdec_debug_set_wait_limit": (i, [vp, ctypes.c_longlong]),
        "zdec_q4k_repacked_bytes": (sz, [i, i]),
        "zdec_q4k_repack": (i, [vp, i, i, vp, vp]),
        "zdec_q4k_gemm_workspace_bytes": (sz, [i, i]),
        "zdec_q4k_gemm": (i, [vp, i, i, vp, i, vp, i, vp, sz, vp]),
        "zdec_q4k_gemm_static": (i, [vp, i, i, vp, i, vp, i, vp]),
    }
    for name, (res, args) in sigs.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _ptr(x) -> int:
    """Address of a numpy array or torch tensor (must be contiguous)."""
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        assert x.flags["C_CONTIGUOUS"], "array must be C-contiguous"
        return x.ctypes.data
    if hasattr(x, "data_ptr"):
        assert x.is_contiguous(), "tensor must be contiguous"
        return x.data_ptr()
    raise TypeError(type(x))


def _is_cuda(x) -> bool:
    return hasattr(x, "is_cuda") and x.is_cuda


@dataclass(frozen=True)
class ModelDesc:
    n_layers: int = 36
    hidden: int = 4096
    n_q_heads: int = 32
    n_kv_heads: int = 8
    head_dim: int = 128
    ffn: int = 14336
    vocab: int = 151936
    rope_theta: float = 1e6
    rms_eps: float = 1e-6

    @classmethod
    def of(cls, d) -> "ModelDesc":
        return cls(d.n_layers, d.hidden, d.n_q_heads, d.n_kv_heads, d.head_dim, d.ffn, d.vocab,
                   d.rope_theta, d.rms_eps)

    def _c(self) -> _Desc:
        return _Desc(self.n_layers, self.hidden, self.n_q_heads, self.n_kv_heads, self.head_dim,
                     self.ffn, self.vocab, self.rope_theta, self.rms_eps)


class Decoder:
    """One decoder context (weights, paged KV pool, workspace) on the current GPU.

    ``weights`` holds canonical Q4_K matrices as uint8 numpy arrays
    [rows, cols/256*144] (per-layer tensors as lists) and fp32 norm gains;
    the library copies and repacks them at creation.  ``kv_dtype`` is one
    cache type for K and V (KV_F16, KV_Q8_0, KV_FP8) or a (k_type, v_type)
    pair; ``pool_tokens`` sizes the shared page pool (0: max_B * max_L)."""

    def __init__(self, desc, weights: dict, kv_dtype=KV_F16, max_B: int = 1, max_L: int = 2048,
                 stream=None, pool_tokens: int = 0):
        self.lib = load_library()
        self.desc = ModelDesc.of(desc)
        d = self.desc
        L = d.n_layers
        keep = []

        def arr(name):
            want = np.float32 if name.endswith("norm") else np.uint8
            mats = [np.ascontiguousarray(weights[name][l], want) for l in range(L)]
            keep.extend(mats)
            a = (ctypes.c_void_p * L)(*[_ptr(m) for m in mats])
            keep.append(a)
            return ctypes.cast(a, _PP)

        fnorm = np.ascontiguousarray(weights["final_norm"], np.float32)
        embed = np.ascontiguousarray(weights["embed"], np.uint8)
        keep += [fnorm, embed]
        w = _Weights(_ptr(embed), _ptr(fnorm),
                     arr("attn_norm"), arr("ffn_norm"), arr("wq"), arr("wk"), arr("wv"), arr("wo"),
                     arr("w_gate"), arr("w_up"), arr("w_down"))
        kt, vt = (int(kv_dtype), int(kv_dtype)) if np.isscalar(kv_dtype) else (int(kv_dtype[0]), int(kv_dtype[1]))
        self.k_type, self.v_type = kt, vt
        self.kv_dtype = kt if kt == vt else (kt, vt)
        self.max_B, self.max_L = max_B, max_L
        self.stream = stream
        h = ctypes.c_void_p()
        desc_c = d._c()
        cache = _Cache(kt, vt, max_B, max_L, int(pool_tokens))
        s = self.lib.zdec_create_cache(ctypes.byref(desc_c), ctypes.byref(w), ctypes.byref(cache),
                                       ctypes.c_void_p(stream) if stream else None, ctypes.byref(h))
        if s != 0:
            raise ZdecError(s, self.lib.zdec_last_global_error().decode())
        self.h = h

    # ---------------------------------------------------------------- utils
    def _check(self, s: int):
        if s != 0:
            raise ZdecError(s, self.lib.zdec_last_error(self.h).decode())

    def close(self):
        if getattr(self, "h", None):
            self.lib.zdec_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    # ------------------------------------------------------------------ API
    def append_kv(self, seq: int, k16, v16):
        """Append rotated fp16 K/V [n_layers][n][n_kv][hd] (uint16 numpy on the host,
        or a torch float16/int16 CUDA tensor) to sequence `seq`."""
        n = k16.shape[1]
        on_dev = 1 if _is_cuda(k16) else 0
        if not on_dev:
            k16 = np.ascontiguousarray(k16, np.uint16)
            v16 = np.ascontiguousarray(v16, np.uint16)
        self._check(self.lib.zdec_append_kv(self.h, seq, n, _ptr(k16), _ptr(v16), on_dev))

    def _run(self, B, slots, tokens, positions, logits, ids, flags):
        if slots is None:
            self._check(self.lib.zdec_decode_step(self.h, B, _ptr(tokens), _ptr(positions),
                                                  _ptr(logits), _ptr(ids), flags))
        else:
            sl = np.ascontiguousarray(slots, np.int32)
            assert sl.shape == (B,)
            self._check(self.lib.zdec_decode_step_slots(self.h, B, _ptr(sl), _ptr(tokens), _ptr(positions),
                                                        _ptr(logits), _ptr(ids), flags))

    def step(self, tokens, positions, logits=None, ids=None, eager: bool = False, slots=None):
        """Device I/O step: tokens/positions int32 CUDA tensors [B], logits float32
        CUDA [B, vocab] or None, ids int32 CUDA [B]; row b uses cache slot
        slots[b] (host ints; default b).  Asynchronous."""
        B = tokens.shape[0]
        self._run(B, slots, tokens, positions, logits, ids, STEP_EAGER if eager else 0)

    def step_host(self, tokens, positions, logits: np.ndarray | None = None,
                  ids: np.ndarray | None = None, eager: bool = False, slots=None):
        """Host I/O step: numpy int32 tokens/positions; returns (logits, ids) numpy.
        Copies in, runs, copies out and waits.  Row b uses slot slots[b]."""
        tokens = np.ascontiguousarray(tokens, np.int32)
        positions = np.ascontiguousarray(positions, np.int32)
        B = tokens.shape[0]
        if ids is None:
            ids = np.empty(B, np.int32)
        self._run(B, slots, tokens, positions, logits, ids, STEP_HOST_IO | (STEP_EAGER if eager else 0))
        return logits, ids

    def sync(self):
        self._check(self.lib.zdec_sync(self.h))

    def reset_seq(self, seq: int):
        self._check(self.lib.zdec_reset_seq(self.h, seq))

    def seq_len(self, seq: int) -> int:
        n = ctypes.c_int()
        self._check(self.lib.zdec_seq_len(self.h, seq, ctypes.byref(n)))
        return n.value

    def set_gemm_impl(self, impl: int):
        self._check(self.lib.zdec_set_gemm_impl(self.h, impl))

    def set_trace(self, on: bool):
        """Record the launch timeline of the following steps (run eagerly)."""
        self._check(self.lib.zdec_set_trace(self.h, int(bool(on))))

    def step_trace(self) -> np.ndarray:
        """Timeline of the last traced step (see zdec.h): [launches][8] uint64."""
        n = ctypes.c_size_t()
        self._check(self.lib.zdec_debug_step_trace(self.h, None, 0, ctypes.byref(n)))
        if n.value == 0:
            return np.zeros((0, 8), np.uint64)
        out = np.empty(n.value, np.uint64)
        self._check(self.lib.zdec_debug_step_trace(self.h, _ptr(out), n.value, ctypes.byref(n)))
        return out.reshape(-1, 8)

    def info(self) -> dict:
        inf = _Info()
        self._check(self.lib.zdec_get_info(self.h, ctypes.byref(inf)))
        return {f: getattr(inf, f) for f, _ in _Info._fields_}

    def profile_step(self, tokens, positions, logits, ids, cap: int = 4096):
        """One eager step with CUDA events around every launch; returns a list of
        (kind name, milliseconds)."""
        kind = np.zeros(cap, np.int32)
        ms = np.zeros(cap, np.float32)
        n = ctypes.c_int()
        B = tokens.shape[0]
        self._check(self.lib.zdec_profile_step(self.h, B, _ptr(tokens), _ptr(positions), _ptr(logits),
                                               _ptr(ids), _ptr(kind), _ptr(ms), cap, ctypes.byref(n)))
        return [(KERNEL_KINDS[kind[i]], float(ms[i])) for i in range(min(n.value, cap))]

    # ---------------------------------------------------------------- debug
    def set_wait_limit(self, cycles: int):
        """Bound of the projection kernels' stage waits in clock cycles (0: the
        default ~2 s); a wait that runs out makes sync() raise a timeout."""
        self._check(self.lib.zdec_debug_set_wait_limit(self.h, int(cycles)))

    def _cols(self, which: int) -> int:
        d = self.desc
        return {T_WO: d.n_q_heads * d.head_dim, T_DOWN: d.ffn}.get(which, d.hidden)

    def export_q4k(self, which: int, layer: int, row0: int, nrows: int) -> np.ndarray:
        out = np.empty((nrows, self._cols(which) // 256 * 144), np.uint8)
        self._check(self.lib.zdec_debug_export_q4k(self.h, which, layer, row0, nrows, _ptr(out)))
        return out

    def dequant(self, which: int, layer: int, row0: int, nrows: int) -> np.ndarray:
        out = np.empty((nrows, self._cols(which)), np.float32)
        self._check(self.lib.zdec_debug_dequant(self.h, which, layer, row0, nrows, _ptr(out)))
        return out

    def read_kv(self, seq: int, layer: int, t0: int, n: int):
        """Stored K/V of one layer, canonical token-major layout [n][n_kv][hd],
        each tensor in its type: fp16 uint16, Q8_0 int8 codes, FP8 uint8 e4m3
        codes.  Returns (k, v) when neither tensor is Q8_0, else (k, v,
        k_scales, v_scales) with uint16 scales [n][n_kv][hd/32] (None for a
        tensor that is not Q8_0)."""
        d = self.desc
        shape = (n, d.n_kv_heads, d.head_dim)
        dt = {KV_F16: np.uint16, KV_Q8_0: np.int8, KV_FP8: np.uint8}
        k, v = np.empty(shape, dt[self.k_type]), np.empty(shape, dt[self.v_type])
        sshape = (n, d.n_kv_heads, d.head_dim // 32)
        ks = np.empty(sshape, np.uint16) if self.k_type == KV_Q8_0 else None
        vs = np.empty(sshape, np.uint16) if self.v_type == KV_Q8_0 else None
        self._check(self.lib.zdec_debug_read_kv(self.h, seq, layer, t0, n, _ptr(k), _ptr(v), _ptr(ks), _ptr(vs)))
        if ks is None and vs is None:
            return k, v
        return k, v, ks, vs

    def block_table(self, seq: int) -> np.ndarray:
        """Page of each 64 tokens of slot `seq` (-1: none), as the device holds it."""
        n = ctypes.c_int()
        self._check(self.lib.zdec_debug_block_table(self.h, seq, None, 0, ctypes.byref(n)))
        out = np.empty(n.value, np.int32)
        self._check(self.lib.zdec_debug_block_table(self.h, seq, _ptr(out), n.value, ctypes.byref(n)))
        return out

    def step_capture_hidden(self, tokens, positions, logits=None, ids=None):
        """Host I/O step that also returns the fp32 residual after the embedding and
        after every layer: [B, n_layers+1, hidden]."""
        B = len(tokens)
        hid = np.empty((B, self.desc.n_layers + 1, self.desc.hidden), np.float32)
        self._check(self.lib.zdec_debug_capture_hidden(self.h, _ptr(hid)))
        logits, ids = self.step_host(tokens, positions, logits, ids)
        return logits, ids, hid

    def attention(self, layer: int, q: np.ndarray, positions) -> np.ndarray:
        """Attention alone over cached tokens 0..positions[b]: q [B, n_q, hd] fp32
        (already rotated) -> o [B, n_q, hd] fp32."""
        q = np.ascontiguousarray(q, np.float32)
        pos = np.ascontiguousarray(positions, np.int32)
        o = np.empty_like(q)
        self._check(self.lib.zdec_debug_attention(self.h, layer, q.shape[0], _ptr(q), _ptr(pos), _ptr(o)))
        return o


# ------------------------------------------------------------ stateless ops
def _glob_check(s: int):
    if s != 0:
        raise ZdecError(s, load_library().zdec_last_global_error().decode())


def q4k_repacked_bytes(N: int, K: int) -> int:
    return int(load_library().zdec_q4k_repacked_bytes(N, K))


def q4k_repack(canonical_dev, N: int, K: int, repacked_dev, stream=None):
    _glob_check(load_library().zdec_q4k_repack(_ptr(canonical_dev), N, K, _ptr(repacked_dev),
                                               ctypes.c_void_p(stream) if stream else None))


def q4k_gemm_workspace_bytes(K: int, B: int) -> int:
    return int(load_library().zdec_q4k_gemm_workspace_bytes(K, B))


def q4k_gemm(repacked_dev, N: int, K: int, x_dev, y_dev, impl: int, workspace_dev, stream=None):
    B = x_dev.shape[0]
    _glob_check(load_library().zdec_q4k_gemm(_ptr(repacked_dev), N, K, _ptr(x_dev), B, _ptr(y_dev), impl,
                                             _ptr(workspace_dev), workspace_dev.numel() * workspace_dev.element_size(),
                                             ctypes.c_void_p(stream) if stream else None))


def q4k_gemm_static(repacked_dev, N: int, K: int, x_dev, y_dev, impl: int, stream=None):
    """q4k_gemm without a workspace: the library's own per-device scratch
    (K*B <= Q4K_GEMM_STATIC_MAX_KB); calls that may overlap in time race on it."""
    B = x_dev.shape[0]
    _glob_check(load_library().zdec_q4k_gemm_static(_ptr(repacked_dev), N, K, _ptr(x_dev), B, _ptr(y_dev), impl,
                                                    ctypes.c_void_p(stream) if stream else None))
