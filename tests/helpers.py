"""Shared helpers of the parity tests."""
from __future__ import annotations

import functools
import json
import os

import numpy as np
import pytest

TOL = 2e-3          # max normwise relative error of floats against the oracle
GAP = 1e-2          # argmax ids must match where the oracle's top-2 gap exceeds this


def normwise(a, ref) -> float:
    """max|a - ref| / max|ref| (the reading of 'max relative error per vector')."""
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.abs(ref).max()
    return float(np.abs(a - ref).max() / (den if den > 0 else 1.0))


def top2_gap(logits: np.ndarray) -> np.ndarray:
    s = np.sort(np.asarray(logits, np.float64), axis=-1)
    return s[..., -1] - s[..., -2]


def cuda_ok() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


gpu = pytest.mark.gpu
needs_cuda = pytest.mark.skipif(not cuda_ok(), reason="needs a CUDA GPU")


@functools.lru_cache(maxsize=4)
def cached_model(desc, seed):
    from synth.model import make_model
    return make_model(desc, seed)


def record_margin(tag: str, hidden_err: float, logits_err: float, ids_checked: int, rows: int):
    """Print a parity check's worst normwise errors (and append them as a JSON
    line to $ZDEC_MARGINS_FILE when that is set)."""
    rec = {"case": tag, "worst_hidden": hidden_err, "worst_logits": logits_err, "tol": TOL,
           "ids_checked": ids_checked, "rows": rows}
    print(f"[margin] {tag}: hidden {hidden_err:.3g} logits {logits_err:.3g} (tol {TOL:g}), "
          f"ids checked {ids_checked}/{rows}")
    path = os.environ.get("ZDEC_MARGINS_FILE")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")
