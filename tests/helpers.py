"""Shared helpers of the test suite (no arithmetic of the method here)."""
import os

import numpy as np
import pytest
import torch

# Tolerances on the max relative error max|x - ref| / max|ref| per tensor:
# fp32 inputs 1e-4; bf16 inputs with fp32 state 2e-2.
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


# Every comparison made through rel_err() is recorded here as (test, max-normalised error, floored
# elementwise error); the end of the run prints the worst pair per test (tests/conftest.py).
ERRORS = []


def elem_rel_err(x, ref, floor: float = 1e-6) -> float:
    """Largest elementwise relative error |x - ref| / max(|ref|, floor * max|ref|): unlike the
    max-normalised error it shows how well small entries are reproduced."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    scale = float(np.max(np.abs(ref)))
    den = np.maximum(np.abs(ref), max(floor * scale, 1e-300))
    return float(np.max(np.abs(x - ref) / den))


def rel_err(x, ref) -> float:
    """max|x - ref| / max|ref| (the tolerance the tests assert on); records the floored elementwise
    error beside it."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    den = float(np.max(np.abs(ref)))
    e = float(np.max(np.abs(x - ref)) / max(den, 1e-30))
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    ERRORS.append((test, e, elem_rel_err(x, ref)))
    return e


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def cuda_device():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import linear_attention_recurrence_chunked_gb300 as la
    from linear_attention_recurrence_chunked_gb300 import _build
    _build.build()
    la.load_library()
    return torch.device("cuda:0")
