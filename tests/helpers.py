"""Shared helpers of the test suite (no arithmetic of the method here)."""
import numpy as np
import pytest
import torch

# Tolerances on the max relative error max|x - ref| / max|ref| per tensor:
# fp32 inputs 1e-4; bf16 inputs with fp32 state 2e-2.
TOL = {torch.float32: 1e-4, torch.bfloat16: 2e-2}


def rel_err(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(x - ref)) / max(den, 1e-30))


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
