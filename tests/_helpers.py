"""Shared test utilities: seeded inputs to torch / numpy, parity metrics."""
from __future__ import annotations

import numpy as np

from synthetic import bf16_bits_to_f32, generate


def host_arrays(spec):
    """(array_for_gpu, float64_for_oracle) of one TensorSpec."""
    a = generate(spec, workers=1)
    if spec.dtype == "bf16":
        return a, bf16_bits_to_f32(a).astype(np.float64)
    return a, a.astype(np.float64)


def to_device(a: np.ndarray, dtype: str, device="cuda"):
    import torch

    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(device)


def rel_fro(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / np.linalg.norm(b))


def reversed_upper_factor(Hd: np.ndarray) -> np.ndarray:
    """Upper F with Hd = F F^T, from numpy's lower Cholesky of the index-reversed matrix."""
    J = np.arange(Hd.shape[0])[::-1]
    L = np.linalg.cholesky(Hd[np.ix_(J, J)])
    return L[np.ix_(J, J)]
