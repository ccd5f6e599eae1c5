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


def check_sigma(sg, sig, r, rtol=1e-3, reach=16):
    """The GPU's r singular values against the oracle's.  Where sigma_i stands apart from sigma_(i+1)
    by more than rtol, within rtol of it.  Inside a cluster of nearly equal values an individual value
    is not determined to rtol by a subspace of finite accuracy, only the cluster is: there sigma_i of
    the GPU lies between sigma_(i+reach) and sigma_i, each widened by rtol.  The compensated loss is
    the criterion on the subspace as a whole."""
    sg = np.asarray(sg, dtype=np.float64)
    for i in range(r):
        if sig[i] > sig[i + 1] * (1 + rtol):
            assert abs(sg[i] - sig[i]) <= rtol * sig[i], (i, sg[i], sig[i])
        else:
            lo = sig[min(i + reach, len(sig) - 1)] * (1 - rtol)
            assert lo <= sg[i] <= sig[i] * (1 + rtol), (i, sg[i], sig[i], lo)
