"""EoRA low-rank compensation of the quantization error, float64.  TEST INFRASTRUCTURE ONLY.

[EoRA-blog], "Bucear en el espacio propio en busca de un adaptador":

* the compression error ``ΔW = W - Ŵ`` is approximated by a rank-r product
  ``B A`` with ``A`` (r x cols) and ``B`` (rows x r) the two LoRA factors;
* the plain method takes the SVD ``ΔW = U Σ V^T`` and keeps ``B = U_r Σ_r``,
  ``A = V_r^T``;
* EoRA first projects ΔW into the eigenspace of the input covariance,
  ``X~ X~^T = Q Λ Q^T`` (our ``H``, cols x cols), ``ΔW' = ΔW Q'``, truncates the
  SVD of ΔW' and projects the result back to the original space.

Readings of points the pages leave open:

* ``Q' = Q sqrt(Λ)``.  The page prints ``Q' = QΛ``, but states that the
  projection makes the truncation minimise the layer loss rather than the raw
  weight error; that holds only with the square root, because then
  ``||ΔW'||_F^2 = tr(ΔW H ΔW^T)``.
* "Project back": ``B = U_r Σ_r`` and ``A = V_r^T Q'^{-1} = V_r^T Λ^{-1/2} Q^T``,
  so that ``B A = (ΔW' truncated) Q'^{-1}``.
* H is used as passed (undamped) and must be positive definite.
* Each rank-1 term's sign is fixed so that the largest-magnitude entry of its
  column of B is positive.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


def _normalize_signs(A: np.ndarray, B: np.ndarray):
    for i in range(B.shape[1]):
        k = int(np.argmax(np.abs(B[:, i])))
        if B[k, i] < 0:
            B[:, i] *= -1.0
            A[i, :] *= -1.0
    return A, B


def plain_svd(dW: np.ndarray, r: int):
    """Plain truncated SVD of the error: ``B = U_r Σ_r``, ``A = V_r^T``."""
    U, sig, Vt = np.linalg.svd(np.asarray(dW, dtype=F64), full_matrices=False)
    B = U[:, :r] * sig[:r]
    A = Vt[:r].copy()
    A, B = _normalize_signs(A, B)
    return A, B, sig


def eora(dW: np.ndarray, H: np.ndarray, r: int):
    """EoRA factors (A, B) and the singular values of the projected error."""
    H = np.asarray(H, dtype=F64)
    lam, Q = np.linalg.eigh(0.5 * (H + H.T))
    if lam.min() <= 0:
        raise ValueError("EoRA needs a positive definite H")
    root = np.sqrt(lam)
    M = np.asarray(dW, dtype=F64) @ (Q * root)  # ΔW' = ΔW Q sqrt(Λ)
    U, sig, Vt = np.linalg.svd(M, full_matrices=False)
    B = U[:, :r] * sig[:r]
    A = (Vt[:r] / root) @ Q.T
    A, B = _normalize_signs(A, B)
    return A, B, sig


def compensated_loss(dW: np.ndarray, A: np.ndarray, B: np.ndarray, H0: np.ndarray) -> float:
    """``1/2 tr((ΔW - B A) H0 (ΔW - B A)^T)``: the layer loss left after compensation."""
    Rm = np.asarray(dW, dtype=F64) - np.asarray(B, dtype=F64) @ np.asarray(A, dtype=F64)
    return 0.5 * float(np.einsum("ij,ij->", Rm @ np.asarray(H0, dtype=F64), Rm))
