"""GPTQ layer quantization, float64, eager and unblocked.  TEST INFRASTRUCTURE ONLY.

What it computes, and from where:

* The layer loss is the squared output error of the linear layer on the
  calibration set, ``||X W^T - X Ŵ^T||_F^2`` ([GPTQ-LoRA], "Declaración del
  Problema", the objective ``min ||XW - X(Q+LR)||_F^2`` with L R = 0; [LowBit]
  section 2: a weight perturbation ΔW produces output error ΔW x, amplified by
  the second-order statistics of the input).  Its Hessian in each weight row
  is ``H = 2 X^T X`` ([GPTQ-wiki] "Enfoque Técnico": GPTQ uses the Hessian of
  the loss), so ``loss = 1/2 tr(ΔW H ΔW^T)``.
* GPTQ quantizes the columns of W one at a time in a fixed order and, after
  each column, applies the closed-form Optimal-Brain-Quantization update to
  the columns not yet quantized ([GPTQ-wiki] "Enfoque Técnico").  With
  ``U`` the upper Cholesky factor of the (damped) inverse Hessian, ``U^T U =
  H^-1``, that update is ``e_j = (w_j - ŵ_j) / U_jj`` and
  ``W[:, k] -= e_j U_jk`` for every later column k.
* The grid is uniform affine, one scale and zero point per group of ``g``
  consecutive input columns of each row ([LowBit] section 1; [GPTQ-wiki]
  "Enfoque Técnico": per-group scale factors).

Readings of points the pages leave open:

* H is the literal ``2 X^T X`` (no 1/N).  Codes do not depend on the scale of
  H because the damping is relative to ``mean(diag H)``.
* Damping: ``H += damp * mean(diag H) * I``.  A dead input (``H_ii == 0``)
  gets ``H_ii = 1`` before damping and its weights are set to zero.
* The grid always contains 0: ``xmin = min(0, min w)``, ``xmax = max(0, max
  w)``; an all-zero group uses ``[-1, 1]``.  ``s = (xmax - xmin) / maxq``,
  ``z = rint(-xmin / s)``, ``q = clamp(rint(w / s) + z, 0, maxq)``,
  ``ŵ = s (q - z)``, ``maxq = 2^bits - 1``.  ``rint`` rounds ties to even.
* A group's scale and zero are taken at its first column, from the weights as
  updated by every earlier column.
* The decisions that produce integers -- the grid (s, z), the code q and the
  dequantized value ŵ -- are taken in float32, the precision of the GPU
  kernel, from the float32 rounding of the oracle's float64 weights.  All
  other arithmetic is float64.
"""
from __future__ import annotations

import numpy as np

F32 = np.float32
F64 = np.float64


# --------------------------------------------------------------------------- H
def hessian(X: np.ndarray, H: np.ndarray | None = None, chunk: int = 8192) -> np.ndarray:
    """``H += 2 X^T X`` in float64 from the exact input values ([GPTQ-wiki] "Enfoque Técnico")."""
    n, c = X.shape
    if H is None:
        H = np.zeros((c, c), dtype=F64)
    for r0 in range(0, n, chunk):
        xc = np.asarray(X[r0:r0 + chunk], dtype=F64)
        H += 2.0 * (xc.T @ xc)
    return H


def prepare_hessian(H: np.ndarray, damp: float):
    """Dead inputs and relative damping.  Returns (H_damped, dead_mask)."""
    Hd = np.array(H, dtype=F64, copy=True)
    d = np.diagonal(Hd).copy()
    dead = d == 0.0
    idx = np.flatnonzero(dead)
    Hd[idx, idx] = 1.0
    Hd[np.diag_indices_from(Hd)] += damp * np.mean(np.diagonal(Hd))
    return Hd, dead


def inverse_cholesky_upper(Hd: np.ndarray) -> np.ndarray:
    """Upper-triangular U with ``U^T U = Hd^-1`` (Cholesky factor of the inverse Hessian)."""
    Hinv = np.linalg.inv(Hd)
    Hinv = 0.5 * (Hinv + Hinv.T)
    return np.linalg.cholesky(Hinv).T


# ------------------------------------------------------------------------ grid
def quant_grid(wg: np.ndarray, bits: int):
    """Per-row scale and zero point of one group, in float32.  ``wg``: rows x g."""
    maxq = F32(2 ** bits - 1)
    w = np.asarray(wg, dtype=F32)
    xmin = np.minimum(w.min(axis=1), F32(0))
    xmax = np.maximum(w.max(axis=1), F32(0))
    flat = (xmin == 0) & (xmax == 0)
    xmin = np.where(flat, F32(-1), xmin).astype(F32)
    xmax = np.where(flat, F32(1), xmax).astype(F32)
    s = ((xmax - xmin) / maxq).astype(F32)
    z = np.rint(-xmin / s).astype(F32)
    return s, z


def quantize(w: np.ndarray, s: np.ndarray, z: np.ndarray, bits: int):
    """Codes and dequantized values of one column, in float32."""
    maxq = F32(2 ** bits - 1)
    w = np.asarray(w, dtype=F32)
    q = np.clip(np.rint(w / s) + z, F32(0), maxq).astype(F32)
    wq = (s * (q - z)).astype(F32)
    return q, wq


# ----------------------------------------------------------------------- sweep
def sweep(W: np.ndarray, U: np.ndarray, bits: int, group: int, dead: np.ndarray | None = None) -> dict:
    """The GPTQ column sweep, one column at a time, every later column updated eagerly.

    Returns codes (rows x cols, uint8), scales and zeros ([cols/g][rows]),
    W_hat (float32), row_err = sum_j e_j^2 per row, and the final working W.
    """
    W = np.array(W, dtype=F64, copy=True)
    R, C = W.shape
    if C % group:
        raise ValueError("cols must be a multiple of group")
    if dead is not None and dead.any():
        W[:, dead] = 0.0
    codes = np.zeros((R, C), dtype=np.uint8)
    What = np.zeros((R, C), dtype=F32)
    scales = np.zeros((C // group, R), dtype=F32)
    zeros = np.zeros((C // group, R), dtype=np.uint8)
    row_err = np.zeros(R, dtype=F64)
    for j in range(C):
        if j % group == 0:
            s, z = quant_grid(W[:, j:j + group], bits)
            scales[j // group] = s
            zeros[j // group] = z.astype(np.uint8)
        q, wq = quantize(W[:, j], s, z, bits)
        e = (W[:, j] - wq.astype(F64)) / U[j, j]
        if j + 1 < C:
            W[:, j + 1:] -= np.outer(e, U[j, j + 1:])
        codes[:, j] = q.astype(np.uint8)
        What[:, j] = wq
        row_err += e * e
    return dict(codes=codes, scales=scales, zeros=zeros, W_hat=What, row_err=row_err)


def quantize_layer(W: np.ndarray, H: np.ndarray, bits: int, group: int, damp: float = 0.01) -> dict:
    """The whole layer: dead inputs and damping, U = chol(H^-1)^T, sweep."""
    Hd, dead = prepare_hessian(H, damp)
    U = inverse_cholesky_upper(Hd)
    out = sweep(W, U, bits, group, dead=dead)
    out.update(Hd=Hd, U=U, dead=dead)
    return out


def rtn(W: np.ndarray, bits: int, group: int) -> dict:
    """Round-to-nearest on the same per-group grid: the sweep with no error propagation.

    [GPTQ-wiki] "Rendimiento y Precisión" compares GPTQ against rounding to the
    nearest integer; this is that baseline.
    """
    W = np.asarray(W, dtype=F64)
    R, C = W.shape
    codes = np.zeros((R, C), dtype=np.uint8)
    What = np.zeros((R, C), dtype=F32)
    scales = np.zeros((C // group, R), dtype=F32)
    zeros = np.zeros((C // group, R), dtype=np.uint8)
    for g0 in range(0, C, group):
        s, z = quant_grid(W[:, g0:g0 + group], bits)
        scales[g0 // group] = s
        zeros[g0 // group] = z.astype(np.uint8)
        for j in range(g0, g0 + group):
            q, wq = quantize(W[:, j], s, z, bits)
            codes[:, j] = q.astype(np.uint8)
            What[:, j] = wq
    return dict(codes=codes, scales=scales, zeros=zeros, W_hat=What)


# ------------------------------------------------------------------------ loss
def layer_loss(W: np.ndarray, W_hat: np.ndarray, H0: np.ndarray) -> float:
    """``1/2 tr(ΔW H0 ΔW^T)``; equals ``||X ΔW^T||_F^2`` when ``H0 = 2 X^T X``."""
    dW = np.asarray(W, dtype=F64) - np.asarray(W_hat, dtype=F64)
    return 0.5 * float(np.einsum("ij,ij->", dW @ H0, dW))


def row_losses(W: np.ndarray, W_hat: np.ndarray, H: np.ndarray) -> np.ndarray:
    """Per row ``ΔW_r H ΔW_r^T``."""
    dW = np.asarray(W, dtype=F64) - np.asarray(W_hat, dtype=F64)
    return np.einsum("ij,ij->i", dW @ H, dW)


def output_error(X: np.ndarray, W: np.ndarray, W_hat: np.ndarray) -> float:
    """``||X W^T - X Ŵ^T||_F^2`` computed directly from the activations."""
    dW = np.asarray(W, dtype=F64) - np.asarray(W_hat, dtype=F64)
    Y = np.asarray(X, dtype=F64) @ dW.T
    return float(np.einsum("ij,ij->", Y, Y))
