"""OLrC + Bid-Up refinement of a quantized layer with a low-rank correction, float64.
TEST INFRASTRUCTURE ONLY.

[GPTQ-LoRA] "Resumen Técnico: GPTQ-intrinsic LoRA", "Metodología" item 4
"Refinamiento Bid-Up": the layer W ≈ Q + L R is refined by alternating two
steps, each of which minimizes the layer objective ||X W^T - X (Q + R L^T)^T||^2
over part of the variables, so the objective never increases:

* OLrC (optimal low-rank compensation): the best rank-r correction for a fixed
  Q.  In this library's notation the correction is B A (B rows x r, A r x cols)
  and the objective is 1/2 tr(D H D^T) with D = W - Q - B A, H = 2 X^T X; the
  minimizer over rank-r B A is the truncated SVD of the error in the metric of
  H, which is the EoRA problem (oracle.eora).
* Bid-Up: Q on the fixed grid (each group's scale and zero point kept), B A
  fixed, improved by coordinate updates.  With target T = W - B A, residual
  r = T - Ŵ and gradient g = r H (per row), changing ŵ_j by d changes the
  row's objective r H r^T by -2 d g_j + d^2 H_jj, so the best grid value for
  coordinate j alone is the grid point nearest ŵ_j + g_j / H_jj:
  q' = clamp(q + rint(g_j / (H_jj s)), 0, 2^b - 1).  One sweep takes the
  columns in order (Gauss-Seidel), updating r and g after every change.

Readings of points the pages leave open:

* H is used undamped (as EoRA uses it); it must be positive definite for OLrC.
* The integer decision rint(g_j / (H_jj s)) is taken in float32 from the
  float32 roundings of g_j, H_jj and s (ties to even), the precision of the
  GPU kernel; ŵ' = s (q' - z) is stored rounded to float32, as the GPTQ sweep
  stores Ŵ.  Everything else is float64.
"""
from __future__ import annotations

import numpy as np

from . import eora as oe

F32 = np.float32
F64 = np.float64


def objective(W, W_hat, H, A=None, B=None) -> float:
    """1/2 tr(D H D^T), D = W - Ŵ - B A (= ||X (W - Ŵ - B A)^T||^2 for H = 2 X^T X)."""
    D = np.asarray(W, F64) - np.asarray(W_hat, F64)
    if A is not None and B is not None and np.asarray(A).shape[0] > 0:
        D = D - np.asarray(B, F64) @ np.asarray(A, F64)
    return 0.5 * float(np.einsum("ij,ij->", D @ np.asarray(H, F64), D))


def olrc(W, W_hat, H, r: int):
    """The optimal rank-r correction for fixed Ŵ: (A, B, sigma) of EoRA on W - Ŵ."""
    return oe.eora(np.asarray(W, F64) - np.asarray(W_hat, F64), H, r)


def dequant(codes, scales, zeros, group: int) -> np.ndarray:
    """Ŵ = s (q - z), rounded to float32 (rows x cols), from codes and [cols/g][rows] scales and zeros."""
    s = np.repeat(np.asarray(scales, F32).T, group, axis=1)
    z = np.repeat(np.asarray(zeros).T.astype(F32), group, axis=1)
    return (s * (np.asarray(codes).astype(F32) - z)).astype(F32)


def bidup_sweep(W, codes, scales, zeros, H, bits: int, group: int, A=None, B=None) -> dict:
    """One Bid-Up sweep over all columns in order.  Returns the new codes, Ŵ and the number of
    changed codes."""
    W = np.asarray(W, F64)
    H = np.asarray(H, F64)
    rows, cols = W.shape
    maxq = 2 ** bits - 1
    T = W - (np.asarray(B, F64) @ np.asarray(A, F64) if A is not None and np.asarray(A).shape[0] > 0 else 0.0)
    q = np.array(codes, dtype=np.int64, copy=True)
    What = dequant(q, scales, zeros, group)
    res = T - What.astype(F64)
    g = res @ H
    changed = 0
    for j in range(cols):
        s = np.asarray(scales, F32)[j // group]
        z = np.asarray(zeros)[j // group].astype(np.int64)
        u = g[:, j].astype(F32) / (F32(H[j, j]) * s)
        qn = np.clip(q[:, j] + np.rint(u).astype(np.int64), 0, maxq)
        moved = qn != q[:, j]
        if moved.any():
            wn = (s * (qn - z).astype(F32)).astype(F32)
            d = wn.astype(F64) - What[:, j].astype(F64)
            d[~moved] = 0.0
            res[:, j] -= d
            g -= np.outer(d, H[j])
            q[:, j] = qn
            What[:, j] = np.where(moved, wn, What[:, j])
            changed += int(moved.sum())
    return dict(codes=q.astype(np.uint8), W_hat=What, changed=changed)


def refine(W, codes, scales, zeros, H, bits: int, group: int, r: int, cycles: int) -> dict:
    """`cycles` rounds of OLrC then Bid-Up, from the given codes.  Returns the final codes, Ŵ, A, B and
    the objective after every step (starting with the objective of the codes alone)."""
    q = np.array(codes, copy=True)
    What = dequant(q, scales, zeros, group)
    hist = [objective(W, What, H)]
    A = B = None
    for _ in range(cycles):
        A, B, _ = olrc(W, What, H, r)
        hist.append(objective(W, What, H, A, B))
        out = bidup_sweep(W, q, scales, zeros, H, bits, group, A, B)
        q, What = out["codes"], out["W_hat"]
        hist.append(objective(W, What, H, A, B))
    return dict(codes=q, W_hat=What, A=A, B=B, objective=hist)
