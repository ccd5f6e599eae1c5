"""GPTQ-intrinsic LoRA, float64.  TEST INFRASTRUCTURE ONLY.

[GPTQ-LoRA] "Resumen Técnico: GPTQ-intrinsic LoRA", "Algoritmo GPTQ-intrinsic
LoRA": the low-rank correction is built inside the GPTQ sweep instead of after
it.

* The calibration matrix is augmented with r extra columns, X~ = [X, X L],
  where L (cols x r) holds the r leading right singular vectors of X
  ("L = V_r").  Its Hessian is H~ = 2 X~^T X~ = [[H, H L], [L^T H, L^T H L]]
  with H = 2 X^T X, so it follows from H and L alone.
* GPTQ runs on the augmented weights W~ = [W, 0] (the page's [W; 0] in its
  input-by-output orientation): the first cols columns are quantized (Q), the
  last r columns start at zero, are never quantized and absorb the
  quantization error through the ordinary GPTQ updates; their final values
  are R (rows x r).
* Then X~ [Q, R]^T = X Q^T + X L R^T, i.e. W ~ Q + R L^T: a LoRA pair with
  B = R and A = L^T.

Readings of points the pages leave open:

* The Hessian is damped like GPTQ's, H~ + damp * mean(diag H~) * I, which
  makes it positive definite for damp > 0.  Two factorizations give the upper
  factor U of its inverse (U^T U = H~_d^-1): GPTQ's (inverse, then Cholesky)
  and the page's eigendecomposition + QR ("Detalles de Implementación"):
  H~_d = Q Λ Q^T, M = Λ^(-1/2) Q^T, M = O R with O orthogonal and R upper
  triangular, so M^T M = R^T R = H~_d^-1 and U = R with a positive diagonal.
  The second never forms the inverse; its rounding grows with the square root
  of the condition number instead of the condition number, which is what lets
  the damping be small.  damp must be > 0: at 0 the augmented Hessian is
  singular (its last r columns are combinations of the first ones) and the
  factor of its inverse does not exist.
* L is an input.  The leading singular subspace of X is not unique when
  singular values are close, so GPTQ-intrinsic LoRA is defined here for a given
  L (orthonormal columns); top_right_singular_vectors gives the page's choice.
"""
from __future__ import annotations

import numpy as np

from . import gptq as og

F64 = np.float64


def top_right_singular_vectors(H: np.ndarray, r: int):
    """Leading r eigenvectors of H = 2 X^T X (the right singular vectors of X), eigenvalues
    descending; each vector's largest-magnitude entry is made positive."""
    lam, Q = np.linalg.eigh(0.5 * (np.asarray(H, F64) + np.asarray(H, F64).T))
    idx = np.argsort(lam)[::-1][:r]
    V = Q[:, idx].copy()
    for i in range(r):
        k = int(np.argmax(np.abs(V[:, i])))
        if V[k, i] < 0:
            V[:, i] *= -1.0
    return V, lam[idx]


def augmented_hessian(H: np.ndarray, L: np.ndarray) -> np.ndarray:
    """H~ = [[H, H L], [L^T H, L^T H L]]: the Hessian of the augmented calibration [X, X L]."""
    H = np.asarray(H, F64)
    L = np.asarray(L, F64)
    HL = H @ L
    top = np.concatenate([H, HL], axis=1)
    bot = np.concatenate([HL.T, L.T @ HL], axis=1)
    return np.concatenate([top, bot], axis=0)


def sweep_partial(W: np.ndarray, U: np.ndarray, bits: int, group: int, n_quant: int, dead=None) -> dict:
    """The GPTQ column sweep over the first n_quant columns only: each of them is quantized and its
    scaled error updates every later column, including the columns from n_quant on, which are never
    quantized.  Returns the outputs of gptq.sweep for the quantized columns (row_err = sum_j e_j^2 over
    them) and `free`, the final values of the other columns."""
    W = np.array(W, dtype=F64, copy=True)
    R, C = W.shape
    if n_quant % group:
        raise ValueError("n_quant must be a multiple of group")
    if dead is not None and dead.any():
        W[:, dead] = 0.0
    codes = np.zeros((R, n_quant), dtype=np.uint8)
    What = np.zeros((R, n_quant), dtype=np.float32)
    scales = np.zeros((n_quant // group, R), dtype=np.float32)
    zeros = np.zeros((n_quant // group, R), dtype=np.uint8)
    row_err = np.zeros(R, dtype=F64)
    for j in range(n_quant):
        if j % group == 0:
            s, z = og.quant_grid(W[:, j:j + group], bits)
            scales[j // group] = s
            zeros[j // group] = z.astype(np.uint8)
        q, wq = og.quantize(W[:, j], s, z, bits)
        e = (W[:, j] - wq.astype(F64)) / U[j, j]
        W[:, j + 1:] -= np.outer(e, U[j, j + 1:])
        codes[:, j] = q.astype(np.uint8)
        What[:, j] = wq
        row_err += e * e
    return dict(codes=codes, scales=scales, zeros=zeros, W_hat=What, row_err=row_err, free=W[:, n_quant:].copy())


def inverse_cholesky_upper_eigqr(Hd: np.ndarray) -> np.ndarray:
    """Upper-triangular U with U^T U = Hd^-1 from the eigendecomposition of Hd and a QR factorization
    ([GPTQ-LoRA] "Detalles de Implementación"): Hd = Q Λ Q^T, M = Λ^(-1/2) Q^T = O R, U = R with its
    rows' signs chosen so that the diagonal is positive.  Hd must be positive definite."""
    Hd = np.asarray(Hd, F64)
    lam, Q = np.linalg.eigh(0.5 * (Hd + Hd.T))
    if lam.min() <= 0:
        raise ValueError("the damped Hessian is not positive definite")
    M = (Q / np.sqrt(lam)).T
    R = np.linalg.qr(M, mode="r")
    return R * np.sign(np.diagonal(R))[:, None]


def intrinsic_lora(W: np.ndarray, H: np.ndarray, L: np.ndarray, bits: int, group: int, damp: float = 0.01,
                   factor: str = "cholesky") -> dict:
    """GPTQ-intrinsic LoRA of one layer for a given L (cols x r).  Returns the sweep outputs for Q,
    B = R (rows x r), A = L^T (r x cols) and the damped augmented Hessian.  factor: "cholesky"
    (GPTQ's inverse + Cholesky) or "eigqr" (the page's eigendecomposition + QR)."""
    W = np.asarray(W, F64)
    rows, cols = W.shape
    r = L.shape[1]
    if not damp > 0:
        raise ValueError("damp must be > 0: the augmented Hessian itself is singular")
    Ht = augmented_hessian(H, L)
    Hd, dead = og.prepare_hessian(Ht, damp)
    U = inverse_cholesky_upper_eigqr(Hd) if factor == "eigqr" else og.inverse_cholesky_upper(Hd)
    Wt = np.concatenate([W, np.zeros((rows, r))], axis=1)
    out = sweep_partial(Wt, U, bits, group, cols, dead=dead)
    out.update(B=out.pop("free"), A=np.asarray(L, F64).T.copy(), Hd=Hd, dead=dead)
    return out


def free_columns_optimum(W: np.ndarray, W_hat: np.ndarray, Hd: np.ndarray) -> np.ndarray:
    """For fixed quantized columns, the values of the free columns that minimize the (damped)
    augmented quadratic (w~ - [q, f]) Hd (w~ - [q, f])^T per row, with w~ = [w, 0]:
    f = Hd_ff^-1 Hd_fq (w - q).  A closed form that the sweep's final free columns must equal."""
    W = np.asarray(W, F64)
    cols = W.shape[1]
    d = W - np.asarray(W_hat, F64)
    Hff = Hd[cols:, cols:]
    Hfq = Hd[cols:, :cols]
    return np.linalg.solve(Hff, Hfq @ d.T).T
