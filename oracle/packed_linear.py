"""The quantized linear layer computed from its packed form, float64.  TEST INFRASTRUCTURE ONLY.

[LowBit] "El balance de errores de la inferencia de pocos bits", section 1: a
quantized weight is stored as integer codes with a per-group scale and zero
point, and the dequantized weight is ``ŵ = s (q - z)``; section 6: inference
kernels unpack the codes and dequantize them on the fly inside the matrix
product.  [EoRA-blog], "Bucear en el espacio propio en busca de un adaptador":
the compensated layer adds the rank-r adapter, ``W ≈ Ŵ + B A``.  The same
adapter form carries the GPTQ-intrinsic LoRA (B = R, A = L^T).

So the layer output on inputs X (n x cols) is

    Y = X Ŵ^T + (X A^T) B^T,     Ŵ[m, k] = s[k / g, m] (q[m, k] - z[k / g, m])

and the loss of the quantized layer, measured from the packed form, is
``||X W^T - Y||_F^2``.

Here Ŵ is the exact real value s (q - z) (float64 product of the float32 scale
and the integer), not its float32 rounding: that is the value the packed form
stores.
"""
from __future__ import annotations

import numpy as np

from . import pack as opk

F64 = np.float64


def dequantize(qweight, scales, qzeros, bits: int, group: int, rows: int, cols: int) -> np.ndarray:
    """Ŵ (rows x cols, float64) from qweight [cols*b/32][rows], scales [cols/g][rows] and
    qzeros [cols/g][rows*b/32]."""
    codes = opk.unpack_qweight(np.asarray(qweight), bits, rows, cols).astype(F64)
    zeros = opk.unpack_qzeros(np.asarray(qzeros), bits, rows).astype(F64)  # [cols/g][rows]
    s = np.asarray(scales, dtype=F64)                                       # [cols/g][rows]
    zr = np.repeat(zeros.T, group, axis=1)                                  # rows x cols
    sr = np.repeat(s.T, group, axis=1)
    return sr * (codes - zr)


def packed_linear(X, qweight, scales, qzeros, bits: int, group: int, rows: int, cols: int, A=None, B=None):
    """Y = X Ŵ^T (+ (X A^T) B^T), float64."""
    X = np.asarray(X, dtype=F64)
    Y = X @ dequantize(qweight, scales, qzeros, bits, group, rows, cols).T
    if A is not None and B is not None and np.asarray(A).shape[0] > 0:
        Y = Y + (X @ np.asarray(A, dtype=F64).T) @ np.asarray(B, dtype=F64).T
    return Y


def output_loss(X, W, Y) -> float:
    """||X W^T - Y||_F^2: the layer's output error on X, from the packed layer's output Y."""
    D = np.asarray(X, dtype=F64) @ np.asarray(W, dtype=F64).T - np.asarray(Y, dtype=F64)
    return float(np.einsum("ij,ij->", D, D))
