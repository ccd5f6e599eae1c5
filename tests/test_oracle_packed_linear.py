"""Pins of the packed-linear oracle (CPU only).

* Unpacking the GPTQ oracle's packed output gives back its Ŵ (float32 rounding
  of s (q - z)) exactly: the packed form loses nothing.
* On a tiny layer the output equals a brute-force triple loop over the codes.
* The loss measured from the output, ||X W^T - Y||^2, equals the Hessian form
  1/2 tr(ΔW H ΔW^T) with H = 2 X^T X (two independent routes).
* A full-rank EoRA adapter of the GPTQ error makes the layer exact: the loss
  from the packed form drops to rounding level.
"""
import numpy as np
import pytest

from oracle import eora as oe
from oracle import gptq as og
from oracle import pack as opk
from oracle import packed_linear as pl


def _quantized_layer(rows, cols, n, bits, group, seed):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((n, cols))
    X[:, rng.choice(cols, 2, replace=False)] *= 20.0
    W = rng.standard_normal((rows, cols)) * 0.02
    H = og.hessian(X)
    q = og.quantize_layer(W, H, bits, group, 0.01)
    packed = (opk.pack_qweight(q["codes"], bits), q["scales"], opk.pack_qzeros(q["zeros"], bits))
    return X, W, H, q, packed


@pytest.mark.parametrize("bits,group", [(2, 32), (3, 64), (4, 128)])
def test_unpacking_returns_the_sweep_weights(bits, group):
    rows, cols = 64, 256
    X, W, H, q, (qw, s, qz) = _quantized_layer(rows, cols, 512, bits, group, 1 + bits)
    W_hat = pl.dequantize(qw, s, qz, bits, group, rows, cols)
    assert np.array_equal(W_hat.astype(np.float32), q["W_hat"])


def test_tiny_layer_against_a_triple_loop():
    rows, cols, n, bits, group = 32, 64, 3, 3, 32
    rng = np.random.default_rng(2)
    codes = rng.integers(0, 8, (rows, cols)).astype(np.uint8)
    zeros = rng.integers(0, 8, (cols // group, rows)).astype(np.uint8)
    scales = rng.uniform(0.01, 0.1, (cols // group, rows)).astype(np.float32)
    X = rng.standard_normal((n, cols))
    A = rng.standard_normal((2, cols))
    B = rng.standard_normal((rows, 2))
    Y = pl.packed_linear(X, opk.pack_qweight(codes, bits), scales, opk.pack_qzeros(zeros, bits), bits, group, rows,
                         cols, A, B)
    ref = np.zeros((n, rows))
    for t in range(n):
        for m in range(rows):
            acc = 0.0
            for k in range(cols):
                g = k // group
                acc += X[t, k] * float(scales[g, m]) * (int(codes[m, k]) - int(zeros[g, m]))
            for i in range(2):
                acc += sum(X[t, k] * A[i, k] for k in range(cols)) * B[m, i]
            ref[t, m] = acc
    assert np.allclose(Y, ref, rtol=1e-12, atol=1e-12)


def test_loss_from_the_output_equals_the_hessian_form():
    rows, cols, n, bits, group = 64, 256, 600, 2, 64
    X, W, H, q, (qw, s, qz) = _quantized_layer(rows, cols, n, bits, group, 3)
    rng = np.random.default_rng(4)
    A = rng.standard_normal((4, cols)) * 1e-3
    B = rng.standard_normal((rows, 4)) * 1e-3
    Y = pl.packed_linear(X, qw, s, qz, bits, group, rows, cols, A, B)
    W_eff = pl.dequantize(qw, s, qz, bits, group, rows, cols) + B @ A
    assert pl.output_loss(X, W, Y) == pytest.approx(og.layer_loss(W, W_eff, H), rel=1e-10)


def test_full_rank_adapter_makes_the_layer_exact():
    rows, cols, n, bits, group = 64, 64, 400, 2, 32
    X, W, H, q, (qw, s, qz) = _quantized_layer(rows, cols, n, bits, group, 5)
    W_hat = pl.dequantize(qw, s, qz, bits, group, rows, cols)
    A, B, _ = oe.eora(W - W_hat, H, cols)
    l_plain = pl.output_loss(X, W, pl.packed_linear(X, qw, s, qz, bits, group, rows, cols))
    l_adapted = pl.output_loss(X, W, pl.packed_linear(X, qw, s, qz, bits, group, rows, cols, A, B))
    assert l_adapted <= 1e-18 * l_plain + 1e-20
