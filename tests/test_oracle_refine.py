"""Pins of the OLrC + Bid-Up oracle (CPU only).

* Bid-Up never increases the objective (each coordinate step minimizes a 1-D
  quadratic over a grid that contains the current value), and at a fixed point
  every coordinate is optimal on its grid: checked by trying every grid value of
  every coordinate (brute force).
* With a diagonal H the coordinates decouple: one sweep lands on the nearest grid
  point of the target W - B A (round to nearest on the fixed grid).
* On tiny layers the refined objective is never below the exhaustive optimum over
  all code vectors on the grid, and a sweep started at that optimum stays there.
* OLrC is the EoRA optimum: no other rank-r correction tried does better, and the
  alternating cycle never increases the objective.
"""
import itertools

import numpy as np
import pytest

from oracle import gptq as og
from oracle import refine as rf


def _layer(rows, cols, n, bits, group, seed, outliers=2):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((n, cols))
    if outliers:
        X[:, rng.choice(cols, outliers, replace=False)] *= 20.0
    W = rng.standard_normal((rows, cols)) * 0.02
    H = og.hessian(X)
    q = og.quantize_layer(W, H, bits, group, 0.01)
    return W, H, q


def _coordinate_optimal(W, codes, scales, zeros, H, bits, group, A=None, B=None, tol=1e-12):
    rows, cols = W.shape
    base = rf.dequant(codes, scales, zeros, group)
    for i in range(rows):
        for j in range(cols):
            f0 = rf.objective(W[i:i + 1], base[i:i + 1], H, A, None if B is None else B[i:i + 1])
            for v in range(2 ** bits):
                c = codes[i:i + 1].copy()
                c[0, j] = v
                wv = rf.dequant(c, scales[:, i:i + 1], zeros[:, i:i + 1], group)
                f = rf.objective(W[i:i + 1], wv, H, A, None if B is None else B[i:i + 1])
                assert f >= f0 * (1 - tol) - 1e-18, (i, j, v, f, f0)


def test_bidup_never_increases_and_ends_coordinate_optimal():
    rows, cols, bits, group = 6, 16, 2, 8
    W, H, q = _layer(rows, cols, 64, bits, group, 1)
    codes = q["codes"]
    f = rf.objective(W, q["W_hat"], H)
    for _ in range(10):
        out = rf.bidup_sweep(W, codes, q["scales"], q["zeros"], H, bits, group)
        f_new = rf.objective(W, out["W_hat"], H)
        assert f_new <= f * (1 + 1e-12)
        f, codes = f_new, out["codes"]
        if out["changed"] == 0:
            break
    assert out["changed"] == 0
    _coordinate_optimal(W, codes, q["scales"], q["zeros"], H, bits, group)


def test_diagonal_hessian_is_round_to_nearest_of_the_target():
    rows, cols, bits, group = 20, 32, 3, 16
    rng = np.random.default_rng(2)
    W = rng.standard_normal((rows, cols)) * 0.02
    H = np.diag(rng.uniform(0.5, 2.0, cols))
    q = og.rtn(W, bits, group)
    A = rng.standard_normal((2, cols)) * 0.01
    B = rng.standard_normal((rows, 2)) * 0.01
    out = rf.bidup_sweep(W, q["codes"], q["scales"], q["zeros"], H, bits, group, A, B)
    T = (W - B @ A).astype(np.float32)
    s = np.repeat(q["scales"].T, group, axis=1)
    z = np.repeat(q["zeros"].T.astype(np.float32), group, axis=1)
    expect = np.clip(np.rint(T / s) + z, 0, 2 ** bits - 1).astype(np.uint8)
    assert np.array_equal(out["codes"], expect)


def test_tiny_layers_against_exhaustive_search():
    rows, cols, bits, group = 5, 6, 2, 6
    W, H, q = _layer(rows, cols, 24, bits, group, 3, outliers=1)
    out = q
    codes = q["codes"]
    for _ in range(20):
        out = rf.bidup_sweep(W, codes, q["scales"], q["zeros"], H, bits, group)
        codes = out["codes"]
    for i in range(rows):
        grid = np.array(list(itertools.product(range(2 ** bits), repeat=cols)), dtype=np.uint8)
        s, z = q["scales"][0, i], np.float32(q["zeros"][0, i])
        deq = (s * (grid.astype(np.float32) - z)).astype(np.float64)
        D = W[i][None, :] - deq
        vals = 0.5 * np.einsum("ij,jk,ik->i", D, H, D)
        best = vals.min()
        mine = rf.objective(W[i:i + 1], out["W_hat"][i:i + 1], H)
        assert mine >= best * (1 - 1e-12)
        # a sweep from the optimum stays there
        c_opt = grid[np.argmin(vals)][None, :]
        stay = rf.bidup_sweep(W[i:i + 1], c_opt, q["scales"][:, i:i + 1], q["zeros"][:, i:i + 1], H, bits, group)
        assert stay["changed"] == 0


def test_olrc_is_optimal_and_the_cycle_never_increases():
    rows, cols, bits, group, r = 48, 64, 2, 32, 4
    W, H, q = _layer(rows, cols, 256, bits, group, 4)
    A, B, _ = rf.olrc(W, q["W_hat"], H, r)
    f_opt = rf.objective(W, q["W_hat"], H, A, B)
    rng = np.random.default_rng(5)
    for _ in range(20):  # perturbed or random rank-r corrections do no better
        Bp = B + rng.standard_normal(B.shape) * 1e-3
        Ap = A + rng.standard_normal(A.shape) * 1e-3
        assert rf.objective(W, q["W_hat"], H, Ap, Bp) >= f_opt * (1 - 1e-12)
    res = rf.refine(W, q["codes"], q["scales"], q["zeros"], H, bits, group, r, cycles=3)
    hist = res["objective"]
    assert all(b <= a * (1 + 1e-12) for a, b in zip(hist, hist[1:])), hist
    assert hist[-1] < hist[1]  # Bid-Up improved on OLrC alone for this layer


def test_planted_mistake_in_the_decision_is_caught():
    """A sign error in the coordinate step (moving against the gradient) raises the objective."""
    rows, cols, bits, group = 6, 16, 2, 8
    W, H, q = _layer(rows, cols, 64, bits, group, 6)
    codes = q["codes"].astype(np.int64)
    What = rf.dequant(codes, q["scales"], q["zeros"], group)
    g = (W - What) @ H
    j = 3
    s = q["scales"][j // group]
    u = g[:, j].astype(np.float32) / (np.float32(H[j, j]) * s)
    bad = codes.copy()
    bad[:, j] = np.clip(codes[:, j] - np.rint(u).astype(np.int64), 0, 2 ** bits - 1)
    good = rf.bidup_sweep(W, codes.astype(np.uint8), q["scales"], q["zeros"], H, bits, group)
    f0 = rf.objective(W, What, H)
    assert rf.objective(W, rf.dequant(bad, q["scales"], q["zeros"], group), H) > f0
    assert rf.objective(W, good["W_hat"], H) <= f0
