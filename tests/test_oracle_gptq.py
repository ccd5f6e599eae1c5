"""Pins of the GPTQ oracle against brute force, closed forms and invariants (CPU only).

Each pin is checked independently of the oracle's own formulas: brute-force
Optimal-Brain-Quantization with explicit inverses of the remaining Hessian,
exhaustive search over all code vectors, the reduction to round-to-nearest for
a diagonal Hessian, the error identity of the OBS update, a blocked lazy-batch
sweep, and the blocked form of the sweep that uses the Cholesky factor of H
itself instead of the factor of its inverse.
"""
import itertools

import numpy as np
import pytest

from oracle import gptq

RNG = np.random.default_rng(1234)


def _spd(c, n=None, outliers=0, rng=RNG):
    n = n or 4 * c
    X = rng.standard_normal((n, c))
    if outliers:
        X[:, rng.choice(c, outliers, replace=False)] *= 20.0
    return gptq.hessian(X), X


def _layer(r, c, rng=RNG, std=0.02):
    return rng.standard_normal((r, c)) * std


# ----------------------------------------------------------------- hessian ---
def test_hessian_exact_on_integer_inputs():
    rng = np.random.default_rng(5)
    X = rng.integers(-7, 8, size=(37, 6)).astype(np.float32)
    H = gptq.hessian(X, chunk=8)
    ref = np.zeros((6, 6), dtype=object)
    for row in X.astype(int).tolist():
        for i in range(6):
            for j in range(6):
                ref[i, j] += 2 * row[i] * row[j]
    assert np.array_equal(H, ref.astype(np.float64))


def test_hessian_accumulates():
    X = RNG.standard_normal((50, 5))
    H = gptq.hessian(X[:20])
    gptq.hessian(X[20:], H=H)
    ref = 2.0 * sum(np.outer(x, x) for x in X)
    assert np.allclose(H, ref, rtol=1e-13, atol=1e-12)


def test_prepare_hessian_dead_and_damping():
    H = np.array([[2.0, 0.0, 1.0], [0.0, 0.0, 0.0], [1.0, 0.0, 4.0]])
    Hd, dead = gptq.prepare_hessian(H, 0.03)
    assert dead.tolist() == [False, True, False]
    delta = 0.03 * (2.0 + 1.0 + 4.0) / 3.0
    ref = np.array([[2.0 + delta, 0.0, 1.0], [0.0, 1.0 + delta, 0.0], [1.0, 0.0, 4.0 + delta]])
    assert np.allclose(Hd, ref, rtol=0, atol=1e-15)
    assert np.array_equal(H[1], [0, 0, 0])  # input untouched


# -------------------------------------------------------- inverse cholesky ---
def test_inverse_cholesky_upper_definition():
    H, _ = _spd(24, outliers=2)
    Hd, _ = gptq.prepare_hessian(H, 0.01)
    U = gptq.inverse_cholesky_upper(Hd)
    assert np.allclose(np.tril(U, -1), 0)
    assert (np.diag(U) > 0).all()
    assert np.allclose(U.T @ U @ Hd, np.eye(24), atol=1e-10)


def test_inverse_cholesky_equals_inverse_of_reversed_factor():
    """U = chol(H^-1)^T equals the inverse of the upper factor of H = Ũ Ũ^T.

    Ũ comes from the ordinary lower Cholesky of the index-reversed matrix, with
    no explicit inverse of H anywhere.  Uniqueness of the Cholesky factor makes
    the two agree."""
    H, _ = _spd(40, outliers=3)
    Hd, _ = gptq.prepare_hessian(H, 0.01)
    J = np.eye(40)[::-1]
    Ut = J @ np.linalg.cholesky(J @ Hd @ J) @ J
    assert np.allclose(np.tril(Ut, -1), 0)
    assert np.allclose(Ut @ Ut.T, Hd, rtol=1e-12, atol=1e-9)
    U = gptq.inverse_cholesky_upper(Hd)
    assert np.allclose(U @ Ut, np.eye(40), atol=1e-10)


# ------------------------------------------------------------------ grid ----
@pytest.mark.parametrize("bits", [2, 3, 4])
def test_grid_membership_and_dequant(bits):
    W = _layer(64, 32)
    W[3, :16] = 0.0  # an all-zero group
    W[5, :16] = np.abs(W[5, :16])  # all-positive group: xmin clamps to 0
    out = gptq.rtn(W, bits, 16)
    maxq = 2 ** bits - 1
    assert out["codes"].max() <= maxq
    assert out["zeros"].max() <= maxq
    s = np.repeat(out["scales"].T, 16, axis=1)
    z = np.repeat(out["zeros"].T.astype(np.float32), 16, axis=1)
    deq = (s * (out["codes"].astype(np.float32) - z)).astype(np.float32)
    assert np.array_equal(deq.view(np.uint32), out["W_hat"].view(np.uint32))
    # zero is exactly representable: the all-zero group dequantizes to 0
    assert np.all(out["W_hat"][3, :16] == 0)
    assert out["scales"][0, 3] == np.float32(2.0 / maxq)
    assert out["zeros"][0, 5] == 0


def test_grid_closed_form_small():
    # w in one group: min -0.3, max 0.9, 2-bit: s = 1.2/3 = 0.4, z = rint(0.75) = 1
    w = np.array([[-0.3, 0.1, 0.5, 0.9]], dtype=np.float32)
    s, z = gptq.quant_grid(w, 2)
    assert s[0] == np.float32(np.float32(1.2) / np.float32(3))
    assert z[0] == 1
    q, wq = gptq.quantize(w[0], s[0], z[0], 2)
    # w/s = -0.75, 0.25, 1.25, 2.25 -> rint -1, 0, 1, 2 -> +z -> 0, 1, 2, 3
    assert q.tolist() == [0, 1, 2, 3]


def test_rint_ties_to_even():
    s = np.array([np.float32(1.0)])
    z = np.array([np.float32(2.0)])
    q, _ = gptq.quantize(np.array([0.5, 1.5, -0.5, -1.5], dtype=np.float32), s, z, 3)
    assert q.tolist() == [2, 4, 2, 0]


# ------------------------------------------------------------ sweep pins ----
def test_diagonal_hessian_reduces_to_rtn():
    W = _layer(48, 64)
    for H in (np.eye(64), np.diag(RNG.uniform(0.5, 3.0, 64))):
        U = gptq.inverse_cholesky_upper(H)
        out = gptq.sweep(W, U, 4, 32)
        ref = gptq.rtn(W, 4, 32)
        assert np.array_equal(out["codes"], ref["codes"])
        assert np.array_equal(out["W_hat"], ref["W_hat"])
        assert np.array_equal(out["scales"], ref["scales"])


def _obq_fixed_order(W, Hd, bits, group):
    """Brute force: after each column, the closed-form OBQ update computed from an
    explicit inverse of the Hessian restricted to the columns not yet quantized."""
    W = np.array(W, dtype=np.float64)
    R, C = W.shape
    codes = np.zeros((R, C), dtype=np.uint8)
    for j in range(C):
        if j % group == 0:
            s, z = gptq.quant_grid(W[:, j:j + group], bits)
        q, wq = gptq.quantize(W[:, j], s, z, bits)
        Hinv = np.linalg.inv(Hd[j:, j:])
        d = (W[:, j] - wq.astype(np.float64)) / Hinv[0, 0]
        W[:, j:] -= np.outer(d, Hinv[0, :])
        codes[:, j] = q
        assert np.allclose(W[:, j], wq, atol=1e-12)
    return codes


@pytest.mark.parametrize("bits,group,C", [(2, 4, 8), (3, 8, 8), (4, 2, 6), (2, 8, 8)])
def test_sweep_matches_bruteforce_obq(bits, group, C):
    rng = np.random.default_rng(77 + C + bits)
    H, _ = _spd(C, n=3 * C, outliers=1, rng=rng)
    Hd, _ = gptq.prepare_hessian(H, 0.01)
    W = _layer(200, C, rng=rng)
    out = gptq.sweep(W, gptq.inverse_cholesky_upper(Hd), bits, group)
    ref = _obq_fixed_order(W, Hd, bits, group)
    assert np.array_equal(out["codes"], ref)


def _min_loss_exhaustive(w, Hd, s, z, bits):
    maxq = 2 ** bits - 1
    grid = np.array(list(itertools.product(range(maxq + 1), repeat=len(w))), dtype=np.float32)
    deq = (s * (grid - z)).astype(np.float64)
    D = w[None, :] - deq
    return float(np.min(np.einsum("ij,jk,ik->i", D, Hd, D)))


def test_sweep_loss_not_below_exhaustive_optimum():
    rng = np.random.default_rng(9)
    C = 7
    H, _ = _spd(C, n=2 * C, rng=rng)
    Hd, _ = gptq.prepare_hessian(H, 0.01)
    W = _layer(12, C, rng=rng)
    out = gptq.sweep(W, gptq.inverse_cholesky_upper(Hd), 2, C)
    losses = gptq.row_losses(W, out["W_hat"], Hd)
    for r in range(12):
        best = _min_loss_exhaustive(W[r], Hd, out["scales"][0, r], np.float32(out["zeros"][0, r]), 2)
        assert losses[r] >= best * (1 - 1e-12)


def test_sweep_optimal_for_diagonal_hessian():
    rng = np.random.default_rng(10)
    C = 6
    Hd = np.diag(rng.uniform(0.5, 2.0, C))
    W = _layer(10, C, rng=rng)
    out = gptq.sweep(W, gptq.inverse_cholesky_upper(Hd), 2, C)
    losses = gptq.row_losses(W, out["W_hat"], Hd)
    for r in range(10):
        best = _min_loss_exhaustive(W[r], Hd, out["scales"][0, r], np.float32(out["zeros"][0, r]), 2)
        assert losses[r] == pytest.approx(best, rel=1e-12, abs=1e-18)


def test_error_identity():
    """sum_j e_j^2 = ΔW Hd ΔW^T per row (each OBS step raises the quadratic by e_j^2/2... times 2)."""
    H, _ = _spd(96, outliers=3)
    Hd, dead = gptq.prepare_hessian(H, 0.01)
    W = _layer(32, 96)
    out = gptq.sweep(W, gptq.inverse_cholesky_upper(Hd), 3, 32)
    ref = gptq.row_losses(W, out["W_hat"], Hd)
    assert np.allclose(out["row_err"], ref, rtol=1e-10, atol=0)


def _sweep_blocked(W, U, bits, group, block):
    """Lazy batch form: in-block updates only; the rest of W is updated once per block."""
    W = np.array(W, dtype=np.float64)
    R, C = W.shape
    codes = np.zeros((R, C), dtype=np.uint8)
    for b0 in range(0, C, block):
        b1 = min(C, b0 + block)
        E = np.zeros((R, b1 - b0))
        for j in range(b0, b1):
            if j % group == 0:
                s, z = gptq.quant_grid(W[:, j:j + group], bits)
            q, wq = gptq.quantize(W[:, j], s, z, bits)
            e = (W[:, j] - wq) / U[j, j]
            W[:, j + 1:b1] -= np.outer(e, U[j, j + 1:b1])
            E[:, j - b0] = e
            codes[:, j] = q
        W[:, b1:] -= E @ U[b0:b1, b1:]
    return codes


def test_blocked_equals_eager():
    H, _ = _spd(64, outliers=2)
    Hd, _ = gptq.prepare_hessian(H, 0.01)
    U = gptq.inverse_cholesky_upper(Hd)
    W = _layer(40, 64)
    out = gptq.sweep(W, U, 4, 16)
    assert np.array_equal(_sweep_blocked(W, U, 4, 16, 32), out["codes"])


def _sweep_factor_form(W, Hd, bits, group, block):
    """The same sweep driven by the Cholesky factor of H itself (Hd = Ũ Ũ^T, Ũ
    upper, from the lower factor of the index-reversed matrix) instead of the
    factor of the inverse.  Since U = Ũ^-1, the weights of block [s, s+B) as
    updated by every earlier column are W0 + (ΔW[:, :s] Ũ[:s, blk]) inv(Ũ[blk, blk]),
    with ΔW = W0 - Ŵ; inside the block the ordinary update runs with
    inv(Ũ[blk, blk]), which is the diagonal block of U."""
    C = Hd.shape[0]
    J = np.eye(C)[::-1]
    Ut = J @ np.linalg.cholesky(J @ Hd @ J) @ J
    W0 = np.array(W, dtype=np.float64)
    R = W0.shape[0]
    dW = np.zeros_like(W0)
    codes = np.zeros((R, C), dtype=np.uint8)
    for s0 in range(0, C, block):
        s1 = min(C, s0 + block)
        Ub = np.linalg.inv(Ut[s0:s1, s0:s1])
        Wb = W0[:, s0:s1] + (dW[:, :s0] @ Ut[:s0, s0:s1]) @ Ub
        for j in range(s0, s1):
            jj = j - s0
            if j % group == 0:
                s, z = gptq.quant_grid(Wb[:, jj:jj + group], bits)
            q, wq = gptq.quantize(Wb[:, jj], s, z, bits)
            e = (Wb[:, jj] - wq) / Ub[jj, jj]
            Wb[:, jj + 1:] -= np.outer(e, Ub[jj, jj + 1:])
            dW[:, j] = W0[:, j] - wq
            codes[:, j] = q
    return codes


def test_sweep_equals_factor_form():
    H, _ = _spd(48, outliers=2)
    Hd, _ = gptq.prepare_hessian(H, 0.01)
    W = _layer(64, 48)
    out = gptq.sweep(W, gptq.inverse_cholesky_upper(Hd), 2, 8)
    assert np.array_equal(_sweep_factor_form(W, Hd, 2, 8, 16), out["codes"])
    assert np.array_equal(_sweep_factor_form(W, Hd, 2, 8, 48), out["codes"])


def test_dead_column():
    rng = np.random.default_rng(3)
    X = rng.standard_normal((80, 16))
    X[:, 5] = 0.0
    H = gptq.hessian(X)
    W = _layer(20, 16, rng=rng)
    out = gptq.quantize_layer(W, H, 4, 8)
    assert out["dead"].tolist() == [i == 5 for i in range(16)]
    assert np.all(out["W_hat"][:, 5] == 0)
    # the dead input does not change the output error: the loss from H equals ||X ΔW^T||^2
    assert gptq.layer_loss(W, out["W_hat"], H) == pytest.approx(gptq.output_error(X, W, out["W_hat"]), rel=1e-12)


def test_loss_equals_output_error():
    H, X = _spd(32, n=100)
    W = _layer(8, 32)
    out = gptq.quantize_layer(W, H, 3, 16)
    assert gptq.layer_loss(W, out["W_hat"], H) == pytest.approx(gptq.output_error(X, W, out["W_hat"]), rel=1e-12)


def test_gptq_beats_rtn_on_correlated_inputs():
    """[GPTQ-wiki] "Rendimiento y Precisión": GPTQ lowers the error relative to round-to-nearest."""
    rng = np.random.default_rng(21)
    C = 128
    base = rng.standard_normal((1024, C))
    X = base @ (np.eye(C) + 0.3 * rng.standard_normal((C, C)) / np.sqrt(C))
    X[:, :3] *= 20
    H = gptq.hessian(X)
    W = _layer(64, C, rng=rng)
    g = gptq.quantize_layer(W, H, 3, 64)
    r = gptq.rtn(W, 3, 64)
    assert gptq.layer_loss(W, g["W_hat"], H) < 0.8 * gptq.layer_loss(W, r["W_hat"], H)


def test_rtn_uniform_noise_model():
    """[LowBit] section 6: the uniform-noise approximation, error variance s^2 / 12."""
    rng = np.random.default_rng(4)
    W = rng.uniform(-1, 1, size=(512, 1024))
    out = gptq.rtn(W, 4, 128)
    s = np.repeat(out["scales"].T, 128, axis=1).astype(np.float64)
    ratio = np.mean((W - out["W_hat"]) ** 2) / np.mean(s ** 2 / 12.0)
    assert 0.97 < ratio < 1.03


# ------------------------------------------------------- planted mistakes ---
def _sweep_mutant(W, U, bits, group, mutation):
    W = np.array(W, dtype=np.float64)
    R, C = W.shape
    W0 = W.copy()
    codes = np.zeros((R, C), dtype=np.uint8)
    for j in range(C):
        if j % group == 0:
            src = W0 if mutation == "grid_from_original" else W
            s, z = gptq.quant_grid(src[:, j:j + group], bits)
        q, wq = gptq.quantize(W[:, j], s, z, bits)
        e = (W[:, j] - wq) / U[j, j]
        if mutation == "sign":
            W[:, j + 1:] += np.outer(e, U[j, j + 1:])
        elif mutation == "transposed":
            W[:, j + 1:] -= np.outer(e, U.T[j, j + 1:])
        elif mutation == "no_diag_scale":
            W[:, j + 1:] -= np.outer(W[:, j] - wq, U[j, j + 1:])
        else:
            W[:, j + 1:] -= np.outer(e, U[j, j + 1:])
        codes[:, j] = q
    return codes


@pytest.mark.parametrize("mutation", ["sign", "transposed", "no_diag_scale", "grid_from_original"])
def test_planted_mistakes_are_caught_by_bruteforce_pin(mutation):
    rng = np.random.default_rng(99)
    C = 8
    H, _ = _spd(C, n=2 * C, outliers=1, rng=rng)
    Hd, _ = gptq.prepare_hessian(H, 0.01)
    W = _layer(400, C, rng=rng)
    U = gptq.inverse_cholesky_upper(Hd)
    ref = _obq_fixed_order(W, Hd, 2, 4)
    assert np.array_equal(_sweep_mutant(W, U, 2, 4, None), ref)
    assert not np.array_equal(_sweep_mutant(W, U, 2, 4, mutation), ref)


# ----------------------------------------------- precision of the integer decisions
def _grid_f64(wg, bits):
    maxq = float(2 ** bits - 1)
    w = np.asarray(wg, dtype=np.float64)
    xmin = np.minimum(w.min(axis=1), 0.0)
    xmax = np.maximum(w.max(axis=1), 0.0)
    flat = (xmin == 0) & (xmax == 0)
    xmin = np.where(flat, -1.0, xmin)
    xmax = np.where(flat, 1.0, xmax)
    s = (xmax - xmin) / maxq
    return s, np.rint(-xmin / s)


def _quantize_f64(w, s, z, bits):
    q = np.clip(np.rint(np.asarray(w, dtype=np.float64) / s) + z, 0.0, float(2 ** bits - 1))
    return q, s * (q - z)


@pytest.mark.parametrize("bits,group", [(4, 128), (3, 128), (2, 64)])
def test_float32_decisions_match_float64_decisions(bits, group, monkeypatch):
    """The oracle takes the grid, code and dequantized value in float32 (the precision the format
    stores).  The same sweep with every decision in float64 must give the same codes on >= 99.99 %
    of entries and the same layer loss within 1e-4, on a 256 x 1024 layer with outlier inputs:
    the float32 choice decides ties only, it does not move the result."""
    from synthetic import custom_layer
    from tests._helpers import host_arrays

    spec = custom_layer("f64dec", 256, 1024, 8192, bits=bits, group=group, n_outliers=10, key=(501, bits))
    _, w64 = host_arrays(spec.W)
    _, x64 = host_arrays(spec.X)
    H = gptq.hessian(x64)
    ref = gptq.quantize_layer(w64, H, bits, group)
    monkeypatch.setattr(gptq, "quant_grid", _grid_f64)
    monkeypatch.setattr(gptq, "quantize", _quantize_f64)
    alt = gptq.quantize_layer(w64, H, bits, group)
    monkeypatch.undo()
    assert np.mean(alt["codes"] == ref["codes"]) >= 0.9999
    l_ref = gptq.layer_loss(w64, ref["W_hat"], H)
    l_alt = gptq.layer_loss(w64, alt["W_hat"], H)
    assert abs(l_alt - l_ref) <= 1e-4 * l_ref
