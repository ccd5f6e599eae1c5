"""Pins of the GPTQ-intrinsic LoRA oracle (CPU only).

Each pin comes from outside the oracle's own formulas:

* the augmented Hessian equals 2 X~^T X~ computed from X~ = [X, X L] itself;
* the basis L equals the leading right singular vectors of X from numpy's SVD
  of X (a different routine from the eigendecomposition of H the oracle uses);
* the sweep's codes and final free columns equal a brute-force
  Optimal-Brain-Quantization that re-inverts the remaining augmented Hessian
  after every column;
* the final free columns are the closed-form least-squares optimum given Q;
* the OBS error identity: sum_j e_j^2 = d~ H~_d d~^T per row;
* r = 0 reduces to plain GPTQ exactly, and a full basis (L = I) absorbs the
  whole quantization error up to the damping.
"""
import numpy as np
import pytest

from oracle import gptq as og
from oracle import intrinsic_lora as il


def _calib(n, cols, rng, outliers=0, scale=20.0):
    X = rng.standard_normal((n, cols))
    if outliers:
        X[:, rng.choice(cols, outliers, replace=False)] *= scale
    return X


def _orthonormal(cols, r, rng):
    Q, _ = np.linalg.qr(rng.standard_normal((cols, r)))
    return Q


def test_augmented_hessian_is_gram_of_augmented_inputs():
    rng = np.random.default_rng(1)
    X = _calib(300, 48, rng, outliers=2)
    L = _orthonormal(48, 5, rng)
    Ht = il.augmented_hessian(og.hessian(X), L)
    ref = og.hessian(np.hstack([X, X @ L]))
    assert np.allclose(Ht, ref, rtol=1e-12, atol=1e-9 * np.abs(ref).max())


def test_basis_is_leading_right_singular_subspace_of_x():
    rng = np.random.default_rng(2)
    cols, r = 40, 6
    U, _ = np.linalg.qr(rng.standard_normal((500, cols)))
    V, _ = np.linalg.qr(rng.standard_normal((cols, cols)))
    sv = np.concatenate([np.linspace(50, 20, r), np.linspace(3, 0.5, cols - r)])
    X = (U * sv) @ V.T
    L, lam = il.top_right_singular_vectors(og.hessian(X), r)
    _, sig, Vt = np.linalg.svd(X, full_matrices=False)
    assert np.allclose(lam, 2 * sig[:r] ** 2, rtol=1e-10)
    P = L @ L.T
    Pref = Vt[:r].T @ Vt[:r]
    assert np.linalg.norm(P - Pref) <= 1e-9
    assert np.allclose(L.T @ L, np.eye(r), atol=1e-12)
    for i in range(r):  # sign rule: largest-magnitude entry positive
        assert L[np.argmax(np.abs(L[:, i])), i] > 0


def _obq_with_free_columns(Wt, Hd, bits, group, n_quant):
    """Brute force on the augmented problem: after each quantized column, the closed-form OBQ update of
    every remaining column (quantized later or free), from an explicit inverse of the remaining Hessian."""
    W = np.array(Wt, dtype=np.float64)
    R, C = W.shape
    codes = np.zeros((R, n_quant), dtype=np.uint8)
    for j in range(n_quant):
        if j % group == 0:
            s, z = og.quant_grid(W[:, j:j + group], bits)
        q, wq = og.quantize(W[:, j], s, z, bits)
        Hinv = np.linalg.inv(Hd[j:, j:])
        d = (W[:, j] - wq.astype(np.float64)) / Hinv[0, 0]
        W[:, j:] -= np.outer(d, Hinv[0, :])
        codes[:, j] = q
    return codes, W[:, n_quant:]


@pytest.mark.parametrize("bits,group,cols,r", [(2, 4, 8, 1), (3, 8, 8, 2), (4, 2, 6, 3), (2, 4, 12, 4)])
def test_sweep_matches_bruteforce_obq_with_free_columns(bits, group, cols, r):
    rng = np.random.default_rng(10 + cols + r + bits)
    X = _calib(3 * cols, cols, rng, outliers=1)
    H = og.hessian(X)
    L, _ = il.top_right_singular_vectors(H, r)
    W = rng.standard_normal((150, cols)) * 0.02
    out = il.intrinsic_lora(W, H, L, bits, group, 0.01)
    codes, free = _obq_with_free_columns(np.hstack([W, np.zeros((150, r))]), out["Hd"], bits, group, cols)
    assert np.array_equal(out["codes"], codes)
    assert np.allclose(out["B"], free, rtol=1e-9, atol=1e-12)


@pytest.mark.parametrize("bits,group,r", [(2, 16, 4), (3, 32, 8), (4, 32, 16)])
def test_free_columns_are_the_optimum_given_q(bits, group, r):
    rng = np.random.default_rng(20 + r)
    cols = 64
    H = og.hessian(_calib(256, cols, rng, outliers=2))
    L, _ = il.top_right_singular_vectors(H, r)
    W = rng.standard_normal((48, cols)) * 0.02
    out = il.intrinsic_lora(W, H, L, bits, group, 0.01)
    ref = il.free_columns_optimum(W, out["W_hat"], out["Hd"])
    assert np.linalg.norm(out["B"] - ref) <= 1e-9 * np.linalg.norm(ref)


def test_error_identity_on_the_augmented_problem():
    rng = np.random.default_rng(3)
    cols, r = 96, 8
    H = og.hessian(_calib(400, cols, rng, outliers=3))
    L, _ = il.top_right_singular_vectors(H, r)
    W = rng.standard_normal((32, cols)) * 0.02
    out = il.intrinsic_lora(W, H, L, 3, 32, 0.01)
    d = np.hstack([W - out["W_hat"].astype(np.float64), -out["B"]])
    quad = np.einsum("ij,jk,ik->i", d, out["Hd"], d)
    assert np.allclose(out["row_err"], quad, rtol=1e-10, atol=0)


def test_rank_zero_is_plain_gptq():
    rng = np.random.default_rng(4)
    cols = 64
    H = og.hessian(_calib(256, cols, rng, outliers=2))
    W = rng.standard_normal((40, cols)) * 0.02
    out = il.intrinsic_lora(W, H, np.zeros((cols, 0)), 2, 32, 0.01)
    ref = og.quantize_layer(W, H, 2, 32, 0.01)
    for k in ("codes", "scales", "zeros", "W_hat"):
        assert np.array_equal(out[k], ref[k]), k
    assert out["B"].shape == (40, 0)


def test_full_basis_absorbs_the_error():
    """L = I (r = cols): the free columns reproduce W - Q up to the damping, so the layer loss of
    Q + B A is a tiny fraction of plain GPTQ's."""
    rng = np.random.default_rng(5)
    cols = 32
    H = og.hessian(_calib(4000, cols, rng))
    W = rng.standard_normal((24, cols)) * 0.02
    out = il.intrinsic_lora(W, H, np.eye(cols), 2, 16, 1e-4)
    BA = out["B"] @ out["A"]
    l_adapter = og.layer_loss(W, out["W_hat"].astype(np.float64) + BA, H)
    l_gptq = og.layer_loss(W, og.quantize_layer(W, H, 2, 16, 1e-4)["W_hat"], H)
    assert l_adapter <= 1e-5 * l_gptq


def test_adapter_lowers_the_loss_with_outlier_inputs():
    """Expected from the method (not a theorem): with a few dominant input directions absorbed by the
    adapter, Q + B A has a lower layer loss than plain GPTQ at the same bits."""
    rng = np.random.default_rng(6)
    cols, r = 128, 8
    H = og.hessian(_calib(1024, cols, rng, outliers=4, scale=30.0))
    L, _ = il.top_right_singular_vectors(H, r)
    W = rng.standard_normal((64, cols)) * 0.02
    out = il.intrinsic_lora(W, H, L, 2, 32, 0.01)
    l_adapter = og.layer_loss(W, out["W_hat"].astype(np.float64) + out["B"] @ out["A"], H)
    l_gptq = og.layer_loss(W, og.quantize_layer(W, H, 2, 32, 0.01)["W_hat"], H)
    assert l_adapter < l_gptq


def _sweep_partial_mutant(W, U, bits, group, n_quant, mutation):
    W = np.array(W, dtype=np.float64, copy=True)
    for j in range(n_quant):
        if j % group == 0:
            s, z = og.quant_grid(W[:, j:j + group], bits)
        _, wq = og.quantize(W[:, j], s, z, bits)
        e = (W[:, j] - wq.astype(np.float64)) / U[j, j]
        stop = n_quant if mutation == "free_not_updated" else W.shape[1]
        sign = -1.0 if mutation == "free_sign" else 1.0
        W[:, j + 1:n_quant] -= np.outer(e, U[j, j + 1:n_quant])
        W[:, n_quant:stop] -= sign * np.outer(e, U[j, n_quant:stop])
    return W[:, n_quant:]


@pytest.mark.parametrize("mutation", ["free_not_updated", "free_sign"])
def test_planted_mistakes_are_caught_by_the_optimality_pin(mutation):
    rng = np.random.default_rng(7)
    cols, r = 32, 4
    H = og.hessian(_calib(200, cols, rng, outliers=1))
    L, _ = il.top_right_singular_vectors(H, r)
    W = rng.standard_normal((16, cols)) * 0.02
    out = il.intrinsic_lora(W, H, L, 2, 16, 0.01)
    U = og.inverse_cholesky_upper(out["Hd"])
    bad = _sweep_partial_mutant(np.hstack([W, np.zeros((16, r))]), U, 2, 16, cols, mutation)
    ref = il.free_columns_optimum(W, out["W_hat"], out["Hd"])
    assert np.linalg.norm(bad - ref) > 1e-3 * np.linalg.norm(ref)
    assert np.linalg.norm(out["B"] - ref) <= 1e-9 * np.linalg.norm(ref)


# ---------------------------------------------- eigendecomposition + QR factorization
def test_eigqr_factor_is_the_upper_factor_of_the_inverse():
    """U^T U Hd = I, U upper triangular with a positive diagonal: the unique upper factor of Hd^-1,
    so it equals GPTQ's inverse + Cholesky route where that one is accurate."""
    rng = np.random.default_rng(30)
    cols, r = 48, 4
    H = og.hessian(_calib(300, cols, rng, outliers=2))
    L, _ = il.top_right_singular_vectors(H, r)
    Hd, _ = og.prepare_hessian(il.augmented_hessian(H, L), 0.01)
    U = il.inverse_cholesky_upper_eigqr(Hd)
    assert np.allclose(np.tril(U, -1), 0.0, atol=0)
    assert np.all(np.diagonal(U) > 0)
    assert np.linalg.norm(U.T @ U @ Hd - np.eye(cols + r)) <= 1e-9
    assert np.allclose(U, og.inverse_cholesky_upper(Hd), rtol=1e-8, atol=1e-12 * np.abs(U).max())


def test_eigqr_is_accurate_at_small_damping():
    """At damping 1e-10 the augmented Hessian has condition number ~1e12: the eigendecomposition + QR
    factor still satisfies U^T U Hd = I to ~1e-4 (rounding grows like sqrt(cond)), where the inverse +
    Cholesky route is far worse or fails."""
    rng = np.random.default_rng(31)
    cols, r = 64, 6
    H = og.hessian(_calib(400, cols, rng, outliers=3))
    L, _ = il.top_right_singular_vectors(H, r)
    Hd, _ = og.prepare_hessian(il.augmented_hessian(H, L), 1e-10)
    cond = np.linalg.cond(Hd)
    assert cond > 1e11
    U = il.inverse_cholesky_upper_eigqr(Hd)
    res_qr = np.linalg.norm(U.T @ U @ Hd - np.eye(cols + r))
    assert res_qr <= 1e-3
    try:
        Uc = og.inverse_cholesky_upper(Hd)
        res_chol = np.linalg.norm(Uc.T @ Uc @ Hd - np.eye(cols + r))
    except np.linalg.LinAlgError:
        res_chol = np.inf
    assert res_qr < res_chol


@pytest.mark.parametrize("damp", [1e-2, 1e-4, 1e-6])
def test_eigqr_sweep_matches_bruteforce_obq_at_small_damping(damp):
    """The sweep through the eigendecomposition + QR factor gives the codes and free columns of the
    brute-force OBQ that re-inverts the remaining augmented Hessian after every column."""
    rng = np.random.default_rng(40)
    cols, r, bits, group = 8, 2, 3, 4
    H = og.hessian(_calib(3 * cols, cols, rng, outliers=1))
    L, _ = il.top_right_singular_vectors(H, r)
    W = rng.standard_normal((120, cols)) * 0.02
    out = il.intrinsic_lora(W, H, L, bits, group, damp, factor="eigqr")
    codes, free = _obq_with_free_columns(np.hstack([W, np.zeros((120, r))]), out["Hd"], bits, group, cols)
    assert np.array_equal(out["codes"], codes)
    assert np.allclose(out["B"], free, rtol=1e-6, atol=1e-9)


def test_zero_damping_is_rejected():
    rng = np.random.default_rng(41)
    H = og.hessian(_calib(100, 16, rng))
    L, _ = il.top_right_singular_vectors(H, 2)
    with pytest.raises(ValueError):
        il.intrinsic_lora(rng.standard_normal((8, 16)), H, L, 2, 8, 0.0, factor="eigqr")
