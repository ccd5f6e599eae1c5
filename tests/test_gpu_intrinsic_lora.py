"""GPTQ-intrinsic LoRA on the GPU (through the C ABI) against the float64 oracle.

The oracle runs the page's augmented sweep literally: H~ = [[H, H L], [L^T H,
L^T H L]] damped over its cols + r diagonal, GPTQ over [W, 0] with the last r
columns never quantized.  The library reaches the same result by block
elimination (GPTQ on the Schur complement, then R in closed form), so the two
share nothing but the inputs.  Both sides get the same float32 H and the same
float32 basis L^T (the oracle's leading eigenvectors, rounded), because the
leading subspace is not unique where eigenvalues cluster; the GPU's own basis is
checked separately on what is unique.

Checked, as for GPTQ: codes identical on >= 99.9 % of entries, packing and Ŵ
bit-exact given the GPU's codes and grid, scales within a bar derived from the
float32 Schur complement (see _check), and the layer loss of Q + R L^T within 0.5 % of the oracle's; plus R within 1e-3
relative Frobenius on rows whose codes all match, and the sum of the sweep's
e_j^2 within 1e-3.
"""
import numpy as np
import pytest

from oracle import gptq as og
from oracle import intrinsic_lora as il
from oracle import pack as opk
from synthetic import custom_layer

from tests._helpers import host_arrays, rel_fro, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import post_weight_quantization_30_b300 as gq

    return gq


def _np(t):
    return t.detach().cpu().numpy()


def _adapter_loss(w64, W_hat, R, Lt64, H64):
    return og.layer_loss(w64, np.asarray(W_hat, np.float64) + np.asarray(R, np.float64) @ Lt64, H64)


def _inputs(rows, cols, n, r, bits, group, key, dtype="bf16", n_outliers=None):
    spec = custom_layer("il", rows, cols, n, bits=bits, group=group, dtype=dtype,
                        n_outliers=max(1, cols // 100) if n_outliers is None else n_outliers, key=key)
    wa, w64 = host_arrays(spec.W)
    _, x64 = host_arrays(spec.X)
    H32 = og.hessian(x64).astype(np.float32)
    L, _ = il.top_right_singular_vectors(H32.astype(np.float64), r)
    Lt32 = np.ascontiguousarray(L.T, dtype=np.float32)
    return spec, wa, w64, H32, Lt32


def _check(gq, out, ref, w64, H64, Lt64, bits, group, rows):
    codes = _np(out["codes"])
    match = np.mean(codes == ref["codes"])
    assert match >= 0.999, f"code identity {match:.6f}"
    assert np.array_equal(_np(out["qweight"]), opk.pack_qweight(codes, bits))
    zeros_gpu = opk.unpack_qzeros(_np(out["qzeros"]), bits, rows)
    assert np.mean(zeros_gpu == ref["zeros"]) >= 0.999
    # Scales follow the updated weights.  The library forms S = H_d - Y Y^T in float32, and rounding at
    # the scale of H_d leaves S a relative error of about kappa * eps32, kappa = ||H_d|| / ||S|| (the
    # cancellation of the absorbed directions); the weights inherit it.  A float64 emulation of that
    # rounding moved the scales by up to 6.6 kappa eps32, so the bar is 64 kappa eps32 (1e-4 at least),
    # on the rows whose codes all match (a flipped code moves its row's later scales) and on >= 99.9 %
    # of all groups.
    Hd = ref["Hd"]
    cols = codes.shape[1]
    S = Hd[:cols, :cols] - Hd[:cols, cols:] @ np.linalg.solve(Hd[cols:, cols:], Hd[cols:, :cols])
    kappa = np.linalg.norm(Hd[:cols, :cols], 2) / np.linalg.norm(S, 2)
    stol = max(1e-4, 64 * kappa * 2.0 ** -24)
    same = np.all(codes == ref["codes"], axis=1)
    assert same.mean() >= 0.5, f"rows with identical codes {same.mean():.3f}, code identity {match:.6f}"
    sc, sr = _np(out["scales"]), ref["scales"]
    serr = np.abs(sc - sr) / np.abs(sr)
    print(f"kappa {kappa:.1f}, scale error max {serr[:, same].max():.2e} (bar {stol:.2e})")
    assert np.all(serr[:, same] <= stol)
    assert np.mean(serr <= stol) >= 0.999
    s = np.repeat(_np(out["scales"]).T, group, axis=1)
    z = np.repeat(zeros_gpu.T.astype(np.float32), group, axis=1)
    assert np.array_equal((s * (codes.astype(np.float32) - z)).astype(np.float32), _np(out["W_hat"]))
    R = _np(out["R"]).astype(np.float64)
    assert rel_fro(R[same], ref["B"][same]) <= 1e-3
    lg = _adapter_loss(w64, _np(out["W_hat"]), R, Lt64, H64)
    lo = _adapter_loss(w64, ref["W_hat"], ref["B"], Lt64, H64)
    print(f"code identity {match:.6f}, rows identical {same.mean():.3f}, loss gpu / oracle {lg / lo:.6f}")
    assert abs(lg - lo) <= 5e-3 * lo, (lg, lo)
    if out.get("row_err") is not None:
        assert np.sum(_np(out["row_err"])) == pytest.approx(np.sum(ref["row_err"]), rel=1e-3)
    return lg, lo


CASES = [
    # rows, cols, n, r, bits, group, dtype
    (64, 256, 2048, 16, 4, 128, "f32"),
    (128, 384, 3000, 64, 2, 64, "bf16"),
    (96, 320, 2000, 6, 3, 64, "bf16"),      # r not a multiple of 4; ragged last block (64 columns)
    (64, 1152, 4096, 32, 2, 64, "bf16"),    # 9 blocks: recursive factor, block inverses from the factor
    (256, 128, 1024, 1, 4, 32, "bf16"),     # rank one
]


@pytest.mark.parametrize("rows,cols,n,r,bits,group,dtype", CASES)
def test_matches_the_augmented_sweep(gq, rows, cols, n, r, bits, group, dtype):
    spec, wa, w64, H32, Lt32 = _inputs(rows, cols, n, r, bits, group, (41, rows, cols, r), dtype)
    H64, Lt64 = H32.astype(np.float64), Lt32.astype(np.float64)
    ref = il.intrinsic_lora(w64, H64, Lt64.T, bits, group, 0.01)
    out = gq.gptq_intrinsic_lora(to_device(wa, spec.W.dtype), torch.from_numpy(H32).cuda(),
                                 torch.from_numpy(Lt32).cuda(), bits, group, 128, 0.01)
    gq.gq_check_device()
    _check(gq, out, ref, w64, H64, Lt64, bits, group, rows)


@pytest.mark.parametrize("rows,cols,n,r,bits,group", [(128, 384, 3000, 64, 2, 64), (64, 1152, 4096, 32, 2, 64)])
def test_small_damping_against_the_eigqr_factorization(gq, rows, cols, n, r, bits, group):
    """Damping 1e-3 (ten times smaller than GPTQ's usual 0.01) against the oracle's eigendecomposition +
    QR factorization of the augmented Hessian (the page's robust route), at the GPTQ bars: codes identical
    on >= 99.9 % of entries, packing bit-exact given the GPU's codes, Ŵ on the GPU's own grid, and the
    layer loss of Q + R L^T within 0.5 %.  The library keeps its float32 Schur-complement route, whose
    rounding grows as the damping shrinks (at 1e-4 the loss still agrees within 0.3 % but codes agree on
    94-99.6 % only), so 1e-3 is the smallest damping checked.  Scales and R are not compared element by
    element here: the rounding of the small directions of the Schur complement (about 2 damp mean(diag))
    moves them beyond the bar derived for damping 0.01, while codes and loss stay within theirs."""
    spec, wa, w64, H32, Lt32 = _inputs(rows, cols, n, r, bits, group, (41, rows, cols, r))
    H64, Lt64 = H32.astype(np.float64), Lt32.astype(np.float64)
    ref = il.intrinsic_lora(w64, H64, Lt64.T, bits, group, 1e-3, factor="eigqr")
    out = gq.gptq_intrinsic_lora(to_device(wa, spec.W.dtype), torch.from_numpy(H32).cuda(),
                                 torch.from_numpy(Lt32).cuda(), bits, group, 128, 1e-3)
    gq.gq_check_device()
    codes = _np(out["codes"])
    match = np.mean(codes == ref["codes"])
    assert match >= 0.999, match
    assert np.array_equal(_np(out["qweight"]), opk.pack_qweight(codes, bits))
    zeros_gpu = opk.unpack_qzeros(_np(out["qzeros"]), bits, rows)
    s = np.repeat(_np(out["scales"]).T, group, axis=1)
    z = np.repeat(zeros_gpu.T.astype(np.float32), group, axis=1)
    assert np.array_equal((s * (codes.astype(np.float32) - z)).astype(np.float32), _np(out["W_hat"]))
    lg = _adapter_loss(w64, _np(out["W_hat"]), _np(out["R"]), Lt64, H64)
    lo = _adapter_loss(w64, ref["W_hat"], ref["B"], Lt64, H64)
    print(f"damping 1e-3: code identity {match:.6f}, loss gpu / oracle {lg / lo:.6f}")
    assert abs(lg - lo) <= 5e-3 * lo, (lg, lo)


def test_adapter_beats_plain_gptq_with_outliers(gq):
    """Expected from the method: absorbing the dominant input directions lowers the layer loss."""
    rows, cols, n, r, bits, group = 128, 512, 4096, 16, 2, 64
    spec, wa, w64, H32, Lt32 = _inputs(rows, cols, n, r, bits, group, (42,), n_outliers=8)
    H = torch.from_numpy(H32).cuda()
    W = to_device(wa, spec.W.dtype)
    out = gq.gptq_intrinsic_lora(W, H, torch.from_numpy(Lt32).cuda(), bits, group, 128, 0.01)
    plain = gq.gptq_quantize_layer(W, H, bits, group, 128, 0.01)
    H64 = H32.astype(np.float64)
    la = _adapter_loss(w64, _np(out["W_hat"]), _np(out["R"]), Lt32.astype(np.float64), H64)
    lp = og.layer_loss(w64, _np(plain["W_hat"]), H64)
    assert la < lp


def test_dead_inputs(gq):
    rows, cols, n, r = 64, 256, 2048, 8
    spec, wa, w64, H32, _ = _inputs(rows, cols, n, r, 4, 64, (43,))
    for i in (3, 130, 255):
        H32[i, :] = 0.0
        H32[:, i] = 0.0
    L, _ = il.top_right_singular_vectors(H32.astype(np.float64), r)
    Lt32 = np.ascontiguousarray(L.T, dtype=np.float32)
    H64, Lt64 = H32.astype(np.float64), Lt32.astype(np.float64)
    ref = il.intrinsic_lora(w64, H64, Lt64.T, 4, 64, 0.01)
    out = gq.gptq_intrinsic_lora(to_device(wa, spec.W.dtype), torch.from_numpy(H32).cuda(),
                                 torch.from_numpy(Lt32).cuda(), 4, 64, 128, 0.01)
    assert np.all(_np(out["W_hat"])[:, [3, 130, 255]] == 0)
    _check(gq, out, ref, w64, H64, Lt64, 4, 64, rows)


def test_not_positive_definite_reports_the_augmented_column(gq):
    cols, r = 64, 4
    H = -torch.eye(cols, dtype=torch.float32, device="cuda")
    Lt = torch.eye(cols, dtype=torch.float32, device="cuda")[:r].contiguous()
    W = torch.zeros((32, cols), dtype=torch.float32, device="cuda")
    with pytest.raises(gq.GQError) as ei:
        gq.gptq_intrinsic_lora(W, H, Lt, 4, 32, 64, 0.01)
    assert ei.value.status == -2
    assert ei.value.info == cols  # row 0 of L^T H L + delta I


# --------------------------------------------------------------------- basis ---
def _check_basis(gq, H32, r, lam_rtol):
    H64 = H32.astype(np.float64)
    o = gq.gptq_lora_basis(torch.from_numpy(H32).cuda(), r)
    Lt = _np(o["Lt"]).astype(np.float64)
    lam = _np(o["lam"]).astype(np.float64)
    L_ref, lam_ref = il.top_right_singular_vectors(H64, r)
    assert np.allclose(Lt @ Lt.T, np.eye(r), atol=1e-5)
    for i in range(r):
        assert Lt[i, np.argmax(np.abs(Lt[i]))] > 0
    # Ritz values: never above the exact eigenvalues (interlacing) beyond float32 rounding at the scale
    # of the largest one, and close to them
    tol = 1e-6 * lam_ref[0]
    assert np.all(lam <= lam_ref * (1 + 1e-5) + tol)
    assert np.all(lam >= lam_ref * (1 - lam_rtol) - tol)
    # the Ritz values are the Rayleigh quotients of the returned vectors
    assert np.allclose(np.einsum("ij,jk,ik->i", Lt, H64, Lt), lam, rtol=1e-4, atol=tol)
    return Lt, lam, L_ref, lam_ref


def test_basis_with_a_planted_gap(gq):
    cols, r = 256, 12
    rng = np.random.default_rng(44)
    V, _ = np.linalg.qr(rng.standard_normal((cols, cols)))
    ev = np.concatenate([np.linspace(100, 50, r), np.linspace(5, 0.1, cols - r)])
    H32 = ((V * ev) @ V.T).astype(np.float32)
    Lt, lam, L_ref, lam_ref = _check_basis(gq, H32, r, 1e-5)
    assert np.linalg.norm(Lt.T @ Lt - L_ref @ L_ref.T) <= 1e-4
    assert np.linalg.norm(Lt - L_ref.T) <= 1e-4 * np.sqrt(r)  # unique up to sign, and signs fixed


@pytest.mark.parametrize("cols,r,n_outliers", [(512, 16, 5), (1024, 64, 10), (320, 8, 0)])
def test_basis_of_calibration_inputs(gq, cols, r, n_outliers):
    """Outlier channels give a few well-separated directions (unique) above a flat bulk (not unique)."""
    spec = custom_layer("b", 32, cols, 8 * cols, n_outliers=n_outliers, key=(45, cols))
    _, x64 = host_arrays(spec.X)
    H32 = og.hessian(x64).astype(np.float32)
    Lt, lam, L_ref, lam_ref = _check_basis(gq, H32, r, 2e-2)
    # captured energy within 5e-3 of the optimum (30 iterations leave the flat bulk's Ritz values
    # a few 1e-3 low; a float64 run of the same iteration on these inputs gives 1.05e-3 at most)
    assert lam.sum() >= (1 - 5e-3) * lam_ref.sum()
    if n_outliers:
        Vo = L_ref[:, :n_outliers]
        assert np.linalg.norm(Vo - Lt.T @ (Lt @ Vo)) <= 1e-3 * np.sqrt(n_outliers)


def test_basis_then_intrinsic_lora(gq):
    """The whole GPU path (basis from H, then the quantization) against the oracle with its own basis:
    the loss of Q + R L^T within 0.5 %."""
    rows, cols, n, r, bits, group = 128, 512, 4096, 16, 2, 64
    spec, wa, w64, H32, Lt32_ref = _inputs(rows, cols, n, r, bits, group, (46,), n_outliers=5)
    H = torch.from_numpy(H32).cuda()
    b = gq.gptq_lora_basis(H, r)
    out = gq.gptq_intrinsic_lora(to_device(wa, spec.W.dtype), H, b["Lt"], bits, group, 128, 0.01)
    H64 = H32.astype(np.float64)
    ref = il.intrinsic_lora(w64, H64, Lt32_ref.astype(np.float64).T, bits, group, 0.01)
    lg = _adapter_loss(w64, _np(out["W_hat"]), _np(out["R"]), _np(b["Lt"]).astype(np.float64), H64)
    lo = _adapter_loss(w64, ref["W_hat"], ref["B"], Lt32_ref.astype(np.float64), H64)
    assert abs(lg - lo) <= 5e-3 * lo, (lg, lo)
