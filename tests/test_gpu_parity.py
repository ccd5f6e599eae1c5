"""Parity of the CUDA path (through the C ABI) against the float64 oracle, on seeded
inputs at sizes the oracle finishes in seconds, spanning several tiles and ragged
tails.  Tolerances (from the method's acceptance criteria):

* H: relative Frobenius error <= 1e-5;
* codes: identical on >= 99.9 % of entries (a float32 near-tie can flip one);
* layer loss ||X W^T - X Ŵ^T||_F^2 within 0.5 % relative;
* packing: bit-exact given the GPU's own codes and zero points.
"""
import numpy as np
import pytest

from oracle import gptq as og
from oracle import pack as opk
from synthetic import LAYERS, custom_layer

from tests._helpers import host_arrays, rel_fro, reversed_upper_factor, to_device

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


# ------------------------------------------------------------------ packing ---
@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("rows,cols", [(37, 64), (256, 384), (1, 32)])
def test_pack_unpack_bit_exact(gq, bits, rows, cols):
    rng = np.random.default_rng(bits * 1000 + rows)
    codes = rng.integers(0, 2 ** bits, size=(rows, cols)).astype(np.uint8)
    qw = gq.gptq_pack(torch.from_numpy(codes).cuda(), bits)
    assert np.array_equal(_np(qw), opk.pack_qweight(codes, bits))
    back = gq.gptq_unpack(qw, rows, cols, bits)
    assert np.array_equal(_np(back), codes)


# ------------------------------------------------------------------ hessian ---
@pytest.mark.parametrize("n,cols,dtype", [(1000, 96, "bf16"), (4099, 384, "bf16"), (2048, 256, "f32"),
                                          (777, 200, "f32"), (8192, 1024, "bf16"), (65536, 512, "bf16")])
def test_hessian_parity(gq, n, cols, dtype):
    spec = custom_layer("h", 32, cols, n, dtype=dtype, n_outliers=max(1, cols // 100), key=(11, n, cols)).X
    a, x64 = host_arrays(spec)
    H = torch.zeros((cols, cols), dtype=torch.float32, device="cuda")
    X = to_device(a, dtype)
    gq.gptq_hessian_accumulate(H, X[: n // 2])
    gq.gptq_hessian_accumulate(H, X[n // 2:])
    ref = og.hessian(x64)
    Hg = _np(H)
    assert rel_fro(Hg, ref) <= 1e-5
    assert np.array_equal(Hg, Hg.T)


def test_hessian_exact_on_small_integers(gq):
    rng = np.random.default_rng(3)
    x = rng.integers(-8, 9, size=(3000, 160)).astype(np.float32)
    H = torch.zeros((160, 160), dtype=torch.float32, device="cuda")
    gq.gptq_hessian_accumulate(H, torch.from_numpy(x).cuda().to(torch.bfloat16))
    assert np.array_equal(_np(H), og.hessian(x.astype(np.float64)))


def test_hessian_strided_input(gq):
    rng = np.random.default_rng(4)
    big = rng.standard_normal((512, 320)).astype(np.float32)
    Xs = torch.from_numpy(big).cuda().to(torch.bfloat16)[:, :256]  # ldx = 320
    H = torch.zeros((256, 256), dtype=torch.float32, device="cuda")
    gq.gptq_hessian_accumulate(H, Xs)
    ref = og.hessian(Xs.float().cpu().numpy().astype(np.float64))
    assert rel_fro(_np(H), ref) <= 1e-5


# ------------------------------------------------------------------- factor ---
@pytest.mark.parametrize("cols", [256, 200, 1000, 1056, 1280])  # >= 1024: recursive order, 1056: ragged panel
def test_factor_parity(gq, cols):
    spec = custom_layer("f", 32, cols, 4 * cols, dtype="f32", n_outliers=2, key=(12, cols)).X
    _, x64 = host_arrays(spec)
    H32 = og.hessian(x64).astype(np.float32)
    F, dead = gq.gptq_factor(torch.from_numpy(H32).cuda(), 0.01)
    Hd, dead_ref = og.prepare_hessian(H32.astype(np.float64), 0.01)
    ref = reversed_upper_factor(Hd)
    Fg = _np(F)
    assert np.all(np.tril(Fg, -1) == 0)
    assert rel_fro(Fg, ref) <= 2e-5
    assert np.array_equal(_np(dead).astype(bool), dead_ref)


def test_factor_not_positive_definite(gq):
    H = torch.eye(64, device="cuda") * -1.0
    H[10, 10] = 5.0
    with pytest.raises(gq.GQError) as ei:
        gq.gptq_factor(H, 0.0)
    assert ei.value.status == -2
    assert 0 <= ei.value.info < 64


# -------------------------------------------------------------------- sweep ---
SWEEP_CASES = [
    # rows, cols, bits, group, block, n
    (64, 256, 4, 128, 128, 2048),
    (96, 384, 3, 128, 128, 3000),
    (128, 320, 2, 64, 128, 2000),   # ragged last block (64 columns)
    (32, 128, 4, 32, 64, 1024),
    (160, 640, 2, 64, 64, 4096),
    (64, 1152, 4, 128, 128, 4096),  # 9 blocks: recursive factor order, block inverses from the factor
]


def _layer_inputs(rows, cols, n, bits, group, block, key):
    spec = custom_layer("s", rows, cols, n, bits=bits, group=group, block=block, n_outliers=max(1, cols // 100),
                        key=key)
    wa, w64 = host_arrays(spec.W)
    xa, x64 = host_arrays(spec.X)
    return spec, wa, w64, xa, x64


def _check_against_oracle(gq, out, ref, w64, H0, bits, group, rows, cols):
    codes = _np(out["codes"])
    match = np.mean(codes == ref["codes"])
    assert match >= 0.999, f"code identity {match:.6f}"
    # packing bit-exact given the GPU's own codes; zeros bit-exact given the GPU's zeros
    assert np.array_equal(_np(out["qweight"]), opk.pack_qweight(codes, bits))
    zeros_gpu = opk.unpack_qzeros(_np(out["qzeros"]), bits, rows)
    assert zeros_gpu.shape == ref["zeros"].shape
    assert np.mean(zeros_gpu == ref["zeros"]) >= 0.999
    assert np.allclose(_np(out["scales"]), ref["scales"], rtol=1e-4, atol=0)
    # Ŵ is s (q - z) of the GPU's own grid, bit for bit
    s = np.repeat(_np(out["scales"]).T, group, axis=1)
    z = np.repeat(zeros_gpu.T.astype(np.float32), group, axis=1)
    deq = (s * (codes.astype(np.float32) - z)).astype(np.float32)
    assert np.array_equal(deq, _np(out["W_hat"]))
    lg = og.layer_loss(w64, _np(out["W_hat"]), H0)
    lo = og.layer_loss(w64, ref["W_hat"], H0)
    assert abs(lg - lo) <= 5e-3 * lo, (lg, lo)


@pytest.mark.parametrize("rows,cols,bits,group,block,n", SWEEP_CASES)
def test_sweep_with_oracle_factor(gq, rows, cols, bits, group, block, n):
    """The sweep alone, fed the oracle's factor: isolates sweep error from H and Cholesky."""
    spec, wa, w64, xa, x64 = _layer_inputs(rows, cols, n, bits, group, block, (13, rows, cols))
    H0 = og.hessian(x64)
    ref = og.quantize_layer(w64, H0, bits, group, 0.01)
    F = torch.from_numpy(reversed_upper_factor(ref["Hd"]).astype(np.float32)).cuda()
    W = to_device(wa, spec.W.dtype)
    out = gq.gptq_sweep(W, F, None, bits, group, block)
    _check_against_oracle(gq, out, ref, w64, H0, bits, group, rows, cols)
    # error identity: sum_j e_j^2 = ΔW Hd ΔW^T per row
    rl = og.row_losses(w64, _np(out["W_hat"]), ref["Hd"])
    assert np.allclose(_np(out["row_err"]), rl, rtol=1e-3)


@pytest.mark.parametrize("rows,cols,bits,group,block,n", SWEEP_CASES)
def test_quantize_layer_end_to_end(gq, rows, cols, bits, group, block, n):
    spec, wa, w64, xa, x64 = _layer_inputs(rows, cols, n, bits, group, block, (14, rows, cols))
    H = torch.zeros((cols, cols), dtype=torch.float32, device="cuda")
    gq.gptq_hessian_accumulate(H, to_device(xa, spec.X.dtype))
    H0 = og.hessian(x64)
    assert rel_fro(_np(H), H0) <= 1e-5
    ref = og.quantize_layer(w64, H0, bits, group, 0.01)
    out = gq.gptq_quantize_layer(to_device(wa, spec.W.dtype), H, bits, group, block, 0.01)
    _check_against_oracle(gq, out, ref, w64, H0, bits, group, rows, cols)


def test_tiny_workload(gq):
    """The 256 x 256 float32 layer with 2048 float32 tokens, 4 outlier channels x20."""
    spec = LAYERS["tiny_256x256"]
    wa, w64 = host_arrays(spec.W)
    xa, x64 = host_arrays(spec.X)
    H = torch.zeros((256, 256), dtype=torch.float32, device="cuda")
    gq.gptq_hessian_accumulate(H, to_device(xa, "f32"))
    H0 = og.hessian(x64)
    assert rel_fro(_np(H), H0) <= 1e-5
    ref = og.quantize_layer(w64, H0, spec.bits, spec.group, spec.damp)
    out = gq.gptq_quantize_layer(to_device(wa, "f32"), H, spec.bits, spec.group, spec.block, spec.damp)
    _check_against_oracle(gq, out, ref, w64, H0, spec.bits, spec.group, 256, 256)
    # the loss from H equals the output error on the activations
    lg = og.layer_loss(w64, _np(out["W_hat"]), H0)
    assert lg == pytest.approx(og.output_error(x64, w64, _np(out["W_hat"])), rel=1e-9)


def test_dead_inputs(gq):
    rows, cols = 64, 256
    spec, wa, w64, xa, x64 = _layer_inputs(rows, cols, 1024, 4, 128, 128, (15,))
    x = x64.copy()
    x[:, [3, 130, 255]] = 0.0
    xa2 = xa.copy()
    xa2[:, [3, 130, 255]] = 0
    H = torch.zeros((cols, cols), dtype=torch.float32, device="cuda")
    gq.gptq_hessian_accumulate(H, to_device(xa2, spec.X.dtype))
    H0 = og.hessian(x)
    ref = og.quantize_layer(w64, H0, 4, 128, 0.01)
    out = gq.gptq_quantize_layer(to_device(wa, spec.W.dtype), H, 4, 128, 128, 0.01)
    assert np.all(_np(out["W_hat"])[:, [3, 130, 255]] == 0)
    _check_against_oracle(gq, out, ref, w64, H0, 4, 128, rows, cols)


def test_rejects_bad_arguments_without_launch(gq):
    W = torch.zeros((64, 256), dtype=torch.bfloat16, device="cuda")
    H = torch.eye(256, device="cuda")
    with pytest.raises(gq.GQError) as ei:
        gq.gptq_quantize_layer(W, H, 5, 128)
    assert ei.value.status == -3
    with pytest.raises(gq.GQError) as ei:
        gq.gptq_quantize_layer(W, H, 4, 128, block=64)
    assert ei.value.status == -1


# ---------------------------------------------------------- code decisions ---
def test_code_decisions_match_ieee_division(gq):
    """The sweep rounds w / s without dividing (RN(1/s) plus one FMA correction).
    Its decisions must equal rint of the IEEE float32 quotient everywhere, in
    particular for w within a few ulps of (k + 1/2) s, where a plain product
    w * RN(1/s) can round to the other integer."""
    rng = np.random.default_rng(21)
    s = (rng.uniform(1.0, 2.0, 200000) * 2.0 ** rng.integers(-20, 4, 200000)).astype(np.float32)
    k = rng.integers(-8, 16, 200000).astype(np.float32)
    w = ((k + np.float32(0.5)) * s).astype(np.float32)
    offs = rng.integers(-3, 4, 200000).astype(np.int32)
    w = (w.view(np.int32) + offs).view(np.float32)
    w = np.concatenate([w, (rng.standard_normal(200000) * 8).astype(np.float32) * s])
    s = np.concatenate([s, s])
    got = _np(gq.gptq_code_decisions(torch.from_numpy(w).cuda(), torch.from_numpy(s).cuda()))
    ref = np.rint(w / s)  # numpy float32 division is IEEE round-to-nearest
    assert np.array_equal(got, ref)
    dev = _np(torch.round(torch.from_numpy(w).cuda() / torch.from_numpy(s).cuda()))  # CUDA's own division
    assert np.array_equal(got, dev)


# --------------------------------------------------------- degenerate cases ---
def test_zero_rows_and_zero_groups(gq):
    """An all-zero row (every group falls back to the [-1, 1] grid, z = rint(maxq / 2)
    rounded half to even) and rows whose first group is zero."""
    rows, cols, bits, group = 64, 256, 4, 128
    spec, wa, w64, xa, x64 = _layer_inputs(rows, cols, 2048, bits, group, 128, (16,))
    w32 = w64.astype(np.float32)
    w32[5, :] = 0.0
    w32[17, :group] = 0.0
    w32[40, :] = 0.0
    H = torch.zeros((cols, cols), dtype=torch.float32, device="cuda")
    gq.gptq_hessian_accumulate(H, to_device(xa, spec.X.dtype))
    H0 = og.hessian(x64)
    ref = og.quantize_layer(w32.astype(np.float64), H0, bits, group, 0.01)
    out = gq.gptq_quantize_layer(torch.from_numpy(w32).cuda(), H, bits, group, 128, 0.01)
    codes = _np(out["codes"])
    assert np.array_equal(codes[[5, 40]], ref["codes"][[5, 40]])
    # grid [-1, 1]: s = RN(2 / 15) lies just above 2/15, so -xmin / s = 7.4999995 and z = 7
    z = np.rint(np.float32(1.0) / (np.float32(2.0) / np.float32(15.0)))
    assert z == 7 and np.all(codes[5] == z) and np.all(_np(out["W_hat"])[5] == 0)
    _check_against_oracle(gq, out, ref, w32.astype(np.float64), H0, bits, group, rows, cols)


@pytest.mark.parametrize("bits,group", [(2, 64), (3, 128), (4, 32)])
def test_diagonal_hessian_is_round_to_nearest(gq, bits, group):
    """With a diagonal H no error propagates: GPTQ is group-wise round-to-nearest, exactly."""
    rows, cols = 96, 384
    rng = np.random.default_rng(bits)
    w = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    d = rng.uniform(0.5, 2.0, cols).astype(np.float32)
    H = torch.from_numpy(np.diag(d)).cuda()
    out = gq.gptq_quantize_layer(torch.from_numpy(w).cuda(), H, bits, group, 128, 0.01)
    ref = og.rtn(w.astype(np.float64), bits, group)
    assert np.array_equal(_np(out["codes"]), ref["codes"])
    assert np.array_equal(_np(out["W_hat"]), ref["W_hat"])
    assert np.array_equal(opk.unpack_qzeros(_np(out["qzeros"]), bits, rows), ref["zeros"])


def test_single_block_layer(gq):
    rows, cols, bits, group, block = 32, 64, 2, 32, 64
    spec, wa, w64, xa, x64 = _layer_inputs(rows, cols, 512, bits, group, block, (17,))
    H = torch.zeros((cols, cols), dtype=torch.float32, device="cuda")
    gq.gptq_hessian_accumulate(H, to_device(xa, spec.X.dtype))
    H0 = og.hessian(x64)
    ref = og.quantize_layer(w64, H0, bits, group, 0.01)
    out = gq.gptq_quantize_layer(to_device(wa, spec.W.dtype), H, bits, group, block, 0.01)
    _check_against_oracle(gq, out, ref, w64, H0, bits, group, rows, cols)
