"""Parity at the full sizes of every quantization workload, in the launch
configuration bench.py times (the whole X in one gptq_hessian_accumulate call,
one gptq_quantize_layer call with block 128), against the float64 oracle.

The oracle computes its own H from the same bf16 bytes (float64, chunked) and
its own U = chol(H_d^-1)^T.  GPTQ rows are independent given U, so the oracle
sweeps a sample of rows one by one.  Checked, for each layer:

* H: relative Frobenius error <= 1e-5 over the whole matrix;
* codes of the sampled rows identical on >= 99.9 % of entries;
* packing: the qweight words of the sampled rows bit-exact given the GPU's codes;
* layer loss of the sampled rows (1/2 sum_r ΔW_r H ΔW_r^T, undamped H) within 0.5 %.

Layers that share a calibration set (q_proj / up_proj, the two Qwen2.5-72B
shapes, the two Qwen3-32B shapes) share the oracle's H: the tests run in that
order and the last H is kept.

EoRA at full size (the 5120 x 5120 and 25600 x 5120 layers at the workloads'
rank r = 64, and the 5120 x 5120 layer at r = 256, the rank of the EoRA
page's own adapter call): both sides take the error of
round-to-nearest on the layer's own 2-bit g64 grid (the library's
gptq_quantize_rtn and the oracle's rtn agree bit for bit), so no input of the
oracle comes from the GPU; the GPU uses its own H, the oracle its float64 H.
Compared as in the small EoRA tests: the 64 singular values (1e-3 relative
where the spectrum has a gap at that index, the interlacing bound inside a
cluster of nearly equal values, see tests/_helpers.check_sigma) and the compensated loss
(never below the oracle's optimum, within 1e-3 of it).
"""
import numpy as np
import pytest

from oracle import eora as oe
from oracle import gptq as og
from oracle import pack as opk
from synthetic import LAYERS, bf16_bits_to_f32, generate
from tests._helpers import check_sigma

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

SAMPLE_ROWS = 64
ORDER = ["llama7b_q_proj_4096x4096", "llama7b_up_proj_11008x4096", "llama7b_down_proj_4096x11008",
         "qwen72b_8192x8192", "qwen72b_29568x8192", "qwen32b_5120x5120", "qwen32b_25600x5120"]

# The last calibration set's host bytes and oracle H (float64), keyed by its spec.
_CACHE = {}


@pytest.fixture(scope="module")
def gq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import post_weight_quantization_30_b300 as gq

    return gq


def _calibration(xspec):
    """(bf16 bytes of X, oracle H = 2 X^T X in float64) for one calibration set, cached."""
    if _CACHE.get("spec") != xspec:
        _CACHE.clear()
        xa = generate(xspec)
        H0 = np.zeros((xspec.cols, xspec.cols), dtype=np.float64)
        for r0 in range(0, xspec.rows, 8192):
            og.hessian(bf16_bits_to_f32(xa[r0:r0 + 8192]).astype(np.float64), H0)
        _CACHE.update(spec=xspec, xa=xa, H0=H0)
    return _CACHE["xa"], _CACHE["H0"]


def _gpu_hessian(gq, xa, cols):
    dev = torch.device("cuda")
    X = torch.from_numpy(xa.view(np.int16)).to(dev).view(torch.bfloat16)
    H = torch.zeros((cols, cols), dtype=torch.float32, device=dev)
    gq.gptq_hessian_accumulate(H, X)
    del X
    return H


@pytest.mark.parametrize("name", ORDER)
def test_full_size_layer(gq, name):
    spec = LAYERS[name]
    R, C = spec.rows, spec.cols
    xa, H0 = _calibration(spec.X)
    wa = generate(spec.W)
    dev = torch.device("cuda")
    H = _gpu_hessian(gq, xa, C)
    W = torch.from_numpy(wa.view(np.int16)).to(dev).view(torch.bfloat16)
    out = gq.gptq_quantize_layer(W, H, spec.bits, spec.group, spec.block, spec.damp, codes=True, W_hat=True,
                                 row_err=False)
    gq.gq_check_device()
    Hg = H.cpu().numpy().astype(np.float64)
    codes = out["codes"].cpu().numpy()
    qweight = out["qweight"].cpu().numpy()
    W_hat = out["W_hat"].cpu().numpy()
    del H, W, out
    torch.cuda.empty_cache()

    rel = np.linalg.norm(Hg - H0) / np.linalg.norm(H0)
    print(f"{name}: H relative Frobenius error {rel:.3e}")
    assert rel <= 1e-5, rel
    del Hg

    # Oracle factor and sweep of sampled rows.
    Hd, dead = og.prepare_hessian(H0, spec.damp)
    U = og.inverse_cholesky_upper(Hd)
    del Hd
    rng = np.random.default_rng(1234)
    rows = np.sort(rng.choice(R, SAMPLE_ROWS, replace=False))
    w64 = bf16_bits_to_f32(wa[rows]).astype(np.float64)
    ref = og.sweep(w64, U, spec.bits, spec.group, dead=dead)
    match = np.mean(codes[rows] == ref["codes"])
    print(f"{name}: codes identical on {match * 100:.4f} % of the sampled rows' entries")
    assert match >= 0.999, match
    assert np.array_equal(qweight[:, rows], opk.pack_qweight(codes[rows], spec.bits))
    lg = og.layer_loss(w64, W_hat[rows], H0)
    lo = og.layer_loss(w64, ref["W_hat"], H0)
    print(f"{name}: sampled-row layer loss {lg:.6e} vs oracle {lo:.6e}")
    assert abs(lg - lo) <= 5e-3 * lo, (lg, lo)


@pytest.mark.parametrize("name,r", [("qwen32b_5120x5120", 64), ("qwen32b_25600x5120", 64), ("qwen32b_5120x5120", 256)])
def test_full_size_eora(gq, name, r):
    spec = LAYERS[name]
    R, C = spec.rows, spec.cols
    xa, H0 = _calibration(spec.X)
    wa = generate(spec.W)
    dev = torch.device("cuda")
    H = _gpu_hessian(gq, xa, C)
    Wf = torch.from_numpy(bf16_bits_to_f32(wa)).to(dev)
    q = gq.gptq_quantize_rtn(Wf, spec.bits, spec.group)
    dW = gq.gptq_weight_error(Wf, q["M_hat"])
    g = gq.eora_compensate(dW, H, r)
    gq.gq_check_device()
    M_hat_gpu = q["M_hat"].cpu().numpy()
    g = {k: v.cpu().numpy().astype(np.float64) for k, v in g.items()}
    del H, Wf, q, dW
    torch.cuda.empty_cache()

    w64 = bf16_bits_to_f32(wa).astype(np.float64)
    ref = og.rtn(w64, spec.bits, spec.group)
    # The error both sides compensate is the same: round-to-nearest decisions agree bit for bit.
    assert np.array_equal(M_hat_gpu.view(np.uint32), ref["W_hat"].view(np.uint32))
    dW0 = w64 - ref["W_hat"].astype(np.float64)
    A_o, B_o, sig = oe.eora(dW0, H0, r)
    print(f"EoRA r={r}: sigma_1 {sig[0]:.6e} (GPU {g['sigma'][0]:.6e}), sigma_r {sig[r - 1]:.6e} "
          f"(GPU {g['sigma'][r - 1]:.6e}), sigma_r/sigma_r+1 = {sig[r - 1] / sig[r]:.6f}")
    check_sigma(g["sigma"], sig, r)
    base = oe.compensated_loss(dW0, 0 * A_o, 0 * B_o, H0)
    lg = oe.compensated_loss(dW0, g["A"], g["B"], H0)
    lo = oe.compensated_loss(dW0, A_o, B_o, H0)
    print(f"EoRA r={r}: compensated loss {lg:.6e} vs oracle optimum {lo:.6e} (uncompensated {base:.6e})")
    assert lg >= lo * (1 - 1e-9) - 1e-12 * base
    assert lg <= lo * (1 + 1e-3) + 1e-9 * base, (lg, lo)
