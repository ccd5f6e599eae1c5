"""Low-precision adapter factors on the GPU against the oracle.

gptq_quantize_rtn is the GPTQ grid without error propagation, so it is compared
bit for bit with the oracle's round-to-nearest (oracle.gptq.rtn): codes, scales,
zeros and the dequantized factor.  Then the page's use of it: an EoRA adapter of
a 2-bit GPTQ layer with A at 4 bits and B at 8 bits ("Resumen Técnico:
GPTQ-intrinsic LoRA", "Resultados Clave"): B at 8 bits is lossless here (the
objective within 0.5 %), and the quantized adapter keeps most of its gain.
"""
import numpy as np
import pytest

from oracle import eora as oe
from oracle import gptq as og
from oracle import refine as rf

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import post_weight_quantization_30_b300 as gq

    return gq


def _gpu_rtn(gq, M, bits, group):
    o = gq.gptq_quantize_rtn(torch.from_numpy(np.ascontiguousarray(M, dtype=np.float32)).cuda(), bits, group)
    return {k: v.cpu().numpy() for k, v in o.items()}


@pytest.mark.parametrize("nrows,ncols,bits,group", [(64, 1024, 4, 128), (1024, 64, 8, 64), (33, 96, 3, 32),
                                                    (8, 256, 2, 256)])
def test_rtn_is_bit_exact(gq, nrows, ncols, bits, group):
    rng = np.random.default_rng(nrows + ncols + bits)
    M = (rng.standard_normal((nrows, ncols)) * rng.uniform(0.01, 1.0, (nrows, 1))).astype(np.float32)
    M[3 % nrows] = 0.0                       # an all-zero row: grid [-1, 1]
    M[5 % nrows, : ncols // 2] = np.abs(M[5 % nrows, : ncols // 2])  # one-signed groups
    g = _gpu_rtn(gq, M, bits, group)
    ref = og.rtn(M.astype(np.float64), bits, group)
    assert np.array_equal(g["codes"], ref["codes"])
    assert np.array_equal(g["scales"], ref["scales"])
    assert np.array_equal(g["zeros"], ref["zeros"])
    assert np.array_equal(g["M_hat"], ref["W_hat"])


def test_quantized_eora_factors(gq):
    rng = np.random.default_rng(0)
    rows, cols, r = 256, 512, 32
    X = rng.standard_normal((2048, cols))
    X[:, rng.choice(cols, 5, replace=False)] *= 20.0
    W = rng.standard_normal((rows, cols)) * 0.02
    H = og.hessian(X)
    q = og.quantize_layer(W, H, 2, 64, 0.01)
    A, B, _ = oe.eora(W - q["W_hat"], H, r)
    Aq = _gpu_rtn(gq, A, 4, 128)["M_hat"].astype(np.float64)
    Bq = _gpu_rtn(gq, B, 8, r)["M_hat"].astype(np.float64)
    f0 = rf.objective(W, q["W_hat"], H)
    f1 = rf.objective(W, q["W_hat"], H, A, B)
    f_b8 = rf.objective(W, q["W_hat"], H, A, Bq)
    f_a4b8 = rf.objective(W, q["W_hat"], H, Aq, Bq)
    print(f"objective: none {f0:.4g}, float32 factors {f1:.4g}, B 8-bit {f_b8 / f1 - 1:+.3%}, "
          f"A 4-bit + B 8-bit {f_a4b8 / f1 - 1:+.3%}")
    assert abs(f_b8 - f1) <= 5e-3 * f1
    assert f_a4b8 < 0.25 * f0
