"""Failure detection on the GPU, in the forms that leave the device usable.

* Non-finite inputs: an Inf or NaN in a calibration token, in W or in EoRA's dW
  is reported as GQ_ENONFINITE by the first call that factors H (the one
  synchronization of the path), with info = 0 for H and 1 for W / dW.  The
  values are planted on the host.
* Bounded waits: gq_set_wait_budget shrinks the budget of every pipeline wait
  of the tensor-core kernels to a few hundred cycles, so ordinary waits for
  TMA copies and MMAs run out.  The Hessian kernel must then end by itself,
  gq_check_device must report GQ_ETIMEOUT, and after the budget is restored the
  same call must give the right H again (the context is still usable).
"""
import numpy as np
import pytest

from oracle import gptq as og
from synthetic import custom_layer

from tests._helpers import host_arrays, rel_fro, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

GQ_ENONFINITE, GQ_ETIMEOUT = -5, -6


@pytest.fixture(scope="module")
def gq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import post_weight_quantization_30_b300 as gq

    return gq


def _layer(rows=128, cols=256, n=2048, key=(61,)):
    spec = custom_layer("fail", rows, cols, n, bits=4, group=128, n_outliers=2, key=key)
    wa, w64 = host_arrays(spec.W)
    xa, x64 = host_arrays(spec.X)
    return wa, w64, xa, x64


def _bf16_with(a, index, value):
    """bf16 bit patterns with one element replaced by `value` (float)."""
    b = a.copy()
    b.reshape(-1)[index] = np.array([value], dtype=np.float32).view(np.uint32)[0] >> 16
    return b


@pytest.mark.parametrize("bad", [np.nan, np.inf, -np.inf])
def test_nonfinite_token_reported_by_the_factoring_call(gq, bad):
    wa, _, xa, _ = _layer()
    cols = xa.shape[1]
    X = to_device(_bf16_with(xa, 1000 * cols + 17, bad), "bf16")
    W = to_device(wa, "bf16")
    H = torch.zeros((cols, cols), dtype=torch.float32, device="cuda")
    gq.gptq_hessian_accumulate(H, X)
    with pytest.raises(gq.GQError) as ei:
        gq.gptq_quantize_layer(W, H, 4, 128)
    assert ei.value.status == GQ_ENONFINITE and ei.value.info == 0
    with pytest.raises(gq.GQError) as ei:
        gq.gptq_factor(H)
    assert ei.value.status == GQ_ENONFINITE and ei.value.info == 0


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_nonfinite_weight_reported(gq, dtype):
    wa, w64, xa, _ = _layer()
    cols = xa.shape[1]
    H = torch.zeros((cols, cols), dtype=torch.float32, device="cuda")
    gq.gptq_hessian_accumulate(H, to_device(xa, "bf16"))
    for idx in (0, 77, w64.size - 1):  # first, middle and last element (the check's aligned part and its ends)
        if dtype == "bf16":
            W = to_device(_bf16_with(wa, idx, np.nan), "bf16")
        else:
            w = w64.astype(np.float32).copy()
            w.reshape(-1)[idx] = np.inf
            W = to_device(w, "f32")
        with pytest.raises(gq.GQError) as ei:
            gq.gptq_quantize_layer(W, H, 4, 128)
        assert ei.value.status == GQ_ENONFINITE and ei.value.info == 1, idx
    # the same layer with finite weights goes through
    gq.gptq_quantize_layer(to_device(wa, "bf16"), H, 4, 128)
    gq.gq_check_device()


def test_nonfinite_weight_error_in_eora(gq):
    _, w64, xa, x64 = _layer(rows=128, cols=128, n=1024, key=(62,))
    cols = 128
    H = to_device(og.hessian(x64).astype(np.float32), "f32")
    dW = np.random.default_rng(0).standard_normal((128, cols)).astype(np.float32) * 1e-3
    dW[5, 9] = np.nan
    with pytest.raises(gq.GQError) as ei:
        gq.eora_compensate(to_device(dW, "f32"), H, 8)
    assert ei.value.status == GQ_ENONFINITE and ei.value.info == 1
    Hn = og.hessian(x64).astype(np.float32)
    Hn[3, 100] = np.inf  # upper triangle: read by the factor
    with pytest.raises(gq.GQError) as ei:
        gq.eora_compensate(to_device(np.nan_to_num(dW), "f32"), to_device(Hn, "f32"), 8)
    assert ei.value.status == GQ_ENONFINITE and ei.value.info == 0


def test_wait_budget_runs_out_and_the_context_stays_usable(gq):
    _, _, xa, x64 = _layer(cols=512, n=4096, key=(63,))
    cols = 512
    X = to_device(xa, "bf16")
    H = torch.zeros((cols, cols), dtype=torch.float32, device="cuda")
    gq.gq_check_device()  # start from a clean record
    assert gq.lib.gq_set_wait_budget(200) == 0
    try:
        gq.gptq_hessian_accumulate(H, X)
        with pytest.raises(gq.GQError) as ei:
            gq.gq_check_device()
        assert ei.value.status == GQ_ETIMEOUT
    finally:
        assert gq.lib.gq_set_wait_budget(0) == 0  # back to the default budget
    gq.gq_check_device()  # the record was cleared by the failed check
    H.zero_()
    gq.gptq_hessian_accumulate(H, X)
    gq.gq_check_device()
    assert rel_fro(H.cpu().numpy(), og.hessian(x64)) <= 1e-5
