"""gptq_quantize_layer_noalloc: the whole-layer call for callers that cannot
allocate device memory (a plugin whose host application owns every byte of
device memory, a service that must not grow its footprint after start-up, a
real-time loop where a synchronizing cudaMalloc is not allowed).  It runs in
the library's fixed 16 MiB scratch array instead of a caller workspace.

Called through the C ABI with ctypes and compared with gptq_quantize_layer on
the same inputs, on two calls in a row with different layers, so that what
the first call leaves in the shared scratch cannot leak into the second.
Tolerances are those of the other parity tests: codes identical on >= 99.9 %
of entries, packing bit-exact given the codes, scales within 1e-4 relative,
layer loss within 0.5 %.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest

from oracle import gptq as og
from oracle import pack as opk
from synthetic import custom_layer

from tests._helpers import host_arrays, to_device

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

BITS, GROUP, BLOCK, DAMP = 3, 128, 128, 0.01


@pytest.fixture(scope="module")
def gq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import post_weight_quantization_30_b300 as gq

    return gq


def _layer(rows, cols, n, key):
    spec = custom_layer("noalloc", rows, cols, n, bits=BITS, group=GROUP, block=BLOCK, n_outliers=3, key=key)
    wa, w64 = host_arrays(spec.W)
    xa, x64 = host_arrays(spec.X)
    return to_device(wa, "bf16"), to_device(xa, "bf16"), w64, og.hessian(x64)


def _outputs(rows, cols):
    dev = "cuda"
    return dict(
        qweight=torch.empty((cols * BITS // 32, rows), dtype=torch.int32, device=dev),
        scales=torch.empty((cols // GROUP, rows), dtype=torch.float32, device=dev),
        qzeros=torch.empty((cols // GROUP, rows * BITS // 32), dtype=torch.int32, device=dev),
        codes=torch.empty((rows, cols), dtype=torch.uint8, device=dev),
        W_hat=torch.empty((rows, cols), dtype=torch.float32, device=dev),
        row_err=torch.empty(rows, dtype=torch.float32, device=dev),
    )


def _call_noalloc(gq, W, H, o):
    rows, cols = W.shape
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    info = ctypes.c_int64(-1)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = gq.lib.gptq_quantize_layer_noalloc(p(W), 1, rows, cols, p(H), BITS, GROUP, BLOCK, DAMP, p(o["qweight"]),
                                            p(o["scales"]), p(o["qzeros"]), p(o["codes"]), p(o["W_hat"]),
                                            p(o["row_err"]), stream, ctypes.byref(info))
    torch.cuda.synchronize()
    return st


def _np(t):
    return t.detach().cpu().numpy()


def test_noalloc_matches_workspace_call_twice(gq):
    for rows, cols, n, key in [(256, 512, 2048, (31,)), (160, 384, 1536, (32,))]:
        W, X, w64, H0 = _layer(rows, cols, n, key)
        H = torch.zeros((cols, cols), dtype=torch.float32, device="cuda")
        gq.gptq_hessian_accumulate(H, X)
        ref = gq.gptq_quantize_layer(W, H, BITS, GROUP, BLOCK, DAMP)
        o = _outputs(rows, cols)
        assert _call_noalloc(gq, W, H, o) == 0
        codes, codes_ref = _np(o["codes"]), _np(ref["codes"])
        assert np.mean(codes == codes_ref) >= 0.999
        assert np.array_equal(_np(o["qweight"]), opk.pack_qweight(codes, BITS))
        assert np.allclose(_np(o["scales"]), _np(ref["scales"]), rtol=1e-4, atol=0)
        lg = og.layer_loss(w64, _np(o["W_hat"]), H0)
        lr = og.layer_loss(w64, _np(ref["W_hat"]), H0)
        assert abs(lg - lr) <= 5e-3 * lr, (lg, lr)


def test_noalloc_rejects_layers_beyond_the_scratch(gq):
    rows, cols = 4096, 4096  # needs ~200 MB of scratch
    assert gq.lib.gptq_quantize_layer_workspace_size(rows, cols, BLOCK) > (16 << 20)
    W = torch.zeros((rows, cols), dtype=torch.bfloat16, device="cuda")
    H = torch.eye(cols, device="cuda")
    o = _outputs(rows, cols)
    assert _call_noalloc(gq, W, H, o) == -7  # GQ_EWORKSPACE, before anything is enqueued
    with pytest.raises(ValueError):
        gq.gptq_quantize_layer_noalloc(W, H, BITS, GROUP, BLOCK, DAMP)
