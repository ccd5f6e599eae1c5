"""gptq_quantize_layer_noalloc: the whole-layer call for callers that cannot
allocate device memory (a plugin whose host application owns every byte of
device memory, a service that must not grow its footprint after start-up, a
real-time loop where a synchronizing cudaMalloc is not allowed).  It runs in
the library's fixed 16 MiB scratch array instead of a caller workspace.

Called through the C ABI with ctypes and compared with gptq_quantize_layer on
the same inputs, on calls in a row with different layers (and the first layer
again at the end), so that what one call leaves in the shared scratch cannot
leak into the next.  Both calls run the same kernels in the same order on the
same inputs, so every output must be identical bit for bit: codes, qweight,
qzeros, scales, W_hat and the row errors.  The layer loss against the float64
oracle's is checked as well, as a sanity check (within 0.5 %).

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
    layers = [(256, 512, 2048, (31,)), (160, 384, 1536, (32,)), (256, 512, 2048, (31,))]
    first = None
    for rows, cols, n, key in layers:
        W, X, w64, H0 = _layer(rows, cols, n, key)
        H = torch.zeros((cols, cols), dtype=torch.float32, device="cuda")
        gq.gptq_hessian_accumulate(H, X)
        ref = gq.gptq_quantize_layer(W, H, BITS, GROUP, BLOCK, DAMP)
        o = _outputs(rows, cols)
        for t in o.values():
            t.fill_(7)  # no output may keep what was there before the call
        assert _call_noalloc(gq, W, H, o) == 0
        for k in ("codes", "qweight", "qzeros", "scales", "W_hat", "row_err"):
            a, b = _np(o[k]), _np(ref[k])
            assert a.dtype == b.dtype and np.array_equal(a.view(np.uint8), b.view(np.uint8)), k
        assert np.array_equal(_np(o["qweight"]), opk.pack_qweight(_np(o["codes"]), BITS))
        lg = og.layer_loss(w64, _np(o["W_hat"]), H0)
        lo = og.layer_loss(w64, og.quantize_layer(w64, H0, BITS, GROUP, DAMP)["W_hat"], H0)
        assert abs(lg - lo) <= 5e-3 * lo, (lg, lo)
        if first is None:
            first = {k: _np(v) for k, v in o.items()}
        elif (rows, cols, key) == layers[0][:2] + (layers[0][3],):
            # the first layer again, after a different layer used the scratch in between
            for k, v in first.items():
                assert np.array_equal(_np(o[k]).view(np.uint8), v.view(np.uint8)), k


def test_noalloc_rejects_layers_beyond_the_scratch(gq):
    rows, cols = 4096, 4096  # needs ~200 MB of scratch
    assert gq.lib.gptq_quantize_layer_workspace_size(rows, cols, BLOCK) > (16 << 20)
    W = torch.zeros((rows, cols), dtype=torch.bfloat16, device="cuda")
    H = torch.eye(cols, device="cuda")
    o = _outputs(rows, cols)
    assert _call_noalloc(gq, W, H, o) == -7  # GQ_EWORKSPACE, before anything is enqueued
    with pytest.raises(ValueError):
        gq.gptq_quantize_layer_noalloc(W, H, BITS, GROUP, BLOCK, DAMP)
