"""Bid-Up (and the OLrC + Bid-Up cycle) on the GPU, through the C ABI, against the float64 oracle.

Inputs: a layer quantized by the GPTQ oracle (codes, scales, zeros packed as the
library packs them), H in float32, an optional rank-r correction from the
oracle's OLrC.  Checked: codes identical to the oracle's sweep on >= 99.9 % of
entries (the integer decision rint(g_j / (H_jj s)) is taken in float32 from
gradients the two sides accumulate differently, so near-ties may differ); the
objective never above the starting one and within 0.5 % of the oracle's; Ŵ and
qweight exact given the GPU's codes; the reported count of moved codes exact.
"""
import numpy as np
import pytest

from oracle import gptq as og
from oracle import pack as opk
from oracle import refine as rf
from synthetic import custom_layer

from tests._helpers import host_arrays, to_device

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


def _inputs(rows, cols, bits, group, key):
    spec = custom_layer("bu", rows, cols, 4 * cols, bits=bits, group=group, n_outliers=max(1, cols // 100), key=key)
    wa, w64 = host_arrays(spec.W)
    _, x64 = host_arrays(spec.X)
    H32 = og.hessian(x64).astype(np.float32)
    q = og.quantize_layer(w64, H32.astype(np.float64), bits, group, 0.01)
    return spec, wa, w64, H32, q


def _gpu_bidup(gq, spec, wa, H32, codes, q, bits, group, A=None, B=None):
    rows, cols = codes.shape
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    c = dev(codes)
    qw = torch.empty((cols * bits // 32, rows), dtype=torch.int32, device="cuda")
    out = gq.gptq_bidup(to_device(wa, spec.W.dtype), dev(H32), c, dev(q["scales"]),
                        dev(opk.pack_qzeros(q["zeros"], bits)), bits, group,
                        None if A is None else dev(A.astype(np.float32)),
                        None if B is None else dev(B.astype(np.float32)), qweight=qw)
    gq.gq_check_device()
    return _np(out["codes"]), _np(out["W_hat"]), _np(out["qweight"]), int(_np(out["changed"])[0])


CASES = [
    # rows, cols, bits, group, r
    (64, 256, 2, 64, 0),
    (96, 320, 3, 64, 8),      # ragged last block (64 columns)
    (128, 384, 4, 128, 16),
    (64, 1152, 2, 64, 4),     # nine blocks: recursive deferred updates
]


@pytest.mark.parametrize("rows,cols,bits,group,r", CASES)
def test_bidup_sweep_matches_the_oracle(gq, rows, cols, bits, group, r):
    spec, wa, w64, H32, q = _inputs(rows, cols, bits, group, (61, rows, cols))
    H64 = H32.astype(np.float64)
    A = B = None
    if r:
        A, B, _ = rf.olrc(w64, q["W_hat"], H64, r)
        A, B = A.astype(np.float32).astype(np.float64), B.astype(np.float32).astype(np.float64)
    ref = rf.bidup_sweep(w64, q["codes"], q["scales"], q["zeros"], H64, bits, group, A, B)
    codes, W_hat, qweight, changed = _gpu_bidup(gq, spec, wa, H32, q["codes"], q, bits, group, A, B)
    match = np.mean(codes == ref["codes"])
    print(f"moved: oracle {ref['changed']}, gpu {changed}; code identity {match:.6f}")
    assert match >= 0.999
    assert changed == int(np.sum(codes != q["codes"]))
    assert np.array_equal(W_hat, rf.dequant(codes, q["scales"], q["zeros"], group))
    assert np.array_equal(qweight, opk.pack_qweight(codes, bits))
    f0 = rf.objective(w64, q["W_hat"], H64, A, B)
    fg = rf.objective(w64, W_hat, H64, A, B)
    fo = rf.objective(w64, ref["W_hat"], H64, A, B)
    assert fg <= f0 * (1 + 1e-9)
    assert abs(fg - fo) <= 5e-3 * fo, (fg, fo)


def test_olrc_bidup_cycles(gq):
    """Two cycles of OLrC (eora_compensate on W - Ŵ) and Bid-Up on the GPU: the objective never increases
    and ends within 0.5 % of the oracle's cycle."""
    rows, cols, bits, group, r = 128, 256, 2, 64, 8
    spec, wa, w64, H32, q = _inputs(rows, cols, bits, group, (62,))
    H64 = H32.astype(np.float64)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    W = to_device(wa, spec.W.dtype)
    Hd = dev(H32)
    codes = dev(q["codes"])
    sc, qz = dev(q["scales"]), dev(opk.pack_qzeros(q["zeros"], bits))
    W_hat = dev(q["W_hat"])
    hist = [rf.objective(w64, q["W_hat"], H64)]
    for _ in range(2):
        dW = gq.gptq_weight_error(W, W_hat)
        ad = gq.eora_compensate(dW, Hd, r)
        A, B = ad["A"], ad["B"]
        hist.append(rf.objective(w64, _np(W_hat), H64, _np(A), _np(B)))
        out = gq.gptq_bidup(W, Hd, codes, sc, qz, bits, group, A, B, W_hat=W_hat)
        gq.gq_check_device()
        hist.append(rf.objective(w64, _np(out["W_hat"]), H64, _np(A), _np(B)))
    print("objective:", ["%.6g" % h for h in hist])
    assert all(b <= a * (1 + 1e-5) for a, b in zip(hist, hist[1:])), hist
    ref = rf.refine(w64, q["codes"], q["scales"], q["zeros"], H64, bits, group, r, cycles=2)
    assert abs(hist[-1] - ref["objective"][-1]) <= 5e-3 * ref["objective"][-1], (hist, ref["objective"])
