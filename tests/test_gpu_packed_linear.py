"""The packed quantized linear layer on the GPU (through the C ABI) against the float64 oracle.

Y = X Ŵ^T + (X A^T) B^T with Ŵ = s (q - z) taken from the packed words.  The
kernel forms exact bf16 x integer products, sums one group's K range on the
tensor cores and scales it in float32, so Y differs from the exact value only by
float32 summation.  The bar is the classic bound for a sum of products,
|fl(sum) - sum| <= gamma * sum |x_k w_k|, for the order used: at most
group / 16 + 2 cols / group + r + 2 float32 additions on the path of a product
of X Ŵ^T on the tensor cores (partial sums of 16 products taken as rounded once
per step; group + 2 cols / group + r + 2 on the decode path, n <= 32, which sums
a group's products one by one and adds its K slices at the end),
and cols + r + 2 on the path of the adapter term (T = X A^T is summed over cols
in float32), with gamma = steps * 2^-23 (round-to-nearest or truncation),
applied to |X| |Ŵ|^T and |X| |A|^T |B|^T respectively; the adapter term adds
2^-15 for the bf16 hi / lo split of T and B on the tensor-core path.

Inputs are seeded: codes, zeros and scales drawn at random and packed, or a
layer quantized by the GPTQ oracle; the loss of the packed layer measured from
its output is compared with the oracle's.
"""
import numpy as np
import pytest

from oracle import gptq as og
from oracle import pack as opk
from oracle import packed_linear as pl

from tests._helpers import rel_fro

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def gq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import post_weight_quantization_30_b300 as gq

    return gq


def _bf16(a):
    """float64 values of `a` rounded to bf16 (nearest even), and the bf16 device tensor."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.float().numpy().astype(np.float64), t.cuda()


def _random_layer(rows, cols, bits, group, seed):
    rng = np.random.default_rng(seed)
    maxq = 2 ** bits - 1
    codes = rng.integers(0, maxq + 1, (rows, cols)).astype(np.uint8)
    zeros = rng.integers(0, maxq + 1, (cols // group, rows)).astype(np.uint8)
    scales = rng.uniform(0.005, 0.05, (cols // group, rows)).astype(np.float32)
    return opk.pack_qweight(codes, bits), scales, opk.pack_qzeros(zeros, bits)


def _run(gq, X, packed, rows, cols, bits, group, A=None, B=None):
    qw, s, qz = packed
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    Y = gq.gptq_packed_linear(X, dev(qw), dev(s), dev(qz), rows, cols, bits, group,
                              None if A is None else dev(A.astype(np.float32)),
                              None if B is None else dev(B.astype(np.float32)))
    gq.gq_check_device()
    return Y.cpu().numpy().astype(np.float64)


def _check(Yg, x64, packed, rows, cols, bits, group, A=None, B=None):
    qw, s, qz = packed
    r = 0 if A is None else A.shape[0]
    A64 = None if A is None else A.astype(np.float32).astype(np.float64)
    B64 = None if B is None else B.astype(np.float32).astype(np.float64)
    ref = pl.packed_linear(x64, qw, s, qz, bits, group, rows, cols, A64, B64)
    W_hat = pl.dequantize(qw, s, qz, bits, group, rows, cols)
    # the decode path (n <= 32) sums a group's products one by one and its K slices in a final pass
    decode = x64.shape[0] <= 32
    steps = (group if decode else group // 16) + 2 * (cols // group) + r + 2
    bound = steps * 2.0 ** -23 * (np.abs(x64) @ np.abs(W_hat).T)
    if r:
        # T = X A^T is a float32 sum of cols products, then r more additions into Y; on the tensor-core
        # path T and B also go through a bf16 hi + lo split (each off by <= 2^-18 relative, the dropped
        # lo x lo term likewise): 2^-15 covers the four of them twice over.
        bound = bound + ((cols + r + 2) * 2.0 ** -23 + 2.0 ** -15) * ((np.abs(x64) @ np.abs(A64).T) @ np.abs(B64).T)
    err = np.abs(Yg - ref)
    assert np.all(err <= bound + 1e-30), float(np.max(err / (bound + 1e-30)))
    assert rel_fro(Yg, ref) <= 1e-5
    return ref


CASES = [
    # n, rows, cols, bits, group, r
    (256, 256, 512, 4, 128, 0),
    (300, 96, 640, 3, 64, 16),     # ragged token tile, a partial 128-row tile of W
    (128, 128, 128, 2, 64, 64),    # one k-tile group pair, the largest adapter
    (1, 64, 256, 4, 64, 8),        # a single token (decode)
    (1000, 384, 1024, 2, 128, 5),  # r = 5
    (129, 160, 192, 3, 192, 0),    # one group spanning three k-tiles
    # decode path (n <= 32): SIMT, split over K, fixed-order reduction
    (16, 256, 1024, 3, 128, 8),
    (32, 96, 640, 2, 64, 0),
    (4, 384, 512, 4, 128, 64),
    (5, 64, 256, 3, 64, 3),
    (33, 128, 256, 4, 64, 4),      # the smallest tensor-core case
]


@pytest.mark.parametrize("n,rows,cols,bits,group,r", CASES)
def test_matches_the_oracle(gq, n, rows, cols, bits, group, r):
    rng = np.random.default_rng(100 + n + rows + r)
    packed = _random_layer(rows, cols, bits, group, n + cols)
    x64, X = _bf16(rng.standard_normal((n, cols)))
    A = rng.standard_normal((r, cols)) * 0.05 if r else None
    B = rng.standard_normal((rows, r)) * 0.05 if r else None
    Yg = _run(gq, X, packed, rows, cols, bits, group, A, B)
    _check(Yg, x64, packed, rows, cols, bits, group, A, B)


def test_strided_input_and_zero_tokens(gq):
    rows, cols, bits, group = 64, 256, 4, 64
    rng = np.random.default_rng(7)
    packed = _random_layer(rows, cols, bits, group, 8)
    big = torch.from_numpy(rng.standard_normal((70, cols + 40)).astype(np.float32)).to(torch.bfloat16).cuda()
    X = big[:, :cols]  # row stride cols + 40 (a multiple of 8)
    x64 = X.float().cpu().numpy().astype(np.float64)
    Yg = _run(gq, X, packed, rows, cols, bits, group)
    _check(Yg, x64, packed, rows, cols, bits, group)
    Y0 = _run(gq, X[:0], packed, rows, cols, bits, group)
    assert Y0.shape == (0, rows)


def test_loss_of_a_gptq_layer_from_its_packed_form(gq):
    """A layer quantized by the oracle: the output loss ||X W^T - Y||^2 computed from the GPU's Y equals the
    oracle's (1e-4), and equals the Hessian form of the layer loss."""
    rows, cols, n, bits, group = 128, 256, 2048, 2, 64
    rng = np.random.default_rng(9)
    x = rng.standard_normal((n, cols))
    x[:, rng.choice(cols, 3, replace=False)] *= 20.0
    x64, X = _bf16(x)
    W = rng.standard_normal((rows, cols)) * 0.02
    H = og.hessian(x64)
    q = og.quantize_layer(W, H, bits, group, 0.01)
    packed = (opk.pack_qweight(q["codes"], bits), q["scales"], opk.pack_qzeros(q["zeros"], bits))
    Yg = _run(gq, X, packed, rows, cols, bits, group)
    ref = _check(Yg, x64, packed, rows, cols, bits, group)
    lg = pl.output_loss(x64, W, Yg)
    lo = pl.output_loss(x64, W, ref)
    assert lg == pytest.approx(lo, rel=1e-4)
    assert lo == pytest.approx(og.layer_loss(W, pl.dequantize(*packed, bits, group, rows, cols), H), rel=1e-9)


def test_rejects_unsupported_layouts(gq):
    rows, cols, bits = 64, 256, 4
    packed = _random_layer(rows, cols, bits, 64, 1)
    _, X = _bf16(np.ones((4, cols)))
    qw, s, qz = (torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in packed)
    with pytest.raises(gq.GQError) as ei:
        gq.gptq_packed_linear(X, qw, s, qz, rows, cols, bits, 32)  # group 32: not supported by this kernel
    assert ei.value.status == -3
    with pytest.raises(gq.GQError) as ei:
        gq.gptq_packed_linear(X, qw, s, qz, rows, cols, 5, 64)
    assert ei.value.status == -3
