"""Pins of the packing, EoRA and storage oracles (CPU only)."""
import os

import numpy as np
import pytest

from oracle import eora, gptq, pack, storage

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- packing ---
@pytest.mark.parametrize("bits", [2, 3, 4])
def test_pack_roundtrip(bits):
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 2 ** bits, size=(24, 96)).astype(np.uint8)
    qw = pack.pack_qweight(codes, bits)
    assert qw.shape == (96 * bits // 32, 24) and qw.dtype == np.int32
    assert np.array_equal(pack.unpack_qweight(qw, bits, 24, 96), codes)
    zeros = rng.integers(0, 2 ** bits, size=(3, 64)).astype(np.uint8)
    qz = pack.pack_qzeros(zeros, bits)
    assert qz.shape == (3, 64 * bits // 32)
    assert np.array_equal(pack.unpack_qzeros(qz, bits, 64), zeros)


def test_pack_hand_computed_words():
    # 4-bit, codes 0..15 along a row of 32: nibble k of word w holds code 8w+k
    c4 = np.tile(np.arange(16, dtype=np.uint8), 2)[None, :]
    w4 = pack.pack_qweight(c4, 4)[:, 0].view(np.uint32)
    assert [hex(v) for v in w4] == ["0x76543210", "0xfedcba98", "0x76543210", "0xfedcba98"]
    # 2-bit, codes 0,1,2,3 repeated: each byte is 0b11_10_01_00 = 0xe4
    c2 = np.tile(np.arange(4, dtype=np.uint8), 8)[None, :]
    assert [hex(v) for v in pack.pack_qweight(c2, 2)[:, 0].view(np.uint32)] == ["0xe4e4e4e4", "0xe4e4e4e4"]
    # 3-bit, codes 0..7 repeated over 32 columns: each run of 8 codes is the 24-bit
    # value 0xfac688 (code k at bit 3k); four runs fill 96 bits = 3 words
    c3 = np.tile(np.arange(8, dtype=np.uint8), 4)[None, :]
    w3 = pack.pack_qweight(c3, 3)[:, 0].view(np.uint32)
    assert [hex(v) for v in w3] == ["0x88fac688", "0xc688fac6", "0xfac688fa"]


def test_pack_rejects_out_of_range():
    with pytest.raises(ValueError):
        pack.pack_last_axis(np.array([[4, 0, 0, 0, 0, 0, 0, 0] * 2]), 2)


# ------------------------------------------------------------------- EoRA ---
def _setup(rows=40, cols=24, n=200, seed=0):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((n, cols))
    X[:, :2] *= 15.0
    H = gptq.hessian(X)
    W = rng.standard_normal((rows, cols)) * 0.02
    q = gptq.quantize_layer(W, H, 2, 8)
    dW = W - q["W_hat"].astype(np.float64)
    return dW, H, X


def test_eora_full_rank_reconstructs():
    dW, H, _ = _setup()
    A, B, _ = eora.eora(dW, H, min(dW.shape))
    assert np.allclose(B @ A, dW, rtol=0, atol=1e-10 * np.abs(dW).max())


def test_eora_identity_hessian_is_plain_svd():
    dW, _, _ = _setup()
    A, B, sig = eora.eora(dW, np.eye(dW.shape[1]), 5)
    A0, B0, sig0 = eora.plain_svd(dW, 5)
    assert np.allclose(B @ A, B0 @ A0, atol=1e-12)
    ref = np.linalg.svd(dW, compute_uv=False)
    assert np.allclose(sig, ref, rtol=1e-12)


def test_eora_eckart_young_residual():
    dW, H, _ = _setup()
    r = 6
    A, B, sig = eora.eora(dW, H, r)
    assert eora.compensated_loss(dW, A, B, H) == pytest.approx(0.5 * np.sum(sig[r:] ** 2), rel=1e-10)
    # and the residual loss equals the output error on the calibration activations
    _, _, X = _setup()
    Rm = dW - B @ A
    assert eora.compensated_loss(dW, A, B, H) == pytest.approx(float(np.sum((X @ Rm.T) ** 2)), rel=1e-10)


def test_eora_square_root_invariance():
    """Any S with S S^T = H gives the same factors: the eigen route Q sqrt(Λ) and the
    Cholesky route L produce the same B and A (after sign normalisation)."""
    dW, H, _ = _setup()
    r = 5
    A, B, sig = eora.eora(dW, H, r)
    L = np.linalg.cholesky(H)
    U, s2, Vt = np.linalg.svd(dW @ L, full_matrices=False)
    B2 = U[:, :r] * s2[:r]
    A2 = np.linalg.solve(L.T, Vt[:r].T).T
    A2, B2 = eora._normalize_signs(A2, B2)
    assert np.all(sig[:r + 1] / np.roll(sig, -1)[:r + 1] > 1 + 1e-6)  # separated spectrum
    assert np.allclose(B, B2, rtol=1e-9, atol=1e-12)
    assert np.allclose(A, A2, rtol=1e-9, atol=1e-9 * np.abs(A).max())


def test_eora_beats_plain_svd_on_layer_loss():
    """[EoRA-blog]: the projection minimises the layer loss, not the raw weight error."""
    dW, H, _ = _setup()
    A, B, _ = eora.eora(dW, H, 4)
    A0, B0, _ = eora.plain_svd(dW, 4)
    assert eora.compensated_loss(dW, A, B, H) < eora.compensated_loss(dW, A0, B0, H)
    assert np.linalg.norm(dW - B0 @ A0) <= np.linalg.norm(dW - B @ A)


def test_eora_rejects_singular_h():
    with pytest.raises(ValueError):
        eora.eora(np.ones((3, 3)), np.zeros((3, 3)), 1)


# ---------------------------------------------------------------- storage ---
def _golden_storage():
    rows = []
    with open(os.path.join(GOLDEN, "storage_examples.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, n, bits, val, unit, tol, cite = [p.strip() for p in line.split("|")]
            rows.append((name, float(n), int(bits), float(val), unit, float(tol), cite))
    return rows


@pytest.mark.parametrize("case", _golden_storage(), ids=lambda c: c[0])
def test_storage_worked_examples(case):
    name, n, bits, val, unit, tol, cite = case
    b = storage.weight_bytes(n, bits)
    got = {"GB": b / storage.GB, "GiB": b / storage.GiB, "B": b}[unit]
    assert abs(got - val) <= tol, (name, got, cite)


def test_llama70b_4bit_with_overhead_below_page_figure():
    # 70B at 4 bits is 35 GB of raw weights; the page's "about 40 GB" includes the rest
    raw = storage.weight_bytes(70e9, 4) / storage.GB
    assert raw == pytest.approx(35.0)
    assert raw < 40.0


def test_qwen3_14b_adapter_overhead():
    """[EoRA-blog] "Consumo de memoria de Eora": +257 MB (r=32) and +514 MB (r=64)
    on Qwen3-14B.  The layer shapes (40 layers; q,o 5120x5120; k,v 1024x5120;
    gate, up 17408x5120; down 5120x17408) are not on the page: public model facts."""
    layer = [(5120, 5120), (1024, 5120), (1024, 5120), (5120, 5120), (17408, 5120), (17408, 5120),
             (5120, 17408)]
    for r, mb in ((32, 257), (64, 514)):
        p = storage.adapter_params(layer * 40, r)
        assert abs(p * 2 / 1e6 - mb) < 1.0


def _golden_layer_storage():
    rows = []
    with open(os.path.join(GOLDEN, "layer_storage_4096x4096_g128.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            rows.append(tuple(int(p) for p in line.split("|")))
    return rows


@pytest.mark.parametrize("case", _golden_layer_storage(), ids=lambda c: f"{c[0]}bit")
def test_layer_storage_hand_computed(case):
    """Weights + per-group scale and zero point of a 4096 x 4096 layer in groups of 128."""
    bits, w_bytes, s_bytes, z_bytes, meta, total = case
    assert storage.weight_bytes(4096 * 4096, bits) == w_bytes
    assert storage.group_metadata_bytes(4096, 4096, 128, bits) == meta == s_bytes + z_bytes
    assert storage.quantized_layer_bytes(4096, 4096, bits, 128) == total == w_bytes + meta


@pytest.mark.parametrize("bits", [2, 3, 4])
def test_layer_storage_equals_packed_arrays(bits):
    """The accounting equals the bytes of the arrays the packing produces (qweight, qzeros)
    plus float32 scales, on a small layer."""
    rows, cols, group = 64, 512, 128
    rng = np.random.default_rng(bits)
    codes = rng.integers(0, 2 ** bits, (rows, cols)).astype(np.uint8)
    zeros = rng.integers(0, 2 ** bits, (cols // group, rows)).astype(np.uint8)
    scales = np.ones((cols // group, rows), dtype=np.float32)
    qw, qz = pack.pack_qweight(codes, bits), pack.pack_qzeros(zeros, bits)
    assert storage.weight_bytes(rows * cols, bits) == qw.nbytes
    assert storage.group_metadata_bytes(rows, cols, group, bits) == scales.nbytes + qz.nbytes
    assert storage.quantized_layer_bytes(rows, cols, bits, group) == qw.nbytes + scales.nbytes + qz.nbytes
