"""The C ABI: the library loads, exports every declared entry point, and rejects bad
arguments on the host before touching the GPU.  CPU only (no kernel runs)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M):
            if m.group(1) not in ("if", "typedef"):
                names.add(m.group(1))
    return sorted(names)


@pytest.fixture(scope="module")
def gq():
    import post_weight_quantization_30_b300 as gq

    return gq


def test_every_declared_symbol_is_exported(gq):
    declared = _declared_functions()
    assert "gptq_quantize_layer" in declared and "gptq_hessian_accumulate" in declared
    for name in declared:
        assert hasattr(gq.lib, name), f"{name} declared in include/ but not exported"
        assert name in gq.SIGNATURES, f"{name} has no binding"


def test_abi_version_and_status_strings(gq):
    assert gq.lib.gq_abi_version() == 1
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert gq.lib.gq_status_string(code).decode().startswith("GQ_")


def test_workspace_queries(gq):
    r, c, b = 4096, 4096, 128
    sw = gq.lib.gptq_sweep_workspace_size(r, c, b)
    assert sw >= r * c * 4 + (c // b) * b * b * 4
    ql = gq.lib.gptq_quantize_layer_workspace_size(r, c, b)
    assert ql >= sw + c * c * 4
    assert gq.lib.gptq_sweep_workspace_size(0, c, b) == 0


def _call_sweep(gq, bits=4, group=128, block=128, rows=64, cols=256, W=1, F=1, ws=None, ws_bytes=0):
    p = ctypes.c_void_p
    return gq.lib.gptq_sweep(p(W), 1, rows, cols, p(F), None, bits, group, block, p(256), p(256), p(256), None, None,
                             None, p(ws), ws_bytes, None)


def test_host_side_validation(gq):
    assert _call_sweep(gq, bits=5) == -3          # unsupported bit width
    assert _call_sweep(gq, bits=1) == -3
    assert _call_sweep(gq, group=48) == -1        # group must be a multiple of 32
    assert _call_sweep(gq, block=192) == -1       # block <= 128
    assert _call_sweep(gq, group=128, block=64) == -1  # block % group
    assert _call_sweep(gq, rows=48) == -1         # rows % 32
    assert _call_sweep(gq, cols=200, group=32, block=32) == -1
    assert _call_sweep(gq, W=0) == -1             # null input
    assert _call_sweep(gq, W=256, F=256) == -7    # missing workspace
    # n == 0 is a no-op that returns before any CUDA call
    assert gq.lib.gptq_hessian_accumulate(None, 256, None, 1, 0, 256, None) == 0
    assert gq.lib.gptq_hessian_accumulate(None, 256, None, 7, 0, 256, None) == -3
    assert gq.lib.gptq_hessian_accumulate(None, 256, None, 1, 10, 100, None) == -1  # ldx < cols
    assert gq.lib.gptq_pack(None, 4, 32, 3, None, None) == -1
    assert gq.lib.gptq_pack(ctypes.c_void_p(16), 4, 36, 3, ctypes.c_void_p(16), None) == -1  # cols*bits % 32


def test_eora_host_side_validation(gq):
    p = ctypes.c_void_p
    f = gq.lib.eora_compensate
    assert f(p(256), 64, 64, p(256), 0, p(256), p(256), None, p(256), 1 << 30, None, None) == -1   # r = 0
    assert f(p(256), 512, 512, p(256), 257, p(256), p(256), None, p(256), 1 << 30, None, None) == -1  # r > 256
    assert f(p(256), 256, 256, p(256), 200, p(256), p(256), None, p(256), 1 << 30, None, None) == -1  # cols < r + 64
    assert f(p(256), 256, 256, p(256), 65, p(256), p(256), None, p(256), 16, None, None) == -7  # r = 65 accepted
    assert f(p(256), 8, 64, p(256), 16, p(256), p(256), None, p(256), 1 << 30, None, None) == -1   # r > rows
    assert f(None, 64, 64, p(256), 4, p(256), p(256), None, p(256), 1 << 30, None, None) == -1     # null dW
    assert f(p(256), 64, 64, p(256), 4, p(256), p(256), None, p(256), 16, None, None) == -7        # workspace
    assert gq.lib.eora_compensate_workspace_size(5120, 5120, 64) >= 3 * 5120 * 5120 * 4
    assert gq.lib.eora_compensate_workspace_size(5120, 5120, 256) > gq.lib.eora_compensate_workspace_size(5120, 5120, 64)


def test_intrinsic_lora_host_side_validation(gq):
    p = ctypes.c_void_p
    b = gq.lib.gptq_lora_basis
    assert b(p(256), 64, 0, p(256), None, p(256), 1 << 30, None) == -1    # r = 0
    assert b(p(256), 256, 65, p(256), None, p(256), 1 << 30, None) == -1  # r > 64
    assert b(p(256), 16, 32, p(256), None, p(256), 1 << 30, None) == -1   # r > cols
    assert b(None, 64, 4, p(256), None, p(256), 1 << 30, None) == -1      # null H
    assert b(p(256), 64, 4, p(256), None, p(256), 16, None) == -7         # workspace
    assert b(p(256), 64, 4, p(256), None, p(260), 1 << 30, None) == -7    # unaligned workspace

    f = gq.lib.gptq_intrinsic_lora
    ws = gq.lib.gptq_intrinsic_lora_workspace_size(256, 256, 16, 128)
    assert ws >= gq.lib.gptq_quantize_layer_workspace_size(256, 256, 128)

    def call(r=16, damp=0.01, W_hat=p(256), R=p(256), Lt=p(256), bits=4, ws_bytes=ws):
        return f(p(256), 0, 256, 256, p(256), Lt, r, bits, 128, 128, damp, p(256), p(256), p(256), None, W_hat, None,
                 R, p(256), ws_bytes, None, None)

    assert call(r=0) == -1
    assert call(r=65) == -1
    assert call(damp=0.0) == -1           # the augmented Hessian needs damping
    assert call(damp=float("nan")) == -1
    assert call(W_hat=None) == -1         # R is formed from W_hat
    assert call(R=None) == -1
    assert call(Lt=None) == -1
    assert call(bits=5) == -3
    assert call(ws_bytes=ws - 1) == -7


def test_packed_linear_host_side_validation(gq):
    p = ctypes.c_void_p
    f = gq.lib.gptq_packed_linear

    def call(n=8, ldx=256, rows=64, cols=256, bits=4, group=64, A=None, B=None, r=0, Y=p(256), ldy=64, ws=None,
             ws_bytes=0, X=p(256)):
        return f(X, n, ldx, p(256), p(256), p(256), rows, cols, bits, group, A, B, r, Y, ldy, ws, ws_bytes, None)

    assert call(group=32) == -3          # group 32: not supported by this kernel
    assert call(bits=8) == -3
    assert call(rows=48) == -1           # rows % 32
    assert call(ldx=260) == -1           # row stride of X not a multiple of 8
    assert call(X=p(258)) == -1          # X not 16-byte aligned
    assert call(ldy=62) == -1
    assert call(X=None) == -1
    assert call(r=65, A=p(256), B=p(256)) == -1
    assert call(r=4, A=None, B=p(256)) == -1
    assert call(r=4, A=p(256), B=p(256)) == -7     # no workspace for X A^T
    assert call(n=8) == -7                          # decode path: no workspace for the partial sums
    assert call(n=0) == 0                           # nothing to do, nothing launched
    assert gq.lib.gptq_packed_linear_workspace_size(1000, 64, 256, 64, 16) >= 1000 * 16 * 4
    assert gq.lib.gptq_packed_linear_workspace_size(1000, 64, 256, 64, 0) == 0     # prefill, no adapter
    assert gq.lib.gptq_packed_linear_workspace_size(16, 64, 256, 64, 0) >= 16 * 64 * 4


def test_bidup_host_side_validation(gq):
    p = ctypes.c_void_p
    f = gq.lib.gptq_bidup
    ws = gq.lib.gptq_bidup_workspace_size(64, 256)
    assert ws >= 4 * 64 * 256 * 4 + 2 * 256 * 256 * 4

    def call(rows=64, cols=256, bits=4, group=64, r=0, A=None, B=None, H=p(256), ws_bytes=ws):
        return f(p(256), 0, rows, cols, H, A, B, r, bits, group, p(256), p(256), p(256), p(256), None, None, p(256),
                 ws_bytes, None)

    assert call(bits=5) == -3
    assert call(rows=48) == -1          # rows % 32 (packing)
    assert call(group=48) == -1
    assert call(r=4) == -1              # a correction needs A and B
    assert call(r=65, A=p(256), B=p(256)) == -1
    assert call(H=p(260)) == -1         # H 16-byte aligned
    assert call(ws_bytes=ws - 1) == -7


def test_rtn_host_side_validation(gq):
    p = ctypes.c_void_p
    f = gq.lib.gptq_quantize_rtn
    assert f(p(256), 8, 64, 9, 64, p(256), None, p(256), p(256), None) == -3   # bits > 8
    assert f(p(256), 8, 64, 1, 64, p(256), None, p(256), p(256), None) == -3   # bits < 2
    assert f(p(256), 8, 64, 4, 48, p(256), None, p(256), p(256), None) == -1   # ncols % group
    assert f(None, 8, 64, 4, 64, p(256), None, p(256), p(256), None) == -1


def test_noalloc_checks_arguments_before_the_size_limit(gq):
    """An oversized layer with a bad argument gets the status gptq_quantize_layer gives that
    argument; only a valid oversized layer gets GQ_EWORKSPACE.  Nothing reaches the GPU."""
    p = ctypes.c_void_p
    rows = cols = 4096  # workspace far above the 16 MiB scratch
    assert gq.lib.gptq_quantize_layer_workspace_size(rows, cols, 128) > gq._lib.NOALLOC_SCRATCH_BYTES

    def call(bits=4, group=128, qweight=256, H=256):
        info = ctypes.c_int64(-1)
        return gq.lib.gptq_quantize_layer_noalloc(p(256), 1, rows, cols, p(H), bits, group, 128, 0.01, p(qweight),
                                                  p(256), p(256), None, None, None, None, ctypes.byref(info))

    assert call(bits=5) == -3           # GQ_EUNSUPPORTED
    assert call(group=100) == -1        # GQ_EINVAL
    assert call(qweight=0) == -1        # GQ_EINVAL: NULL output
    assert call(H=0) == -1              # GQ_EINVAL: NULL H
    assert call() == -7                 # GQ_EWORKSPACE: valid, but larger than the scratch
    info = ctypes.c_int64(-1)
    assert gq.lib.gptq_quantize_layer_noalloc(p(256), 1, 0, cols, p(256), 4, 128, 128, 0.01, p(256), p(256),
                                              p(256), None, None, None, None, ctypes.byref(info)) == -1


def test_binding_rejects_tensors_on_different_devices(gq):
    import torch

    a = torch.empty(4)
    assert gq._lib._same_device(a, None, torch.empty(2)) == a.device
    with pytest.raises(ValueError):
        gq._lib._same_device(a, torch.empty(4, device="meta"))


def test_kernel_timing_without_launches_reports_zeros(gq):
    with gq.kernel_timing() as kt:
        pass
    assert set(kt.ms) == set(gq._lib.TIMING_KINDS)
    assert all(v == 0 for v in kt.ms.values()) and all(v == 0 for v in kt.count.values())
    n = ctypes.c_int(0)
    assert gq.lib.gq_timing_end(None, None, None, 0) == 0
    assert gq.lib.gq_timing_end(None, None, None, 3) == -1  # GQ_EINVAL: NULL outputs
    del n
