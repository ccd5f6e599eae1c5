"""ctypes binding of libgq.so: argument marshalling only.

Every function here forwards to the C entry point of the same name declared in
include/gq.h.  Output and workspace buffers are allocated with PyTorch (device
memory is PyTorch's job; the library never allocates), pointers and the
current CUDA stream are passed through, and a non-OK status raises GQError.
There is no other code path: if libgq.so is missing, importing this module
fails.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgq.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python post_weight_quantization_30_b300/build.py` "
        "(this package has no fallback path)")

lib = ctypes.CDLL(LIB_PATH)

_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t

GQ_F32, GQ_BF16 = 0, 1
STATUS = {0: "GQ_OK", -1: "GQ_EINVAL", -2: "GQ_ENOTPD", -3: "GQ_EUNSUPPORTED", -4: "GQ_ECUDA",
          -5: "GQ_ENONFINITE", -6: "GQ_ETIMEOUT", -7: "GQ_EWORKSPACE"}

# name -> (restype, argtypes); the full exported surface of include/gq.h
SIGNATURES = {
    "gq_abi_version": (_i, []),
    "gq_kernel_launches": (ctypes.c_ulonglong, []),
    "gq_status_string": (ctypes.c_char_p, [_i]),
    "gq_check_device": (_i, [_p]),
    "gq_set_wait_budget": (_i, [ctypes.c_longlong]),
    "gq_timing_begin": (_i, []),
    "gq_timing_end": (_i, [_p, _p, _p, _i]),
    "gptq_hessian_accumulate": (_i, [_p, _i64, _p, _i, _i64, _i64, _p]),
    "gptq_factor_workspace_size": (_sz, [_i64]),
    "gptq_factor": (_i, [_p, _i64, _f, _p, _p, _p, _sz, _p, ctypes.POINTER(_i64)]),
    "gptq_sweep_workspace_size": (_sz, [_i64, _i64, _i]),
    "gptq_sweep": (_i, [_p, _i, _i64, _i64, _p, _p, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _sz, _p]),
    "gptq_quantize_layer_workspace_size": (_sz, [_i64, _i64, _i]),
    "gptq_quantize_layer": (_i, [_p, _i, _i64, _i64, _p, _i, _i, _i, _f, _p, _p, _p, _p, _p, _p, _p, _sz, _p,
                                 ctypes.POINTER(_i64)]),
    "gptq_quantize_layer_noalloc": (_i, [_p, _i, _i64, _i64, _p, _i, _i, _i, _f, _p, _p, _p, _p, _p, _p, _p,
                                         ctypes.POINTER(_i64)]),
    "gptq_weight_error": (_i, [_p, _i, _i64, _i64, _p, _p, _p]),
    "eora_compensate_workspace_size": (_sz, [_i64, _i64, _i]),
    "eora_compensate": (_i, [_p, _i64, _i64, _p, _i, _p, _p, _p, _p, _sz, _p, ctypes.POINTER(_i64)]),
    "gptq_lora_basis_workspace_size": (_sz, [_i64, _i]),
    "gptq_lora_basis": (_i, [_p, _i64, _i, _p, _p, _p, _sz, _p]),
    "gptq_intrinsic_lora_workspace_size": (_sz, [_i64, _i64, _i, _i]),
    "gptq_intrinsic_lora": (_i, [_p, _i, _i64, _i64, _p, _p, _i, _i, _i, _i, _f, _p, _p, _p, _p, _p, _p, _p, _p,
                                 _sz, _p, ctypes.POINTER(_i64)]),
    "gptq_packed_linear_workspace_size": (_sz, [_i64, _i64, _i64, _i, _i]),
    "gptq_packed_linear": (_i, [_p, _i64, _i64, _p, _p, _p, _i64, _i64, _i, _i, _p, _p, _i, _p, _i64, _p, _sz, _p]),
    "gptq_bidup_workspace_size": (_sz, [_i64, _i64]),
    "gptq_bidup": (_i, [_p, _i, _i64, _i64, _p, _p, _p, _i, _i, _i, _p, _p, _p, _p, _p, _p, _p, _sz, _p]),
    "gptq_quantize_rtn": (_i, [_p, _i64, _i64, _i, _i, _p, _p, _p, _p, _p]),
    "gptq_code_decisions": (_i, [_p, _p, _i64, _p, _p]),
    "gptq_pack": (_i, [_p, _i64, _i64, _i, _p, _p]),
    "gptq_unpack": (_i, [_p, _i64, _i64, _i, _p, _p]),
}

for _name, (_res, _args) in SIGNATURES.items():
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class GQError(RuntimeError):
    def __init__(self, status: int, where: str, info: int | None = None):
        self.status = status
        self.info = info
        msg = lib.gq_status_string(status).decode()
        super().__init__(f"{where}: {msg}" + (f" (info={info})" if info is not None and info >= 0 else ""))


def _check(status: int, where: str, info: int | None = None):
    if status != 0:
        raise GQError(status, where, info)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return GQ_BF16
    if t.dtype == torch.float32:
        return GQ_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _need_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors must be CUDA device tensors")


def _same_device(*ts):
    """The one device every given tensor lives on; ValueError if they differ."""
    devs = {t.device for t in ts if t is not None}
    if len(devs) != 1:
        raise ValueError(f"tensors must all live on one device, got {sorted(str(d) for d in devs)}")
    return devs.pop()


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ entry points
def gptq_hessian_accumulate(H: torch.Tensor, X: torch.Tensor) -> torch.Tensor:
    """H += 2 X^T X (in place; returns H).  X: n x cols, row stride >= cols."""
    _need_cuda(H, X)
    n, cols = X.shape
    if X.stride(1) != 1:
        raise ValueError("X must have unit stride along its feature axis")
    if H.dtype != torch.float32 or tuple(H.shape) != (cols, cols) or not H.is_contiguous():
        raise ValueError("H must be a contiguous cols x cols float32 tensor")
    _check(lib.gptq_hessian_accumulate(_ptr(H), cols, _ptr(X), _dtype_code(X), n, X.stride(0), _stream(X.device)),
           "gptq_hessian_accumulate")
    return H


def gptq_factor(H: torch.Tensor, damp: float = 0.01):
    """Returns (F, dead): H + damp*mean(diag)*I = F F^T with F upper; dead inputs."""
    _need_cuda(H)
    cols = H.shape[0]
    F = torch.empty((cols, cols), dtype=torch.float32, device=H.device)
    dead = torch.empty(cols, dtype=torch.uint8, device=H.device)
    ws_bytes = lib.gptq_factor_workspace_size(cols)
    ws = _workspace(ws_bytes, H.device)
    info = _i64(-1)
    _check(lib.gptq_factor(_ptr(H.contiguous()), cols, float(damp), _ptr(F), _ptr(dead), _ptr(ws), ws_bytes,
                           _stream(H.device), ctypes.byref(info)), "gptq_factor", info.value)
    return F, dead


def _sweep_outputs(rows, cols, bits, group, device, codes, W_hat, row_err):
    out = dict(
        qweight=torch.empty((cols * bits // 32, rows), dtype=torch.int32, device=device),
        scales=torch.empty((cols // group, rows), dtype=torch.float32, device=device),
        qzeros=torch.empty((cols // group, rows * bits // 32), dtype=torch.int32, device=device),
        codes=torch.empty((rows, cols), dtype=torch.uint8, device=device) if codes else None,
        W_hat=torch.empty((rows, cols), dtype=torch.float32, device=device) if W_hat else None,
        row_err=torch.empty(rows, dtype=torch.float32, device=device) if row_err else None,
    )
    return out


def gptq_sweep(W: torch.Tensor, F: torch.Tensor, dead: torch.Tensor | None, bits: int, group: int, block: int = 128,
               codes: bool = True, W_hat: bool = True, row_err: bool = True, workspace: torch.Tensor | None = None):
    _need_cuda(W, F, dead)
    rows, cols = W.shape
    W = W.contiguous()
    o = _sweep_outputs(rows, cols, bits, group, W.device, codes, W_hat, row_err)
    ws_bytes = lib.gptq_sweep_workspace_size(rows, cols, block)
    ws = workspace if workspace is not None else _workspace(ws_bytes, W.device)
    _check(lib.gptq_sweep(_ptr(W), _dtype_code(W), rows, cols, _ptr(F), _ptr(dead), bits, group, block,
                          _ptr(o["qweight"]), _ptr(o["scales"]), _ptr(o["qzeros"]), _ptr(o["codes"]),
                          _ptr(o["W_hat"]), _ptr(o["row_err"]), _ptr(ws), ws.numel(), _stream(W.device)),
           "gptq_sweep")
    return o


def gptq_quantize_layer(W: torch.Tensor, H: torch.Tensor, bits: int, group: int, block: int = 128,
                        damp: float = 0.01, codes: bool = True, W_hat: bool = True, row_err: bool = True,
                        workspace: torch.Tensor | None = None, out: dict | None = None):
    """Dead inputs + damping, factor, sweep, packing.  Returns a dict of device tensors."""
    _need_cuda(W, H)
    rows, cols = W.shape
    W = W.contiguous()
    o = out if out is not None else _sweep_outputs(rows, cols, bits, group, W.device, codes, W_hat, row_err)
    ws_bytes = lib.gptq_quantize_layer_workspace_size(rows, cols, block)
    ws = workspace if workspace is not None else _workspace(ws_bytes, W.device)
    info = _i64(-1)
    _check(lib.gptq_quantize_layer(_ptr(W), _dtype_code(W), rows, cols, _ptr(H.contiguous()), bits, group, block,
                                   float(damp), _ptr(o["qweight"]), _ptr(o["scales"]), _ptr(o["qzeros"]),
                                   _ptr(o.get("codes")), _ptr(o.get("W_hat")), _ptr(o.get("row_err")), _ptr(ws),
                                   ws.numel(), _stream(W.device), ctypes.byref(info)),
           "gptq_quantize_layer", info.value)
    return o


NOALLOC_SCRATCH_BYTES = 16 << 20  # GQ_NOALLOC_SCRATCH_BYTES in include/gq.h


def gptq_quantize_layer_noalloc(W: torch.Tensor, H: torch.Tensor, bits: int, group: int, block: int = 128,
                                damp: float = 0.01, out: dict | None = None, codes: bool = True, W_hat: bool = True,
                                row_err: bool = True):
    """gptq_quantize_layer with the library's fixed 16 MiB scratch instead of a workspace.

    For callers that must not allocate device scratch.  Output buffers are
    still the caller's: pass ``out`` (same keys as gptq_quantize_layer returns)
    to allocate nothing at all.  Layers whose workspace exceeds the fixed
    scratch are rejected.  Calls that overlap on the GPU race on the scratch.
    """
    _need_cuda(W, H)
    rows, cols = W.shape
    need = lib.gptq_quantize_layer_workspace_size(rows, cols, block)
    if need > NOALLOC_SCRATCH_BYTES:
        raise ValueError(f"layer {rows}x{cols} (block {block}) needs {need} bytes of scratch; the fixed scratch "
                         f"holds {NOALLOC_SCRATCH_BYTES}: use gptq_quantize_layer with a workspace")
    W = W.contiguous()
    o = out if out is not None else _sweep_outputs(rows, cols, bits, group, W.device, codes, W_hat, row_err)
    # The library takes the scratch of the current device: make W's device current for the call.
    dev = _same_device(W, H, *o.values())
    info = _i64(-1)
    with torch.cuda.device(dev):
        _check(lib.gptq_quantize_layer_noalloc(_ptr(W), _dtype_code(W), rows, cols, _ptr(H.contiguous()), bits,
                                               group, block, float(damp), _ptr(o["qweight"]), _ptr(o["scales"]),
                                               _ptr(o["qzeros"]), _ptr(o.get("codes")), _ptr(o.get("W_hat")),
                                               _ptr(o.get("row_err")), _stream(dev), ctypes.byref(info)),
               "gptq_quantize_layer_noalloc", info.value)
    return o


def gptq_weight_error(W: torch.Tensor, W_hat: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """dW = W - W_hat (float32), the error EoRA compensates."""
    _need_cuda(W, W_hat)
    rows, cols = W.shape
    W = W.contiguous()
    dW = out if out is not None else torch.empty((rows, cols), dtype=torch.float32, device=W.device)
    _check(lib.gptq_weight_error(_ptr(W), _dtype_code(W), rows, cols, _ptr(W_hat.contiguous()), _ptr(dW),
                                 _stream(W.device)), "gptq_weight_error")
    return dW


def eora_compensate(dW: torch.Tensor, H: torch.Tensor, r: int, workspace: torch.Tensor | None = None,
                    out: dict | None = None):
    """EoRA factors of the quantization error dW = W - Ŵ: returns dict(A, B, sigma)."""
    _need_cuda(dW, H)
    rows, cols = dW.shape
    dW = dW.contiguous()
    if dW.dtype != torch.float32 or H.dtype != torch.float32:
        raise ValueError("dW and H must be float32")
    o = out if out is not None else dict(
        A=torch.empty((r, cols), dtype=torch.float32, device=dW.device),
        B=torch.empty((rows, r), dtype=torch.float32, device=dW.device),
        sigma=torch.empty(r, dtype=torch.float32, device=dW.device))
    ws_bytes = lib.eora_compensate_workspace_size(rows, cols, r)
    ws = workspace if workspace is not None else _workspace(ws_bytes, dW.device)
    info = _i64(-1)
    _check(lib.eora_compensate(_ptr(dW), rows, cols, _ptr(H.contiguous()), r, _ptr(o["A"]), _ptr(o["B"]),
                               _ptr(o.get("sigma")), _ptr(ws), ws.numel(), _stream(dW.device), ctypes.byref(info)),
           "eora_compensate", info.value)
    return o


def gptq_lora_basis(H: torch.Tensor, r: int, workspace: torch.Tensor | None = None, out: dict | None = None):
    """The GPTQ-intrinsic LoRA basis: dict(Lt = the r leading eigenvectors of H as rows, lam = their Ritz values)."""
    _need_cuda(H)
    cols = H.shape[0]
    if H.dtype != torch.float32:
        raise ValueError("H must be float32")
    o = out if out is not None else dict(Lt=torch.empty((r, cols), dtype=torch.float32, device=H.device),
                                         lam=torch.empty(r, dtype=torch.float32, device=H.device))
    ws_bytes = lib.gptq_lora_basis_workspace_size(cols, r)
    ws = workspace if workspace is not None else _workspace(ws_bytes, H.device)
    _check(lib.gptq_lora_basis(_ptr(H.contiguous()), cols, r, _ptr(o["Lt"]), _ptr(o.get("lam")), _ptr(ws),
                               ws.numel(), _stream(H.device)), "gptq_lora_basis")
    return o


def gptq_intrinsic_lora(W: torch.Tensor, H: torch.Tensor, Lt: torch.Tensor, bits: int, group: int, block: int = 128,
                        damp: float = 0.01, codes: bool = True, row_err: bool = True,
                        workspace: torch.Tensor | None = None, out: dict | None = None):
    """GPTQ-intrinsic LoRA: W ≈ Ŵ + R Lt.  Returns the gptq_quantize_layer outputs plus R (rows x r)."""
    _need_cuda(W, H, Lt)
    rows, cols = W.shape
    r = Lt.shape[0]
    W = W.contiguous()
    if H.dtype != torch.float32 or Lt.dtype != torch.float32:
        raise ValueError("H and Lt must be float32")
    if out is not None:
        o = out
    else:
        o = _sweep_outputs(rows, cols, bits, group, W.device, codes, True, row_err)
        o["R"] = torch.empty((rows, r), dtype=torch.float32, device=W.device)
    ws_bytes = lib.gptq_intrinsic_lora_workspace_size(rows, cols, r, block)
    ws = workspace if workspace is not None else _workspace(ws_bytes, W.device)
    info = _i64(-1)
    _check(lib.gptq_intrinsic_lora(_ptr(W), _dtype_code(W), rows, cols, _ptr(H.contiguous()), _ptr(Lt.contiguous()),
                                   r, bits, group, block, float(damp), _ptr(o["qweight"]), _ptr(o["scales"]),
                                   _ptr(o["qzeros"]), _ptr(o.get("codes")), _ptr(o["W_hat"]), _ptr(o.get("row_err")),
                                   _ptr(o["R"]), _ptr(ws), ws.numel(), _stream(W.device), ctypes.byref(info)),
           "gptq_intrinsic_lora", info.value)
    return o


def gptq_packed_linear(X: torch.Tensor, qweight: torch.Tensor, scales: torch.Tensor, qzeros: torch.Tensor, rows: int,
                       cols: int, bits: int, group: int, A: torch.Tensor | None = None, B: torch.Tensor | None = None,
                       out: torch.Tensor | None = None, workspace: torch.Tensor | None = None) -> torch.Tensor:
    """Y = X Ŵ^T (+ (X A^T) B^T) from the packed layer; X bf16 (n x cols), Y float32 (n x rows)."""
    _need_cuda(X, qweight, scales, qzeros, A, B)
    if X.dtype != torch.bfloat16:
        raise ValueError("X must be bf16")
    n = X.shape[0]
    r = 0 if A is None else A.shape[0]
    Y = out if out is not None else torch.empty((n, rows), dtype=torch.float32, device=X.device)
    ws_bytes = lib.gptq_packed_linear_workspace_size(n, rows, cols, group, r)
    ws = workspace if workspace is not None else (_workspace(ws_bytes, X.device) if ws_bytes else None)
    _check(lib.gptq_packed_linear(_ptr(X), n, X.stride(0), _ptr(qweight.contiguous()), _ptr(scales.contiguous()),
                                  _ptr(qzeros.contiguous()), rows, cols, bits, group,
                                  _ptr(None if A is None else A.contiguous()),
                                  _ptr(None if B is None else B.contiguous()), r, _ptr(Y), Y.stride(0), _ptr(ws),
                                  0 if ws is None else ws.numel(), _stream(X.device)), "gptq_packed_linear")
    return Y


def gptq_bidup(W: torch.Tensor, H: torch.Tensor, codes: torch.Tensor, scales: torch.Tensor, qzeros: torch.Tensor,
               bits: int, group: int, A: torch.Tensor | None = None, B: torch.Tensor | None = None,
               W_hat: torch.Tensor | None = None, qweight: torch.Tensor | None = None,
               workspace: torch.Tensor | None = None) -> dict:
    """One Bid-Up sweep: `codes` refined in place against W - B A.  Returns dict(codes, W_hat, qweight, changed)."""
    _need_cuda(W, H, codes, scales, qzeros, A, B)
    rows, cols = W.shape
    W = W.contiguous()
    r = 0 if A is None else A.shape[0]
    Wh = W_hat if W_hat is not None else torch.empty((rows, cols), dtype=torch.float32, device=W.device)
    changed = torch.zeros(1, dtype=torch.int64, device=W.device)
    ws = workspace if workspace is not None else _workspace(lib.gptq_bidup_workspace_size(rows, cols), W.device)
    _check(lib.gptq_bidup(_ptr(W), _dtype_code(W), rows, cols, _ptr(H.contiguous()),
                          _ptr(None if A is None else A.contiguous()), _ptr(None if B is None else B.contiguous()), r,
                          bits, group, _ptr(codes), _ptr(scales.contiguous()), _ptr(qzeros.contiguous()), _ptr(Wh),
                          _ptr(qweight), _ptr(changed), _ptr(ws), ws.numel(), _stream(W.device)), "gptq_bidup")
    return dict(codes=codes, W_hat=Wh, qweight=qweight, changed=changed)


def gptq_quantize_rtn(M: torch.Tensor, bits: int, group: int | None = None) -> dict:
    """Round to nearest on the GPTQ grid per row and group (default: the whole row).  float32 M."""
    _need_cuda(M)
    if M.dtype != torch.float32:
        raise ValueError("M must be float32")
    nrows, ncols = M.shape
    group = ncols if group is None else group
    M = M.contiguous()
    o = dict(M_hat=torch.empty_like(M), codes=torch.empty((nrows, ncols), dtype=torch.uint8, device=M.device),
             scales=torch.empty((ncols // group, nrows), dtype=torch.float32, device=M.device),
             zeros=torch.empty((ncols // group, nrows), dtype=torch.uint8, device=M.device))
    _check(lib.gptq_quantize_rtn(_ptr(M), nrows, ncols, bits, group, _ptr(o["M_hat"]), _ptr(o["codes"]),
                                 _ptr(o["scales"]), _ptr(o["zeros"]), _stream(M.device)), "gptq_quantize_rtn")
    return o


TIMING_KINDS = ("hessian", "gemm3", "sweep", "diag", "gemm_tf32")


class kernel_timing:
    """Context manager around gq_timing_begin / gq_timing_end: on exit, ``.ms``,
    ``.flops`` and ``.count`` map each kernel class of TIMING_KINDS to its summed
    CUDA-event time, declared useful flops and launch count."""

    def __enter__(self):
        _check(lib.gq_timing_begin(), "gq_timing_begin")
        return self

    def __exit__(self, *exc):
        n = len(TIMING_KINDS)
        ms, fl = (ctypes.c_double * n)(), (ctypes.c_double * n)()
        cnt = (ctypes.c_ulonglong * n)()
        st = lib.gq_timing_end(ctypes.cast(ms, _p), ctypes.cast(fl, _p), ctypes.cast(cnt, _p), n)
        self.ms = dict(zip(TIMING_KINDS, list(ms)))
        self.flops = dict(zip(TIMING_KINDS, list(fl)))
        self.count = dict(zip(TIMING_KINDS, [int(c) for c in cnt]))
        if exc[0] is None:
            _check(st, "gq_timing_end")
        return False


def gq_check_device(device=None):
    """Raise GQError(GQ_ETIMEOUT) if a bounded device-side wait gave up since the last check."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    _check(lib.gq_check_device(_stream(dev)), "gq_check_device")


def gptq_code_decisions(w: torch.Tensor, s: torch.Tensor) -> torch.Tensor:
    """rint(w / s) elementwise by the sweep's decision rule (float32)."""
    _need_cuda(w, s)
    w = w.contiguous()
    s = s.contiguous()
    k = torch.empty_like(w)
    _check(lib.gptq_code_decisions(_ptr(w), _ptr(s), w.numel(), _ptr(k), _stream(w.device)), "gptq_code_decisions")
    return k


def gptq_pack(codes: torch.Tensor, bits: int) -> torch.Tensor:
    _need_cuda(codes)
    rows, cols = codes.shape
    qw = torch.empty((cols * bits // 32, rows), dtype=torch.int32, device=codes.device)
    _check(lib.gptq_pack(_ptr(codes.contiguous()), rows, cols, bits, _ptr(qw), _stream(codes.device)), "gptq_pack")
    return qw


def gptq_unpack(qweight: torch.Tensor, rows: int, cols: int, bits: int) -> torch.Tensor:
    _need_cuda(qweight)
    codes = torch.empty((rows, cols), dtype=torch.uint8, device=qweight.device)
    _check(lib.gptq_unpack(_ptr(qweight.contiguous()), rows, cols, bits, _ptr(codes), _stream(qweight.device)),
           "gptq_unpack")
    return codes
