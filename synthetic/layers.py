"""Deterministic synthetic GPTQ layers.

Every tensor is generated in independent chunks of ``CHUNK_ROWS`` rows.  Chunk
``c`` of a tensor draws from ``numpy.random.default_rng(SeedSequence(seed,
spawn_key=key + (c,)))`` (PCG64), so any row range can be regenerated on its
own, in any process, with identical bytes.  Values are drawn in float32 and,
for bf16 tensors, rounded to bfloat16 with round-to-nearest-even; bf16 tensors
are returned as their raw uint16 bit patterns so that both sides read the same
bytes.

Distributions (the layer shapes of the quantization workloads):

* ``normal``      -- N(0, 1)
* ``t``           -- Student-t with ``nu`` degrees of freedom, drawn as
                     Z * sqrt(nu / chi2_nu) with chi2_nu = 2 * Gamma(nu / 2)
* ``absnormal_x_normal`` -- |Z1| * Z2 (a post-SiLU-like product)

then multiplied by ``std``.  Outlier channels are whole columns multiplied by
``outlier_scale``; the set of ``n_outliers`` columns is drawn without
replacement from its own stream.
"""
from __future__ import annotations

import multiprocessing as mp
import os
from concurrent.futures import ProcessPoolExecutor
from dataclasses import dataclass, field, replace

import numpy as np

CHUNK_ROWS = 8192
_OUTLIER_STREAM = 1 << 20  # spawn-key component reserved for the outlier-channel draw
SEED = 0


@dataclass(frozen=True)
class TensorSpec:
    rows: int
    cols: int
    dist: str  # "normal" | "t" | "absnormal_x_normal"
    std: float = 1.0
    nu: float = 0.0
    n_outliers: int = 0
    outlier_scale: float = 1.0
    dtype: str = "bf16"  # "bf16" | "f32"
    key: tuple = ()
    seed: int = SEED

    @property
    def nbytes(self) -> int:
        return self.rows * self.cols * (2 if self.dtype == "bf16" else 4)

    @property
    def np_dtype(self):
        return np.uint16 if self.dtype == "bf16" else np.float32


@dataclass(frozen=True)
class LayerSpec:
    """One linear layer W (rows x cols = out x in) with calibration X (n x cols)."""

    name: str
    W: TensorSpec
    X: TensorSpec
    bits: int
    group: int
    block: int = 128
    damp: float = 0.01
    eora_rank: int = 0
    lora_rank: int = 0  # GPTQ-intrinsic LoRA rank (0: plain GPTQ)
    packed_tokens: int = 0  # > 0: the workload is the packed layer applied to this many tokens (X is n x cols)
    refine_cycles: int = 0  # > 0: after GPTQ, this many OLrC (rank eora_rank) + Bid-Up cycles
    notes: str = field(default="", compare=False)

    @property
    def rows(self) -> int:
        return self.W.rows

    @property
    def cols(self) -> int:
        return self.W.cols

    @property
    def n(self) -> int:
        return self.X.rows


def _w(rows, cols, std, key, dtype="bf16"):
    return TensorSpec(rows, cols, "normal", std=std, dtype=dtype, key=key)


_X_LLAMA7B_4096 = TensorSpec(262144, 4096, "t", nu=4.0, n_outliers=41, outlier_scale=30.0, key=(1, 1))
_X_LLAMA7B_11008 = TensorSpec(262144, 11008, "absnormal_x_normal", key=(2, 3))
_X_QWEN72B_8192 = TensorSpec(131072, 8192, "t", nu=3.0, n_outliers=41, outlier_scale=50.0, key=(3, 2))
_X_QWEN32B_5120 = TensorSpec(65536, 5120, "normal", n_outliers=51, outlier_scale=30.0, key=(4, 2))

# The quantization workloads: Llama/Qwen-shaped linear layers.  Outlier counts
# are round(fraction * cols): 1 % of 4096 -> 41, 0.5 % of 8192 -> 41,
# 1 % of 5120 -> 51.
LAYERS: dict[str, LayerSpec] = {
    s.name: s
    for s in [
        LayerSpec(
            "tiny_256x256",
            W=_w(256, 256, 0.02, (0, 0), dtype="f32"),
            X=TensorSpec(2048, 256, "normal", n_outliers=4, outlier_scale=20.0, dtype="f32", key=(0, 1)),
            bits=4, group=128,
        ),
        LayerSpec("llama7b_q_proj_4096x4096", W=_w(4096, 4096, 0.02, (1, 0)), X=_X_LLAMA7B_4096, bits=4, group=128),
        LayerSpec("llama7b_up_proj_11008x4096", W=_w(11008, 4096, 0.02, (2, 0)), X=_X_LLAMA7B_4096, bits=3, group=128),
        LayerSpec("llama7b_down_proj_4096x11008", W=_w(4096, 11008, 0.02, (2, 2)), X=_X_LLAMA7B_11008, bits=3, group=128),
        LayerSpec("qwen72b_8192x8192", W=_w(8192, 8192, 0.015, (3, 0)), X=_X_QWEN72B_8192, bits=2, group=64),
        LayerSpec("qwen72b_29568x8192", W=_w(29568, 8192, 0.015, (3, 1)), X=_X_QWEN72B_8192, bits=2, group=64),
        LayerSpec("qwen32b_5120x5120", W=_w(5120, 5120, 0.02, (4, 0)), X=_X_QWEN32B_5120, bits=2, group=64, eora_rank=64),
        LayerSpec("qwen32b_25600x5120", W=_w(25600, 5120, 0.02, (4, 1)), X=_X_QWEN32B_5120, bits=2, group=64, eora_rank=64),
        # The quantized layer applied from its packed form (inference): prefill and decode
        # token counts; the EoRA-shaped layer with its rank-64 adapter.  X here holds the
        # tokens the layer is applied to.
        LayerSpec("llama7b_q_proj_packed_prefill_n4096", W=_w(4096, 4096, 0.02, (1, 0)),
                  X=TensorSpec(4096, 4096, "t", nu=4.0, n_outliers=41, outlier_scale=30.0, key=(5, 1)), bits=4,
                  group=128, packed_tokens=4096),
        LayerSpec("llama7b_q_proj_packed_decode_n1", W=_w(4096, 4096, 0.02, (1, 0)),
                  X=TensorSpec(1, 4096, "t", nu=4.0, n_outliers=41, outlier_scale=30.0, key=(5, 2)), bits=4,
                  group=128, packed_tokens=1),
        LayerSpec("llama7b_q_proj_packed_decode_n16", W=_w(4096, 4096, 0.02, (1, 0)),
                  X=TensorSpec(16, 4096, "t", nu=4.0, n_outliers=41, outlier_scale=30.0, key=(5, 3)), bits=4,
                  group=128, packed_tokens=16),
        LayerSpec("qwen32b_5120x5120_packed_eora_r64_n4096", W=_w(5120, 5120, 0.02, (4, 0)),
                  X=TensorSpec(4096, 5120, "normal", n_outliers=51, outlier_scale=30.0, key=(5, 4)), bits=2,
                  group=64, eora_rank=64, packed_tokens=4096),
        # GPTQ followed by two OLrC + Bid-Up refinement cycles at rank 64.
        LayerSpec("qwen32b_5120x5120_refine_r64_c2", W=_w(5120, 5120, 0.02, (4, 0)), X=_X_QWEN32B_5120, bits=2,
                  group=64, eora_rank=64, refine_cycles=2),
        # The same two layers with a rank-64 GPTQ-intrinsic LoRA in place of EoRA.
        LayerSpec("qwen32b_5120x5120_intrinsic_r64", W=_w(5120, 5120, 0.02, (4, 0)), X=_X_QWEN32B_5120, bits=2,
                  group=64, lora_rank=64),
        LayerSpec("qwen32b_25600x5120_intrinsic_r64", W=_w(25600, 5120, 0.02, (4, 1)), X=_X_QWEN32B_5120, bits=2,
                  group=64, lora_rank=64),
    ]
}


def custom_layer(name, rows, cols, n, *, bits=4, group=128, block=128, damp=0.01, x_dist="t", nu=4.0,
                 n_outliers=0, outlier_scale=30.0, w_std=0.02, dtype="bf16", key=(9,), eora_rank=0,
                 lora_rank=0) -> LayerSpec:
    """A small layer with the same recipe as the workloads, for parity cases."""
    key = tuple(key)
    return LayerSpec(
        name,
        W=TensorSpec(rows, cols, "normal", std=w_std, dtype=dtype, key=key + (0,)),
        X=TensorSpec(n, cols, x_dist, nu=nu, n_outliers=n_outliers, outlier_scale=outlier_scale, dtype=dtype,
                     key=key + (1,)),
        bits=bits, group=group, block=block, damp=damp, eora_rank=eora_rank, lora_rank=lora_rank,
    )


def _f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return (r >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def outlier_channels(spec: TensorSpec) -> np.ndarray:
    if spec.n_outliers == 0:
        return np.zeros(0, dtype=np.int64)
    rng = np.random.default_rng(np.random.SeedSequence(spec.seed, spawn_key=spec.key + (_OUTLIER_STREAM,)))
    return np.sort(rng.choice(spec.cols, size=spec.n_outliers, replace=False))


def _chunk(spec: TensorSpec, c: int) -> np.ndarray:
    r0 = c * CHUNK_ROWS
    nr = min(CHUNK_ROWS, spec.rows - r0)
    rng = np.random.default_rng(np.random.SeedSequence(spec.seed, spawn_key=spec.key + (c,)))
    shape = (nr, spec.cols)
    if spec.dist == "normal":
        v = rng.standard_normal(shape, dtype=np.float32)
    elif spec.dist == "t":
        z = rng.standard_normal(shape, dtype=np.float32)
        g = rng.standard_gamma(np.float32(spec.nu / 2.0), size=shape, dtype=np.float32)
        v = z * np.sqrt(np.float32(spec.nu) / (np.float32(2.0) * g))
    elif spec.dist == "absnormal_x_normal":
        z1 = rng.standard_normal(shape, dtype=np.float32)
        z2 = rng.standard_normal(shape, dtype=np.float32)
        v = np.abs(z1) * z2
    else:
        raise ValueError(f"unknown distribution {spec.dist!r}")
    if spec.std != 1.0:
        v *= np.float32(spec.std)
    if spec.n_outliers:
        v[:, outlier_channels(spec)] *= np.float32(spec.outlier_scale)
    if spec.dtype == "bf16":
        return _f32_to_bf16_bits(v)
    return v.astype(np.float32, copy=False)


def _chunk_job(args):
    spec, c = args
    return c, _chunk(spec, c)


_POOL = None


def _pool(workers):
    global _POOL
    if _POOL is None:
        # spawn: safe whether or not the parent has already initialised CUDA
        _POOL = ProcessPoolExecutor(max_workers=workers, mp_context=mp.get_context("spawn"))
    return _POOL


def generate_rows(spec: TensorSpec, r0: int, r1: int, out: np.ndarray | None = None, workers: int | None = None):
    """Rows [r0, r1) of the tensor.  r0 must be a multiple of CHUNK_ROWS or r1 - r0 <= one chunk."""
    if out is None:
        out = np.empty((r1 - r0, spec.cols), dtype=spec.np_dtype)
    c0, c1 = r0 // CHUNK_ROWS, (r1 - 1) // CHUNK_ROWS + 1
    chunks = list(range(c0, c1))
    if workers is None:
        workers = min(len(os.sched_getaffinity(0)), 16)
    if len(chunks) <= 1 or workers <= 1:
        it = (_chunk_job((spec, c)) for c in chunks)
    else:
        it = _pool(workers).map(_chunk_job, [(spec, c) for c in chunks])
    for c, a in it:
        lo, hi = c * CHUNK_ROWS, c * CHUNK_ROWS + a.shape[0]
        s0, s1 = max(lo, r0), min(hi, r1)
        out[s0 - r0:s1 - r0] = a[s0 - lo:s1 - lo]
    return out


def generate(spec: TensorSpec, out: np.ndarray | None = None, workers: int | None = None) -> np.ndarray:
    """The whole tensor (uint16 bf16 bits, or float32)."""
    return generate_rows(spec, 0, spec.rows, out=out, workers=workers)


def with_rows(spec: TensorSpec, rows: int) -> TensorSpec:
    return replace(spec, rows=rows)
