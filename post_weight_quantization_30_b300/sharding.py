"""One layer's quantization split over several GPUs, one process per GPU.

The Hessian is a sum over calibration tokens ("GPTQ" (wikiprompt.org),
"Enfoque Técnico": the second-order statistics of the layer inputs), so each
rank accumulates H over its own contiguous range of tokens and one all-reduce
(sum) of the cols x cols float32 matrix gives every rank the whole H.  Given H,
each rank factors it itself (the factor is replicated: at cols <= 11008 that is
cheaper than distributing it), and the rows of W are independent in the sweep,
so each rank quantizes its own range of rows with no further exchange.  The
packed outputs stay sharded along rows (columns of qweight and scales, words of
qzeros) until gather_rows collects them.

The compute steps are passed in (by default the library's own calls), so the
partition logic can be run with any implementation of the per-shard work.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

ROW_UNIT = 32  # the library packs zero points of 32 rows into b words: shards start on multiples of 32 rows


def token_range(n: int, world: int, rank: int, multiple: int = 1) -> tuple[int, int]:
    """Contiguous tokens [t0, t1) of `rank`: every token in exactly one range, ranges as even as
    possible in units of `multiple` tokens (the last unit may be shorter)."""
    if world < 1 or not 0 <= rank < world or multiple < 1 or n < 0:
        raise ValueError("bad token split")
    units = -(-n // multiple)
    u0, u1 = units * rank // world, units * (rank + 1) // world
    return min(n, u0 * multiple), min(n, u1 * multiple)


def row_range(rows: int, world: int, rank: int) -> tuple[int, int]:
    """Rows [r0, r1) of `rank`, in units of 32 rows (rows must be a multiple of 32)."""
    if rows % ROW_UNIT:
        raise ValueError(f"rows must be a multiple of {ROW_UNIT}")
    return token_range(rows, world, rank, ROW_UNIT)


def reduce_hessian(H: torch.Tensor, group=None) -> torch.Tensor:
    """H <- the sum of every rank's H (in place), the one exchange of the path."""
    dist.all_reduce(H, op=dist.ReduceOp.SUM, group=group)
    return H


def hessian_sharded(X_local: torch.Tensor, cols: int, accumulate=None, group=None) -> torch.Tensor:
    """The whole layer's H = 2 X^T X on every rank from this rank's tokens X_local (n_local x cols)."""
    if accumulate is None:
        from ._lib import gptq_hessian_accumulate as accumulate
    dtype = torch.float32 if X_local.is_cuda else torch.float64
    H = torch.zeros((cols, cols), dtype=dtype, device=X_local.device)
    if X_local.shape[0]:
        accumulate(H, X_local)
    return reduce_hessian(H, group)


def quantize_rows(W: torch.Tensor, H: torch.Tensor, bits: int, group_size: int, block: int = 128,
                  damp: float = 0.01, quantize=None, group=None):
    """This rank's rows of the whole layer W quantized against the shared H: ((r0, r1), the outputs
    of the quantize call for rows r0:r1)."""
    if quantize is None:
        from ._lib import gptq_quantize_layer as quantize
    world = dist.get_world_size(group) if dist.is_initialized() else 1
    rank = dist.get_rank(group) if dist.is_initialized() else 0
    r0, r1 = row_range(W.shape[0], world, rank)
    return (r0, r1), quantize(W[r0:r1], H, bits, group_size, block, damp)


# Axis along which each output is sharded when the rows are split, and the number of its
# entries per row (qzeros holds bits words per 32 rows).
def _row_axis(name: str, bits: int):
    if name in ("qweight", "scales"):
        return 1, 1.0
    if name == "qzeros":
        return 1, bits / 32.0
    if name in ("codes", "W_hat", "row_err"):
        return 0, 1.0
    raise KeyError(name)


def gather_rows(out: dict, rows: int, bits: int, group=None) -> dict:
    """Every rank's row shard of the outputs, concatenated in row order (on every rank)."""
    world = dist.get_world_size(group)
    full = {}
    for name, t in out.items():
        if t is None:
            continue
        axis, per_row = _row_axis(name, bits)
        sizes = [int(round((b - a) * per_row)) for a, b in (row_range(rows, world, r) for r in range(world))]
        pad = max(sizes)
        shape = list(t.shape)
        shape[axis] = pad
        buf = torch.zeros(shape, dtype=t.dtype, device=t.device)
        buf.narrow(axis, 0, t.shape[axis]).copy_(t)
        parts = [torch.empty_like(buf) for _ in range(world)]
        dist.all_gather(parts, buf, group=group)
        full[name] = torch.cat([p.narrow(axis, 0, n) for p, n in zip(parts, sizes)], dim=axis)
    return full
