"""Storage accounting of quantized weights and low-rank adapters.  TEST INFRASTRUCTURE ONLY.

[LowBit] section 4 ("El ahorro de memoria requiere una contabilidad completa y
desglosada"): the raw weight storage is exactly parameters x bit width; scales,
zero points, unquantized layers, workspace, activations and the KV cache come
on top and are accounted separately.  [EoRA-blog] "Consumo de memoria de Eora":
a rank-r adapter on a linear layer adds ``r (in + out)`` parameters.
"""
from __future__ import annotations

GB = 1e9
GiB = float(1 << 30)


def weight_bytes(n_params: float, bits: float) -> float:
    """Ideal packed storage of the weights alone."""
    return n_params * bits / 8.0


def group_metadata_bytes(rows: int, cols: int, group: int, bits: int, scale_bytes: int = 4) -> float:
    """Scales (``scale_bytes`` each) and packed zero points of one layer, one pair per group."""
    n_groups = rows * (cols // group)
    return n_groups * scale_bytes + n_groups * bits / 8.0


def quantized_layer_bytes(rows: int, cols: int, bits: int, group: int, scale_bytes: int = 4) -> float:
    return weight_bytes(rows * cols, bits) + group_metadata_bytes(rows, cols, group, bits, scale_bytes)


def adapter_params(shapes, r: int) -> int:
    """Parameters of rank-r adapters on linear layers given as (out, in) shapes."""
    return sum(r * (o + i) for o, i in shapes)
