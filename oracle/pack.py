"""Bit-packing of 2/3/4-bit codes into 32-bit words.  TEST INFRASTRUCTURE ONLY.

[LowBit] section 1 says a quantization format must fix its packing layout but
prints none; the layout here is this library's reading:

* codes are written as a little-endian bitstream along the packed axis, code k
  occupying bits ``[k*b, k*b + b)`` of the stream; the stream is cut into
  32-bit words (so a 3-bit code may straddle two words: 32 codes fill exactly
  three words);
* ``qweight`` = codes of W (rows x cols) packed along the input axis, stored
  as ``[cols*b/32][rows]`` int32 (word-row major, one column of words per
  output row);
* ``qzeros`` = the zero points ``[cols/g][rows]`` packed along the row axis,
  stored as ``[cols/g][rows*b/32]`` int32; zeros are stored as is.

Pure integer arithmetic, one code at a time.
"""
from __future__ import annotations

import numpy as np


def pack_last_axis(vals: np.ndarray, bits: int) -> np.ndarray:
    """Pack ``vals[..., L]`` (each < 2**bits) into ``[..., L*bits/32]`` int32 words."""
    vals = np.asarray(vals)
    L = vals.shape[-1]
    if (L * bits) % 32:
        raise ValueError("packed length * bits must be a multiple of 32")
    if vals.size and (vals.min() < 0 or vals.max() >= (1 << bits)):
        raise ValueError("value out of range for bit width")
    nw = L * bits // 32
    words = np.zeros(vals.shape[:-1] + (nw,), dtype=np.uint64)
    v = vals.astype(np.uint64)
    for k in range(L):
        pos = k * bits
        w, sh = divmod(pos, 32)
        words[..., w] |= (v[..., k] << np.uint64(sh)) & np.uint64(0xFFFFFFFF)
        if sh + bits > 32:  # high bits spill into the next word
            words[..., w + 1] |= v[..., k] >> np.uint64(32 - sh)
    return words.astype(np.uint32).view(np.int32)


def unpack_last_axis(words: np.ndarray, bits: int, L: int) -> np.ndarray:
    w64 = np.asarray(words).view(np.uint32).astype(np.uint64)
    out = np.zeros(w64.shape[:-1] + (L,), dtype=np.uint8)
    mask = np.uint64((1 << bits) - 1)
    for k in range(L):
        pos = k * bits
        w, sh = divmod(pos, 32)
        v = w64[..., w] >> np.uint64(sh)
        if sh + bits > 32:
            v |= w64[..., w + 1] << np.uint64(32 - sh)
        out[..., k] = (v & mask).astype(np.uint8)
    return out


def pack_qweight(codes: np.ndarray, bits: int) -> np.ndarray:
    """codes rows x cols -> qweight ``[cols*b/32][rows]`` int32."""
    return np.ascontiguousarray(pack_last_axis(codes, bits).T)


def unpack_qweight(qweight: np.ndarray, bits: int, rows: int, cols: int) -> np.ndarray:
    return unpack_last_axis(np.ascontiguousarray(np.asarray(qweight).T), bits, cols)


def pack_qzeros(zeros: np.ndarray, bits: int) -> np.ndarray:
    """zeros ``[cols/g][rows]`` -> qzeros ``[cols/g][rows*b/32]`` int32."""
    return pack_last_axis(zeros, bits)


def unpack_qzeros(qzeros: np.ndarray, bits: int, rows: int) -> np.ndarray:
    return unpack_last_axis(qzeros, bits, rows)
