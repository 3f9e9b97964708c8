"""Reference decoding of AWQ checkpoint arrays (test infrastructure).

THIS IS TEST INFRASTRUCTURE (see ``oracle/tf_oracle.py``): only ``tests/``
import it, and it shares no code with the C++ ``tf_prepack_awq``.

The TileFuse pages (Introduction; Contributions 1) present the library as
running AWQ-quantised models as they are published: INT4 weights with
per-group scales and zero points, dequantised as ``(q - z) * s``.  The pages do not
print AWQ's storage layout; the layout below is the one AWQ checkpoints use
for their GEMM kernels, restated here as a definition:

* ``qweight`` int32 ``[K, N/8]``: word ``(k, c)`` carries the 4-bit codes of
  the eight output columns ``8c .. 8c+7`` at input row k; nibble ``i``
  (bits ``4i .. 4i+3``) holds column ``8c + AWQ_ORDER[i]``.
* ``qzeros`` int32 ``[K/g, N/8]``: the zero points, packed the same way.
* ``scales`` IEEE binary16 ``[K/g, N]``.

Reading (the pages fix BF16 as the dequantised precision, Methodology 1): an
imported scale is the BF16 value nearest to the FP16 one (ties to even), so
the imported layer computes ``bf16_rne((q - z) * bf16_rne(s))``.

``awq_encode`` writes the arrays from natural-order codes following the
definition nibble by nibble; ``awq_decode`` reads them back by scattering
each nibble to its column.  Neither uses an inverse permutation table.
"""

from __future__ import annotations

import numpy as np

from oracle.tf_oracle import bf16_round, bf16_value_to_bits

AWQ_ORDER = (0, 2, 4, 6, 1, 3, 5, 7)  # output column (within 8) held by nibble i

__all__ = ["AWQ_ORDER", "awq_encode", "awq_decode", "f16_bits_to_bf16_bits"]


def _pack_columns(v: np.ndarray) -> np.ndarray:
    """[R, N] values 0..15 -> uint32 [R, N/8], nibble i <- column 8c + AWQ_ORDER[i]."""
    R, N = v.shape
    v = v.astype(np.uint32).reshape(R, N // 8, 8)
    words = np.zeros((R, N // 8), dtype=np.uint32)
    for i in range(8):
        words |= v[:, :, AWQ_ORDER[i]] << np.uint32(4 * i)
    return words


def _unpack_columns(words: np.ndarray, N: int) -> np.ndarray:
    """uint32 [R, N/8] -> [R, N] uint8, column 8c + AWQ_ORDER[i] <- nibble i."""
    words = np.asarray(words).view(np.uint32)
    R = words.shape[0]
    out = np.zeros((R, N // 8, 8), dtype=np.uint8)
    for i in range(8):
        out[:, :, AWQ_ORDER[i]] = (words >> np.uint32(4 * i)) & np.uint32(0xF)
    return out.reshape(R, N)


def awq_encode(q: np.ndarray, zeros: np.ndarray, scales_f16: np.ndarray):
    """Natural codes q [N, K], zeros [N, K/g] and FP16 scales [N, K/g] -> AWQ
    (qweight int32 [K, N/8], qzeros int32 [K/g, N/8], scales uint16 [K/g, N])."""
    q = np.asarray(q)
    zeros = np.asarray(zeros)
    s16 = np.asarray(scales_f16)
    s16 = s16.view(np.uint16) if s16.dtype.itemsize == 2 else s16.astype(np.float16).view(np.uint16)
    qweight = _pack_columns(q.T).view(np.int32)
    qzeros = _pack_columns(zeros.T).view(np.int32)
    return qweight, qzeros, np.ascontiguousarray(s16.T)


def f16_bits_to_bf16_bits(bits: np.ndarray) -> np.ndarray:
    """IEEE binary16 bit patterns -> BF16 bit patterns of the nearest BF16 value."""
    v = np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float64)  # exact
    return bf16_value_to_bits(bf16_round(v))


def awq_decode(qweight: np.ndarray, qzeros: np.ndarray, scales_f16_bits: np.ndarray, N: int, K: int,
               group: int):
    """AWQ arrays -> (q [N, K] uint8, scales BF16 bits [N, K/g], zeros [N, K/g] uint8)."""
    g = K if group == 0 else group
    q = _unpack_columns(np.asarray(qweight).reshape(K, N // 8), N).T
    z = _unpack_columns(np.asarray(qzeros).reshape(K // g, N // 8), N).T
    s = f16_bits_to_bf16_bits(np.asarray(scales_f16_bits).reshape(K // g, N)).T
    return np.ascontiguousarray(q), np.ascontiguousarray(s), np.ascontiguousarray(z)
