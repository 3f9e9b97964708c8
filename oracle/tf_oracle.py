"""CPU oracle for the TileFuse fused quantised linear layer (test infrastructure).

THIS IS TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it.  It shares no code with
the CUDA path and the CUDA path never calls it.

What it computes is the plain definition of the method on the TileFuse pages
("TileFuse: A Fused Mixed-Precision Kernel Library for Efficient Quantized
LLM Inference on AMD NPUs", section "Methodology", item 1 "Fused
mixed-precision microkernels"): packed INT4/INT8 weights are *unpacked*,
*dequantised* to BF16 with the per-group or per-channel scale and zero point,
and the result is consumed by a GEMM or a GEMV.  Fusion, tiling and on-chip
reuse change where the work happens, not what it computes, so the oracle is
that definition written out step by step:

1. unpack   ``q[n, k] = (qweight[n, k >> 3] >> 4 (k & 7)) & 0xF``  (INT4,
   eight codes per uint32, low nibble first along K); INT8 codes are bytes.
2. dequant  ``wd[n, k] = bf16_rne((q[n, k] - z[n, j]) * s[n, j])`` with
   ``j = k // g``; the integer difference and its product with the BF16 scale
   are exact, followed by one round-to-nearest-even to BF16.
3. product  ``y[m, n] = sum_k x[m, k] * wd[n, k]`` in float64 (BLAS dgemm).

Precision: float64 everywhere except the BF16 rounding of step 2, which is the
precision the pages fix for the dequantised weights (Methodology 1:
"conversion of low-bit integers to BF16").

The BF16 rounding is implemented from the definition of round-to-nearest-even
on an 8-bit significand (frexp/ldexp), not by float32 bit tricks, so it is
independent of the generator's rounding.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "bf16_round",
    "bf16_value_to_bits",
    "bf16_bits_to_f64",
    "unpack_w4",
    "unpack_w8",
    "unpack",
    "dequant",
    "dequant_bits",
    "linear_f64",
    "reference",
    "reference_rows",
]

_BF16_SIG_BITS = 8          # 1 implicit + 7 stored mantissa bits
_BF16_EMIN = -126           # exponent of the smallest normal, 2**-126
_BF16_MAX = float.fromhex("0x1.fep127")


def bf16_round(v) -> np.ndarray:
    """Round float64 values to the nearest BF16 value, ties to even.

    A finite v is written v = m * 2**e with 0.5 <= |m| < 1 (frexp).  A normal
    BF16 number carries 8 significant bits, so the representable neighbours of
    v are multiples of the quantum 2**(e - 8); below the normal range the
    quantum stays at the subnormal spacing 2**(-126 - 7).  ``np.rint`` rounds
    v / quantum half to even.  Magnitudes that round above the largest finite
    BF16 become infinities; NaN stays NaN.
    """
    v = np.asarray(v, dtype=np.float64)
    out = np.empty_like(v)
    finite = np.isfinite(v)
    out[~finite] = v[~finite]
    vf = v[finite]
    _, e = np.frexp(vf)
    e = np.maximum(e, _BF16_EMIN + 1)          # subnormal spacing below 2**-126
    quantum_exp = e - _BF16_SIG_BITS
    r = np.ldexp(np.rint(np.ldexp(vf, -quantum_exp)), quantum_exp)
    r = np.where(np.abs(r) > _BF16_MAX, np.copysign(np.inf, vf), r)
    out[finite] = r
    return out


def bf16_value_to_bits(v) -> np.ndarray:
    """uint16 bit pattern of values that are already exactly BF16."""
    f32 = np.asarray(v, dtype=np.float64).astype(np.float32)
    u = f32.view(np.uint32)
    if np.any(u & 0xFFFF):
        raise ValueError("value is not exactly representable in BF16")
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f64(b) -> np.ndarray:
    u = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def unpack_w4(qweight: np.ndarray, K: int) -> np.ndarray:
    """INT4 codes: q[n, k] = (qweight[n, k >> 3] >> 4*(k & 7)) & 0xF."""
    qweight = np.asarray(qweight, dtype=np.uint32)
    k = np.arange(K)
    words = qweight[:, k >> 3]
    shifts = (4 * (k & 7)).astype(np.uint32)
    return ((words >> shifts[None, :]) & np.uint32(0xF)).astype(np.uint8)


def unpack_w8(qweight: np.ndarray, K: int) -> np.ndarray:
    """INT8 codes are stored one per byte, [N, K]."""
    q = np.asarray(qweight, dtype=np.uint8)
    if q.shape[1] != K:
        raise ValueError("INT8 qweight must be [N, K]")
    return q.copy()


def unpack(qweight: np.ndarray, bits: int, K: int) -> np.ndarray:
    if bits == 4:
        return unpack_w4(qweight, K)
    if bits == 8:
        return unpack_w8(qweight, K)
    raise ValueError(f"bits={bits}")


def dequant(q: np.ndarray, scales_bits: np.ndarray, zeros: np.ndarray, group: int) -> np.ndarray:
    """wd = bf16_rne((q - z) * s) as float64 values, [N, K].

    ``group`` 0 means per output channel (one group spanning all of K).
    """
    q = np.asarray(q)
    n, k = q.shape
    g = k if group == 0 else group
    j = np.arange(k) // g
    s = bf16_bits_to_f64(scales_bits)[:, j]
    z = np.asarray(zeros).astype(np.int64)[:, j]
    diff = q.astype(np.int64) - z                   # exact integer difference
    return bf16_round(diff.astype(np.float64) * s)  # exact product, one RNE


def dequant_bits(q, scales_bits, zeros, group) -> np.ndarray:
    """Dequantised weights as BF16 bit patterns (uint16 [N, K])."""
    return bf16_value_to_bits(dequant(q, scales_bits, zeros, group))


def linear_f64(x_bits: np.ndarray, wd: np.ndarray, rows_per_chunk: int = 4096) -> np.ndarray:
    """y[m, n] = sum_k x[m, k] * wd[n, k] in float64 (dgemm, chunked over N)."""
    x = bf16_bits_to_f64(x_bits)
    wd = np.asarray(wd, dtype=np.float64)
    n = wd.shape[0]
    y = np.empty((x.shape[0], n), dtype=np.float64)
    for r0 in range(0, n, rows_per_chunk):
        y[:, r0:r0 + rows_per_chunk] = x @ wd[r0:r0 + rows_per_chunk].T
    return y


def reference(qweight, scales_bits, zeros, bits: int, group: int, K: int,
              x_bits: np.ndarray, rows_per_chunk: int = 2048) -> np.ndarray:
    """Full layer: unpack -> dequant -> float64 product, chunked over N rows."""
    n = qweight.shape[0]
    y = np.empty((x_bits.shape[0], n), dtype=np.float64)
    for r0 in range(0, n, rows_per_chunk):
        r1 = min(n, r0 + rows_per_chunk)
        q = unpack(qweight[r0:r1], bits, K)
        wd = dequant(q, scales_bits[r0:r1], zeros[r0:r1], group)
        y[:, r0:r1] = linear_f64(x_bits, wd, rows_per_chunk=r1 - r0)
    return y


def reference_rows(qweight, scales_bits, zeros, bits: int, group: int, K: int,
                   x_bits: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """The layer's outputs for a subset of output rows n (for sampled checks)."""
    rows = np.asarray(rows)
    q = unpack(qweight[rows], bits, K)
    wd = dequant(q, scales_bits[rows], zeros[rows], group)
    return linear_f64(x_bits, wd)
