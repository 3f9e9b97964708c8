"""Seeded synthetic inputs for the fused quantised linear layer.

This module produces the *inputs* of the method and nothing else: a random
weight matrix quantised to AWQ-style packed INT4/INT8 codes with per-group (or
per-channel) BF16 scales and integer zeros, and BF16 activations.  It holds
none of the method's own arithmetic (unpack, dequantise, multiply); both the
CUDA path and the CPU oracle consume what it returns.

Recipe (TileFuse, "Methodology 1": INT4/INT8 weights with per-group or
per-channel scales and zero points; W4A16 and W8A16, "Main contributions 1"):

* ``W = default_rng(seed).standard_normal((N, K), float32) * 0.02``.
* Asymmetric min/max quantiser per row and group of ``g`` consecutive K
  elements, all in float32:
  ``s = bf16_rne((max - min) / Q)``, ``z = clip(rint(-min / s), 0, Q)``,
  ``q = clip(rint(w / s) + z, 0, Q)`` with ``Q = 2**bits - 1`` and ``rint``
  rounding half to even.  The scale is rounded to BF16 *before* z and q are
  derived from it.
* INT4 codes are packed eight per uint32, low nibble first along K
  (``qweight[n, c] = sum_j q[n, 8c + j] << 4j``; per channel K need not be a
  multiple of 8, and the last word's unused nibbles are zero); INT8 codes are a uint8
  ``[N, K]`` array.
* ``x = default_rng([seed, M, 1]).standard_normal((M, K), float32)``, then
  optionally ``round(0.01 K)`` outlier columns (drawn from the same generator
  after x) scaled by 20, then rounded to BF16.

All BF16 values travel as their uint16 bit patterns.
"""

from __future__ import annotations

import dataclasses

import numpy as np

__all__ = [
    "QuantisedWeights",
    "quantise",
    "make_weights",
    "make_activations",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "WORKLOADS",
    "workload",
]


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 values to BF16 (round to nearest, ties to even); uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = r.astype(np.uint16)
    nan = np.isnan(a)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class QuantisedWeights:
    """AWQ-style quantised weight of an N (out) x K (in) linear layer."""

    N: int
    K: int
    bits: int
    group: int  # 0 = per output channel (one group spanning all of K)
    qweight: np.ndarray  # uint32 [N, K/8] (4 bit) or uint8 [N, K] (8 bit)
    scales: np.ndarray  # uint16 BF16 bits [N, K/g]
    zeros: np.ndarray  # uint8 [N, K/g], values 0..2**bits-1

    @property
    def g(self) -> int:
        return self.K if self.group == 0 else self.group


def pack_w4(q: np.ndarray) -> np.ndarray:
    """Pack INT4 codes [N, K] eight per uint32, low nibble first along K."""
    n, k = q.shape
    k8 = (k + 7) // 8 * 8  # a last, partial word keeps its unused nibbles zero
    qp = np.zeros((n, k8), dtype=np.uint32)
    qp[:, :k] = q
    q = qp.reshape(n, k8 // 8, 8)
    out = np.zeros((n, k8 // 8), dtype=np.uint32)
    for j in range(8):
        out |= q[:, :, j] << np.uint32(4 * j)
    return out


def quantise(w: np.ndarray, bits: int, group: int) -> QuantisedWeights:
    """Quantise a float32 [N, K] matrix with the asymmetric min/max recipe."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    g = k if group == 0 else group
    if (k % 8 and group != 0) or k % g:
        raise ValueError(f"K={k} must be a multiple of the group {g} (and of 8 unless per channel)")
    qmax = np.float32(2**bits - 1)
    wg = w.reshape(n, k // g, g)
    mn = wg.min(axis=2)
    mx = wg.max(axis=2)
    if not (mx > mn).all():
        raise ValueError("degenerate group (max == min) in synthetic weights")
    s_bits = f32_to_bf16_bits((mx - mn) / qmax)
    s = bf16_bits_to_f32(s_bits)
    z = np.clip(np.rint(-mn / s), 0, qmax)
    q = np.clip(np.rint(wg / s[:, :, None]) + z[:, :, None], 0, qmax)
    q = q.astype(np.uint8).reshape(n, k)
    qweight = pack_w4(q) if bits == 4 else q
    return QuantisedWeights(n, k, bits, group, qweight, s_bits, z.astype(np.uint8))


def make_weights(N: int, K: int, bits: int, group: int, seed: int,
                 rows_per_chunk: int = 2048) -> QuantisedWeights:
    """Draw W ~ N(0, 0.02) with ``default_rng(seed)`` and quantise it.

    The draw is made in row chunks (the same stream as one draw) so that the
    32768 x 32768 layer needs no 4 GB float32 temporary.
    """
    rng = np.random.default_rng(seed)
    parts = []
    for r0 in range(0, N, rows_per_chunk):
        rows = min(rows_per_chunk, N - r0)
        w = rng.standard_normal((rows, K), dtype=np.float32) * np.float32(0.02)
        parts.append(quantise(w, bits, group))
    if len(parts) == 1:
        return parts[0]
    return QuantisedWeights(
        N, K, bits, group,
        np.concatenate([p.qweight for p in parts]),
        np.concatenate([p.scales for p in parts]),
        np.concatenate([p.zeros for p in parts]),
    )


def make_activations(M: int, K: int, seed: int, outliers: bool = False) -> np.ndarray:
    """BF16 activations x [M, K] (uint16 bits) from ``default_rng([seed, M, 1])``."""
    rng = np.random.default_rng([seed, M, 1])
    x = rng.standard_normal((M, K), dtype=np.float32)
    if outliers:
        n_out = int(np.rint(0.01 * K))
        cols = rng.choice(K, n_out, replace=False)
        x[:, cols] *= np.float32(20.0)
    return f32_to_bf16_bits(x)


# Synthetic Llama-class workloads (shapes of the layers the pages evaluate on).
WORKLOADS = {
    "tiny_w4g128": dict(Ms=(1, 16), shapes=[(256, 512)], bits=4, group=128, seeds=[0], outliers=False),
    "decode_w4g128": dict(Ms=(1,), shapes=[(12288, 4096), (4096, 4096), (22016, 4096), (4096, 11008)],
                          bits=4, group=128, seeds=[1, 2, 3, 4], outliers=False),
    "square_w8pc": dict(Ms=(1, 8, 64), shapes=[(8192, 8192)], bits=8, group=0, seeds=[5], outliers=False),
    "square_w4g64": dict(Ms=(1, 8, 64), shapes=[(8192, 8192)], bits=4, group=64, seeds=[6], outliers=False),
    "prefill_w4g128": dict(Ms=(128, 512, 2048), shapes=[(11008, 4096), (4096, 11008), (12288, 4096)],
                           bits=4, group=128, seeds=[7, 8, 9], outliers=True),
    "large_w4g128": dict(Ms=(1, 4096), shapes=[(32768, 8192), (8192, 32768), (32768, 32768)],
                         bits=4, group=128, seeds=[10, 11, 12], outliers=False),
}


def workload(name: str):
    """Yield (M, N, K, bits, group, seed, outliers) for every case of a workload."""
    w = WORKLOADS[name]
    for (n, k), seed in zip(w["shapes"], w["seeds"]):
        for m in w["Ms"]:
            yield m, n, k, w["bits"], w["group"], seed, w["outliers"]
