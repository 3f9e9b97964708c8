"""CPU oracle of the fused output epilogues (test infrastructure).

THIS IS TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import it; it shares no code with the
CUDA path.

The TileFuse pages' kernels end at the product; the steps either side of the
linear layer (attention and the non-linear layers) run elsewhere in their
hybrid runtime ("Main contributions", item 4: linear layers on the NPU,
attention and non-linear layers on the iGPU).  The library fuses three such
steps into the store of the product, and this module writes out their plain
definitions on top of the float64 layer outputs of ``tf_oracle.reference``:

* bias:      ``y[m, n] = s[m, n] + b[n]`` (the biased sum; rounded to BF16
  once at the end, like the product itself);
* SiLU gate: the gate and up projections of a gated MLP, computed as one
  layer whose rows alternate in blocks of 8 (gate rows 8j..8j+7, then up rows
  8j..8j+7), give ``h[m, f] = silu(g[m, f]) * u[m, f]`` with
  ``silu(a) = a * sigmoid(a) = a / (1 + exp(-a))`` (the sigmoid-weighted
  linear unit, Elfwing, Uchibe and Doya 2018; the gated form is the SwiGLU
  feed-forward layer, Shazeer 2020);
* QKV split: the stacked projection's outputs ``[0, nq)``, ``[nq, nq + nk)``
  and ``[nq + nk, N)`` are the three tensors q, k, v.

Everything here is float64; the one rounding to BF16 is the caller's (the
kernels round h, q, k and v once, as they round y).
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "silu",
    "gate_up_row",
    "interleave_gate_up",
    "silu_gate",
    "split_qkv",
]


def silu(a) -> np.ndarray:
    """a / (1 + exp(-a)) in float64 (exp overflow for a << 0 gives -0 / +inf = -0)."""
    a = np.asarray(a, dtype=np.float64)
    with np.errstate(over="ignore"):
        return a / (1.0 + np.exp(-a))


def gate_up_row(r):
    """Source of row r of the interleaved layer: (is_up, f) with f the row of
    the gate (is_up false) or up (is_up true) projection."""
    r = np.asarray(r)
    return (r % 16) >= 8, (r // 16) * 8 + r % 8


def interleave_gate_up(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """Rows of the interleaved layer from the two [F, ...] per-row arrays
    (codes, scales or zeros), F a multiple of 8."""
    gate, up = np.asarray(gate), np.asarray(up)
    F = gate.shape[0]
    if up.shape != gate.shape or F % 8:
        raise ValueError("gate and up must have the same shape, F a multiple of 8")
    out = np.empty((2 * F,) + gate.shape[1:], dtype=gate.dtype)
    for r in range(2 * F):
        is_up, f = gate_up_row(r)
        out[r] = up[f] if is_up else gate[f]
    return out


def silu_gate(y: np.ndarray) -> np.ndarray:
    """h [M, N/2] from the biased sums y [M, N] of an interleaved gate/up layer."""
    y = np.asarray(y, dtype=np.float64)
    M, N = y.shape
    if N % 16:
        raise ValueError("N must be a multiple of 16")
    h = np.empty((M, N // 2), dtype=np.float64)
    for r in range(N):
        is_up, f = gate_up_row(r)
        if not is_up:
            h[:, f] = silu(y[:, r]) * y[:, r + 8]
    return h


def split_qkv(y: np.ndarray, nq: int, nk: int):
    """(q, k, v) = (y[:, :nq], y[:, nq:nq + nk], y[:, nq + nk:])."""
    y = np.asarray(y)
    if not (nq >= 1 and nk >= 0 and nq + nk <= y.shape[1]):
        raise ValueError("need nq >= 1, nk >= 0, nq + nk <= N")
    return y[:, :nq], y[:, nq:nq + nk], y[:, nq + nk:]
