"""Helpers of the GPU parity tests: seeded layers, transfers, tolerances."""

import numpy as np

from gemv_tf_prepack_gb300 import synth
from oracle import tf_oracle

# Tolerances of the fused outputs against the float64 oracle (relative
# Frobenius error and worst element relative to the largest reference value).
REL_FRO = 5e-3
REL_MAX = 1e-2


def to_dev_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_host_bits(t) -> np.ndarray:
    import torch
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def layer(N, K, bits, group, seed):
    import gemv_tf_prepack_gb300 as tf
    qw = synth.make_weights(N, K, bits, group, seed)
    blob = tf.prepack(qw.qweight, qw.scales, qw.zeros, N, K, bits, group)
    return qw, tf.Weights.upload(blob)


def check_close(y_bits: np.ndarray, ref: np.ndarray, what: str = ""):
    got = tf_oracle.bf16_bits_to_f64(y_bits)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    mx = np.abs(got - ref).max() / max(np.abs(ref).max(), 1e-300)
    assert rel <= REL_FRO and mx <= REL_MAX, f"{what}: rel_fro={rel:.3e} rel_max={mx:.3e}"
    return rel, mx
