"""Parity at the full sizes of every synthetic workload, in the launch
configuration the benchmark times.

The kernels compute every output; the float64 oracle checks a sample of
output rows (all rows where that is cheap) — rows at the first and last
positions, around every 128-row block boundary the sample reaches, and
random rows — for every token.  Tolerances as in the other parity tests:
relative Frobenius error <= 5e-3 and worst element <= 1e-2 * max|ref|.
"""

import numpy as np
import pytest

import gemv_tf_prepack_gb300 as tf
from gemv_tf_prepack_gb300 import synth
from oracle import tf_oracle
from tests._gpu_util import check_close, to_dev_bf16, to_host_bits

pytestmark = pytest.mark.gpu

_LAYERS = {}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gemv_tf_prepack_gb300 import build as b
    b.build()
    import torch
    torch.cuda.set_device(0)
    yield
    _LAYERS.clear()
    torch.cuda.empty_cache()
    assert tf.device_error() == 0


def _layer(N, K, bits, group, seed):
    key = (N, K, bits, group, seed)
    if key not in _LAYERS:
        if len(_LAYERS) > 2:  # keep host and device memory bounded
            _LAYERS.clear()
        qw = synth.make_weights(N, K, bits, group, seed)
        W = tf.Weights.upload(tf.prepack(qw.qweight, qw.scales, qw.zeros, N, K, bits, group))
        _LAYERS[key] = (qw, W)
    return _LAYERS[key]


def _sample_rows(N, n_random=192, seed=0):
    rng = np.random.default_rng(seed)
    edges = [0, 1, 15, 16, 127, 128, 129, N // 2, N - 129, N - 128, N - 2, N - 1]
    rows = np.unique(np.clip(np.concatenate([edges, rng.integers(0, N, n_random)]), 0, N - 1))
    return rows


def _check(case, M, N, K, bits, group, seed, outliers, fn, rows=None):
    qw, W = _layer(N, K, bits, group, seed)
    xb = synth.make_activations(M, K, seed, outliers=outliers)
    y = to_host_bits(fn(W, to_dev_bf16(xb)))
    assert y.shape == (M, N)
    if rows is None:
        ref = tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, bits, group, K, xb)
        check_close(y, ref, case)
    else:
        ref = tf_oracle.reference_rows(qw.qweight, qw.scales, qw.zeros, bits, group, K, xb, rows)
        check_close(y[:, rows], ref, case)


@pytest.mark.parametrize("M", [1, 16])
def test_tiny_w4g128(M):
    """256 x 512, W4 g128, seed 0: the whole output."""
    for m, n, k, bits, group, seed, out in synth.workload("tiny_w4g128"):
        if m != M:
            continue
        _check(f"tiny gemm M={M}", M, n, k, bits, group, seed, out, tf.gemm)
        if M <= 8:
            _check(f"tiny gemv M={M}", M, n, k, bits, group, seed, out, tf.gemv)


@pytest.mark.parametrize("shape", [(12288, 4096, 1), (4096, 4096, 2), (22016, 4096, 3), (4096, 11008, 4)])
def test_decode_w4g128(shape):
    """The four Llama-7B-like projections at M = 1 through tf_gemv (sampled rows)."""
    N, K, seed = shape
    _check(f"decode {N}x{K}", 1, N, K, 4, 128, seed, False, tf.gemv, _sample_rows(N))


@pytest.mark.parametrize("name", ["square_w8pc", "square_w4g64"])
@pytest.mark.parametrize("M", [1, 8, 64])
def test_square_8192(name, M):
    """8192^2, W8 per channel and W4 g64, M in {1, 8, 64}: GEMV for M <= 8, GEMM always."""
    for m, n, k, bits, group, seed, out in synth.workload(name):
        if m != M:
            continue
        rows = _sample_rows(n)
        if M <= 8:
            _check(f"{name} gemv M={M}", M, n, k, bits, group, seed, out, tf.gemv, rows)
        _check(f"{name} gemm M={M}", M, n, k, bits, group, seed, out, tf.gemm, rows)


@pytest.mark.parametrize("shape", [(11008, 4096, 7), (4096, 11008, 8), (12288, 4096, 9)])
@pytest.mark.parametrize("M", [128, 512, 2048])
def test_prefill_w4g128(shape, M):
    """Prefill GEMMs with 1% outlier activation columns (sampled weight rows, every token)."""
    N, K, seed = shape
    _check(f"prefill {N}x{K} M={M}", M, N, K, 4, 128, seed, True, tf.gemm, _sample_rows(N, 96))


@pytest.mark.parametrize("shape", [(32768, 8192, 10), (8192, 32768, 11), (32768, 32768, 12)])
@pytest.mark.parametrize("M", [1, 4096])
def test_large_w4g128(shape, M):
    """The 32K range: GEMV at M = 1, GEMM at M = 4096 (sampled rows)."""
    N, K, seed = shape
    fn = tf.gemv if M == 1 else tf.gemm
    _check(f"large {N}x{K} M={M}", M, N, K, 4, 128, seed, False, fn, _sample_rows(N, 64 if M > 1 else 192))


def test_large_gemv_deterministic():
    """Run-to-run identical bits on the 32768^2 GEMV (split-K order is fixed)."""
    qw, W = _layer(32768, 32768, 4, 128, 12)
    x = to_dev_bf16(synth.make_activations(1, 32768, 12))
    a = to_host_bits(tf.gemv(W, x))
    b = to_host_bits(tf.gemv(W, x))
    np.testing.assert_array_equal(a, b)
