"""Per-channel layers whose K is not a multiple of 8, against the float64 oracle.

Groups of 32, 64 or multiples of 128 divide K, so only per-channel layers can
have K % 8 != 0.  Their activation rows are not 16-byte aligned: the stream
GEMV loads the activations element by element and takes every such layer (on
fewer CTAs than SMs when the layer has fewer 16-row slabs), the GEMM first
copies x into rows of a multiple of 8 in its workspace, and tf_dequant stores
element by element.  The cases cover INT4 and INT8, a single partial word
(K = 5), few and many rows, M from 1 to 300, and a layer reaching the
stream-K split.
"""

import numpy as np
import pytest

import gemv_tf_prepack_gb300 as tf
from gemv_tf_prepack_gb300 import synth
from oracle import tf_oracle
from tests._gpu_util import check_close, layer, to_dev_bf16, to_host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from gemv_tf_prepack_gb300 import build as b
    b.build()
    import torch
    torch.cuda.set_device(0)
    yield
    assert tf.device_error() == 0


SHAPES = [(200, 1003, 4), (130, 77, 8), (17, 5, 4), (2448, 4100, 4), (3000, 2050, 8), (4096, 8197, 4)]


@pytest.mark.parametrize("N,K,bits", SHAPES)
def test_dequant_bit_exact(N, K, bits):
    qw, W = layer(N, K, bits, 0, 61)
    q = tf_oracle.unpack(qw.qweight, bits, K)
    np.testing.assert_array_equal(to_host_bits(tf.dequant(W)), tf_oracle.dequant_bits(q, qw.scales, qw.zeros, 0))


@pytest.mark.parametrize("N,K,bits", SHAPES)
@pytest.mark.parametrize("M", [1, 3, 8])
def test_gemv(N, K, bits, M):
    qw, W = layer(N, K, bits, 0, 62)
    assert tf.gemv_workspace_size(N, K, bits, 0, M) == 0  # the stream GEMV
    xb = synth.make_activations(M, K, 62)
    y = to_host_bits(tf.gemv(W, to_dev_bf16(xb)))
    check_close(y, tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, bits, 0, K, xb),
                f"gemv K%8 {N}x{K} w{bits} M={M}")


@pytest.mark.parametrize("N,K,bits", SHAPES)
@pytest.mark.parametrize("M", [1, 37, 300])
def test_gemm(N, K, bits, M):
    import torch
    qw, W = layer(N, K, bits, 0, 63)
    assert tf.gemm_workspace_size(N, K, bits, 0, M) >= M * ((K + 7) // 8 * 8) * 2  # room for padded x
    xb = synth.make_activations(M, K, 63, outliers=True)
    x = to_dev_bf16(xb)
    y = to_host_bits(tf.gemm(W, x))
    check_close(y, tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, bits, 0, K, xb),
                f"gemm K%8 {N}x{K} w{bits} M={M}")
    np.testing.assert_array_equal(y, to_host_bits(tf.gemm(W, x)))  # same sums every run
    with pytest.raises(tf.TFError) as e:  # the padded activations need the workspace
        tf.gemm(W, x, stream_k=False)
    assert e.value.status == -4
    torch.cuda.synchronize()


def test_epilogues_on_ragged_k():
    """The split and bias epilogues on a K % 8 != 0 layer, through both kernels."""
    N, K = 2440, 1001
    qw, W = layer(N, K, 4, 0, 64)
    for M, fn, name in ((2, tf.gemv_qkv, "gemv"), (40, tf.gemm_qkv, "gemm")):
        xb = synth.make_activations(M, K, 64)
        ref = tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, 4, 0, K, xb)
        q, k, v = fn(W, to_dev_bf16(xb), 1000, 440)
        got = np.concatenate([to_host_bits(t) for t in (q, k, v)], axis=1)
        check_close(got, ref, f"{name} qkv K%8 M={M}")
