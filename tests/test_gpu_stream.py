"""The stream GEMV (M <= 8, groups of 64, multiples of 128 or per channel,
activations that fit in shared memory; one CTA per SM, or per 16-row slab on
smaller layers) against the float64 oracle.

Its arithmetic differs from the other kernels' (codes exact as FP16
subnormals, activations scaled per token by a power of two, scale and zero
applied per group in FP32), and each warp streams its own run of units,
which may cross slab boundaries.  These tests cover: every format it takes
at ragged N and K and several M, activations far outside FP16's range (both
ends), zero tokens, run-to-run determinism, the bias epilogue, and a blob
whose header does not match the call.
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


def _sms():
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count


def _is_stream(N, K, bits, group, M):
    """The routing rule: groups other than 32, M <= 8, activations of at most
    64K elements, no workspace."""
    return group != 32 and M <= 8 and M * K <= 65536 and tf.gemv_workspace_size(N, K, bits, group, M) == 0


STREAM_FORMATS = [
    (2440, 1016, 4, 0), (2440, 1152, 4, 128), (2432, 4096, 4, 64), (3000, 2048, 8, 0),
    (2560, 1280, 8, 64), (5000, 3072, 4, 128), (2450, 384, 4, 128), (2448, 1024, 4, 256),
    (2447, 520, 4, 0), (2500, 640, 8, 128), (2433, 136, 8, 0), (4104, 8192, 4, 128),
    (2600, 8192, 8, 0), (2440, 8192, 4, 64),  # M = 8: activations of 128 KB, half-size ring stages
    # fewer 16-row slabs than SMs: one CTA per slab
    (1024, 4096, 4, 128), (256, 512, 4, 128), (136, 200, 8, 0), (1000, 1016, 4, 0), (8, 8, 4, 0),
    (2048, 4096, 8, 64), (130, 256, 8, 128), (2431, 1024, 4, 128),
]


@pytest.mark.parametrize("N,K,bits,group", STREAM_FORMATS)
@pytest.mark.parametrize("M", [1, 2, 3, 8])
def test_stream_parity(N, K, bits, group, M):
    assert _is_stream(N, K, bits, group, M), "shape meant for the stream GEMV"
    qw, W = layer(N, K, bits, group, 31)
    xb = synth.make_activations(M, K, 31)
    y = to_host_bits(tf.gemv(W, to_dev_bf16(xb)))
    ref = tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, bits, group, K, xb)
    check_close(y, ref, f"stream gemv {N}x{K} w{bits} g{group} M={M}")


def _scaled_activations(M, K, seed, scales):
    x = synth.bf16_bits_to_f32(synth.make_activations(M, K, seed)).astype(np.float64)
    x *= np.asarray(scales, np.float64)[:, None]
    return synth.f32_to_bf16_bits(x.astype(np.float32))


@pytest.mark.parametrize("bits,group", [(4, 128), (8, 0), (4, 64)])
def test_stream_activation_range(bits, group):
    """Tokens far above FP16's largest value (2^17 N(0,1), up to ~10^6), far
    below its normal range (2^-30 N(0,1)), ordinary, and all zero."""
    N, K = 2600, 2048
    qw, W = layer(N, K, bits, group, 37)
    xb = _scaled_activations(4, K, 37, [2.0**17, 2.0**-30, 1.0, 0.0])
    y = to_host_bits(tf.gemv(W, to_dev_bf16(xb)))
    ref = tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, bits, group, K, xb)
    for m in range(3):  # each token against its own scale
        check_close(y[m:m + 1], ref[m:m + 1], f"token {m}")
    assert (tf_oracle.bf16_bits_to_f64(y[3]) == 0).all()


def test_stream_deterministic():
    N, K = 4096, 11008
    qw, W = layer(N, K, 4, 128, 4)
    for M in (1, 3):
        x = to_dev_bf16(synth.make_activations(M, K, 4))
        a = to_host_bits(tf.gemv(W, x))
        for _ in range(3):
            np.testing.assert_array_equal(a, to_host_bits(tf.gemv(W, x)))


@pytest.mark.parametrize("M", [1, 5])
def test_stream_bias(M):
    import torch
    N, K = 3000, 1536
    qw, W = layer(N, K, 4, 128, 41)
    rng = np.random.default_rng(41)
    b = synth.f32_to_bf16_bits((rng.standard_normal(N) * 0.5).astype(np.float32))
    xb = synth.make_activations(M, K, 41)
    y = to_host_bits(tf.gemv(W, to_dev_bf16(xb), bias=to_dev_bf16(b)))
    ref = tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, 4, 128, K, xb) + tf_oracle.bf16_bits_to_f64(b)[None]
    check_close(y, ref, f"stream gemv bias M={M}")
    torch.cuda.synchronize()


def test_stream_rejects_mismatched_header():
    """Blobs of 4096 x 11008 and 11008 x 4096 have the same size (22016
    units); a call that describes one and passes the other is caught on the
    device: the error word holds 0x800 and y is left untouched."""
    import torch
    qa, Wa = layer(4096, 11008, 4, 128, 43)
    qb, Wb = layer(11008, 4096, 4, 128, 44)
    assert Wa.nbytes == Wb.nbytes
    assert tf.device_error() == 0
    wrong = tf.Weights(Wb.blob, 4096, 11008, 4, 128)   # 11008 x 4096 blob described as 4096 x 11008
    x = to_dev_bf16(synth.make_activations(1, 11008, 43))
    y = torch.full((1, 4096), 7.0, dtype=torch.bfloat16, device="cuda")
    tf.gemv(wrong, x, y)
    torch.cuda.synchronize()
    assert tf.device_error() == 0x800
    assert bool((y == 7.0).all())
    # the library is still usable after a rejected call
    y2 = to_host_bits(tf.gemv(Wa, x))
    check_close(y2, tf_oracle.reference(qa.qweight, qa.scales, qa.zeros, 4, 128, 11008,
                                        to_host_bits(x)), "after a rejected call")
