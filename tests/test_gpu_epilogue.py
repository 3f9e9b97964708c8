"""The fused epilogues (tf_gemv_silu_gate / tf_gemm_silu_gate, tf_gemv_qkv /
tf_gemm_qkv) against the float64 oracle.

The gate/up reference is computed from the two projections separately
(oracle layer outputs of each, plus their biases, then silu(g) * u), so the
pre-tiling's interleaving and the kernels' pairing of a gate row with its up
row are both checked end to end.  The shapes reach every kernel and store
site: the stream GEMV (full and compact parking of sums), the tile GEMV
(whole row blocks and the split-K last arriver), the slab GEMV (groups of
32), the GEMM's whole-tile element stores and its stream-K fixup.
"""

import numpy as np
import pytest

import gemv_tf_prepack_gb300 as tf
from gemv_tf_prepack_gb300 import synth
from oracle import epilogue as E
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


def _bias_bits(n, seed):
    b = np.random.default_rng([seed, n]).standard_normal(n) * 0.5
    return tf_oracle.bf16_value_to_bits(tf_oracle.bf16_round(b))


def _ref(qw, K, xb):
    return tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, qw.bits, qw.group, K, xb)


# (F, K, bits, group, M, kind): N = 2F rows
GATE_CASES = [
    (1224, 1024, 4, 128, 1, "gemv"), (1224, 2048, 8, 0, 3, "gemv"), (1536, 1024, 4, 64, 8, "gemv"),
    (2056, 8192, 4, 128, 8, "gemv"),   # M = 8 on a long K: half-size ring stages
    (4096, 1024, 4, 128, 1, "gemv"),   # 512 slabs: compact parking of the sums
    (96, 1024, 4, 128, 1, "gemv"),     # stream GEMV, one CTA per slab
    (96, 896, 4, 32, 1, "gemv"), (96, 768, 8, 32, 5, "gemv"),  # tile GEMV (K < 1024): split-K last arriver
    (1224, 1024, 4, 32, 2, "gemv"),    # slab GEMV (groups of 32)
    (1024, 1024, 4, 128, 37, "gemm"), (1024, 2048, 8, 64, 300, "gemm"), (200, 1024, 4, 0, 1, "gemm"),
]


@pytest.mark.parametrize("F,K,bits,group,M,kind", GATE_CASES)
@pytest.mark.parametrize("with_bias", [False, True])
def test_silu_gate(F, K, bits, group, M, kind, with_bias):
    import torch
    g = synth.make_weights(F, K, bits, group, 71)
    u = synth.make_weights(F, K, bits, group, 72)
    blob = tf.prepack_gate_up((g.qweight, g.scales, g.zeros), (u.qweight, u.scales, u.zeros), F, K, bits, group)
    W = tf.Weights.upload(blob)
    xb = synth.make_activations(M, K, 73, outliers=kind == "gemm")
    yg, yu = _ref(g, K, xb), _ref(u, K, xb)
    bias = None
    if with_bias:
        bg, bu = _bias_bits(F, 74), _bias_bits(F, 75)
        yg = yg + tf_oracle.bf16_bits_to_f64(bg)[None, :]
        yu = yu + tf_oracle.bf16_bits_to_f64(bu)[None, :]
        bias = to_dev_bf16(E.interleave_gate_up(bg, bu))
    ref = E.silu(yg) * yu
    x = to_dev_bf16(xb)
    call = tf.gemv_silu_gate if kind == "gemv" else tf.gemm_silu_gate
    h = to_host_bits(call(W, x, bias=bias))
    check_close(h, ref, f"{kind} silu gate F={F} K={K} w{bits} g{group} M={M} bias={with_bias}")
    # same sums as the plain call: h from the plain output, silu in float64
    y = tf_oracle.bf16_bits_to_f64(to_host_bits((tf.gemv if kind == "gemv" else tf.gemm)(W, x, bias=bias)))
    check_close(h, E.silu_gate(y), f"{kind} silu gate vs plain output")
    if kind == "gemm":  # every tile whole (no workspace)
        h2 = to_host_bits(tf.gemm_silu_gate(W, x, bias=bias, stream_k=False))
        check_close(h2, ref, f"gemm silu gate whole tiles F={F} M={M}")
    torch.cuda.synchronize()
    assert tf.device_error() == 0


def test_silu_gate_deterministic_and_output_only():
    """h is written exactly, run after run, and nothing outside [M, N/2]."""
    import torch
    F, K = 1224, 1024
    g = synth.make_weights(F, K, 4, 128, 81)
    blob = tf.prepack_gate_up((g.qweight, g.scales, g.zeros), (g.qweight, g.scales, g.zeros), F, K, 4, 128)
    W = tf.Weights.upload(blob)
    for M, fn in ((1, tf.gemv_silu_gate), (8, tf.gemv_silu_gate), (40, tf.gemm_silu_gate)):
        x = to_dev_bf16(synth.make_activations(M, K, 82))
        buf = torch.full((M * F + 64,), 7.0, dtype=torch.bfloat16, device="cuda")
        h = buf[:M * F].view(M, F)
        fn(W, x, h=h)
        a = to_host_bits(h.clone())
        fn(W, x, h=h)
        np.testing.assert_array_equal(a, to_host_bits(h))
        assert bool((buf[M * F:] == 7.0).all())
    torch.cuda.synchronize()


# (N, K, bits, group, M, kind, nq, nk)
QKV_CASES = [
    (2440, 1024, 4, 128, 1, "gemv", 1000, 720), (3072, 2048, 8, 0, 4, "gemv", 2048, 512),
    (4104, 8192, 4, 64, 8, "gemv", 4096, 0), (384, 1024, 4, 128, 2, "gemv", 128, 128),
    (384, 896, 4, 32, 2, "gemv", 128, 128),  # tile GEMV (K < 1024)
    (2440, 1024, 4, 32, 1, "gemv", 2, 2000), (1536, 2048, 4, 128, 33, "gemm", 1024, 257),
    (3000, 1024, 8, 128, 300, "gemm", 1500, 500), (1004, 1016, 4, 0, 17, "gemm", 1, 1),
]


@pytest.mark.parametrize("N,K,bits,group,M,kind,nq,nk", QKV_CASES)
@pytest.mark.parametrize("with_bias", [False, True])
def test_qkv_split(N, K, bits, group, M, kind, nq, nk, with_bias):
    import torch
    qw, W = layer(N, K, bits, group, 91)
    xb = synth.make_activations(M, K, 92, outliers=kind == "gemm")
    ref = _ref(qw, K, xb)
    bias = None
    if with_bias:
        bb = _bias_bits(N, 93)
        ref = ref + tf_oracle.bf16_bits_to_f64(bb)[None, :]
        bias = to_dev_bf16(bb)
    x = to_dev_bf16(xb)
    call = tf.gemv_qkv if kind == "gemv" else tf.gemm_qkv
    outs = call(W, x, nq, nk, bias=bias)
    plain = to_host_bits((tf.gemv if kind == "gemv" else tf.gemm)(W, x, bias=bias))
    for name, got, r, p in zip("qkv", outs, E.split_qkv(ref, nq, nk), E.split_qkv(plain, nq, nk)):
        got = to_host_bits(got)
        if r.shape[1]:
            check_close(got, r, f"{kind} qkv {name} N={N} M={M}")
        # the split changes where each value goes, not its bits
        np.testing.assert_array_equal(got, p)
    if kind == "gemm":  # every tile whole (no workspace)
        outs2 = tf.gemm_qkv(W, x, nq, nk, bias=bias, stream_k=False)
        np.testing.assert_array_equal(np.concatenate([to_host_bits(t) for t in outs2], axis=1),
                                      to_host_bits(tf.gemm(W, x, bias=bias, stream_k=False)))
    torch.cuda.synchronize()
    assert tf.device_error() == 0
