"""Parity of the CUDA path (through the C ABI) with the float64 CPU oracle.

* tf_dequant: BF16 bits identical to the oracle's dequant for every format
  (this pins the pre-tiling permutation, unpack and dequant together; the
  GEMV and GEMM kernels share the same device dequant code).
* tf_gemv / tf_gemm: relative Frobenius error <= 5e-3 and worst element
  <= 1e-2 * max|ref| against the oracle on identical seeded inputs, at sizes
  spanning several tiles with ragged edges, and at the full workload sizes
  (all outputs, or sampled output rows where the oracle would be too slow).
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


FORMATS = [
    (256, 512, 4, 128), (200, 192, 4, 64), (136, 200, 8, 0), (64, 96, 4, 32),
    (130, 256, 8, 128), (8, 8, 4, 0), (128, 1024, 4, 256), (300, 384, 8, 64), (72, 96, 8, 32),
    (1000, 1016, 4, 0), (384, 4096, 4, 128),
    (1, 8, 4, 0), (3, 256, 8, 64),  # a single output row; three rows of one partial slab
]


@pytest.mark.parametrize("N,K,bits,group", FORMATS)
def test_dequant_bit_exact(N, K, bits, group):
    qw, W = layer(N, K, bits, group, 13)
    got = to_host_bits(tf.dequant(W))
    q = tf_oracle.unpack(qw.qweight, bits, K)
    want = tf_oracle.dequant_bits(q, qw.scales, qw.zeros, group)
    mism = np.argwhere(got != want)
    assert mism.size == 0, f"{len(mism)} mismatches, first at {mism[:3].tolist()}"


@pytest.mark.parametrize("N,K,bits,group", FORMATS)
@pytest.mark.parametrize("M", [1, 3, 8])
def test_gemv_small(N, K, bits, group, M):
    qw, W = layer(N, K, bits, group, 21)
    xb = synth.make_activations(M, K, 21)
    y = to_host_bits(tf.gemv(W, to_dev_bf16(xb)))
    ref = tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, bits, group, K, xb)
    check_close(y, ref, f"gemv {N}x{K} w{bits} g{group} M={M}")


# Groups of 64, multiples of 128 and per channel take the stream GEMV; groups
# of 32 with K >= 1024 the slab GEMV (whole slabs per CTA, one CTA per slab on
# layers with fewer slabs than SMs, no workspace).
SLAB_FORMATS = [
    (2440, 1016, 4, 0), (2440, 1152, 4, 128), (4104, 2048, 4, 32), (2432, 4096, 4, 64),
    (3000, 2048, 8, 0), (2560, 1280, 8, 64), (2448, 1024, 8, 32), (5000, 3072, 4, 128),
    (1024, 2048, 4, 32), (520, 1152, 8, 32), (16, 4096, 4, 32),  # fewer slabs than SMs
]


@pytest.mark.parametrize("N,K,bits,group", SLAB_FORMATS)
@pytest.mark.parametrize("M", [1, 3, 8])
def test_gemv_slab(N, K, bits, group, M):
    assert -(-K // 128) >= 8, "shape meant for the slab GEMV"
    if not (M == 8 and bits == 4 and group == 32):  # those stages do not fit twice per SM: tile GEMV
        assert tf.gemv_workspace_size(N, K, bits, group, M) == 0
    qw, W = layer(N, K, bits, group, 23)
    xb = synth.make_activations(M, K, 23)
    y = to_host_bits(tf.gemv(W, to_dev_bf16(xb)))
    ref = tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, bits, group, K, xb)
    check_close(y, ref, f"slab gemv {N}x{K} w{bits} g{group} M={M}")


def test_gemv_slab_deterministic():
    N, K = 4096, 11008
    qw, W = layer(N, K, 4, 128, 4)
    x = to_dev_bf16(synth.make_activations(1, K, 4))
    a = to_host_bits(tf.gemv(W, x))
    for _ in range(3):
        np.testing.assert_array_equal(a, to_host_bits(tf.gemv(W, x)))


def test_gemv_deterministic_and_workspace_reusable():
    """Tile GEMV with K split over many CTAs (eight tokens at K = 32768: x too
    large to stay resident)."""
    N, K = 1024, 32768
    qw, W = layer(N, K, 4, 128, 4)
    xb = synth.make_activations(8, K, 4)
    x = to_dev_bf16(xb)
    assert tf.gemv_workspace_size(N, K, 4, 128, 8) > 0
    a = to_host_bits(tf.gemv(W, x))
    check_close(a, tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, 4, 128, K, xb), "tile gemv")
    for _ in range(3):
        b = to_host_bits(tf.gemv(W, x))
        np.testing.assert_array_equal(a, b)
    # the counters (first 16 KB of the workspace) are handed back at zero
    ws = W.workspace(8)
    import torch
    assert ws.numel() > 16384
    assert int(ws[:16384].view(torch.int32).abs().sum()) == 0


@pytest.mark.parametrize("N,K,bits,group", FORMATS)
@pytest.mark.parametrize("M", [1, 9, 16, 37, 64])
def test_gemm_small(N, K, bits, group, M):
    """tf_gemm with its workspace (M <= 8 on these layers: the slab or tile GEMV;
    above: the tensor-memory pipeline with K-split tiles) and without one
    (every tile whole in the tensor-memory pipeline), both against the
    oracle."""
    qw, W = layer(N, K, bits, group, 31)
    xb = synth.make_activations(M, K, 31, outliers=True)
    x = to_dev_bf16(xb)
    ref = tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, bits, group, K, xb)
    check_close(to_host_bits(tf.gemm(W, x)), ref, f"gemm {N}x{K} w{bits} g{group} M={M}")
    check_close(to_host_bits(tf.gemm(W, x, stream_k=False)), ref, f"tcgen05 gemm {N}x{K} w{bits} g{group} M={M}")


@pytest.mark.parametrize("N,K,bits,group,M", [(3000, 4096, 4, 128, 40), (1000, 8192, 8, 0, 64), (2440, 1536, 4, 64, 9),
                                              (1024, 768, 4, 128, 4)])
def test_gemm_few_tokens_deterministic(N, K, bits, group, M):
    """Few tokens: K is split across CTAs (tensor-memory stream-K, or the tile
    GEMV at M <= 8 with K < 1024) and the partial sums are added in a fixed order: the same
    bits every run."""
    qw, W = layer(N, K, bits, group, 36)
    xb = synth.make_activations(M, K, 36)
    x = to_dev_bf16(xb)
    assert tf.gemm_workspace_size(N, K, bits, group, M) > 0
    a = to_host_bits(tf.gemm(W, x))
    check_close(a, tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, bits, group, K, xb), f"gemm M={M}")
    for _ in range(2):
        np.testing.assert_array_equal(a, to_host_bits(tf.gemm(W, x)))


def test_gemm_few_tokens_on_the_slab_gemv():
    """M <= 8 on a layer with a 16-row slab per SM: tf_gemm runs the slab GEMV
    (per-weight BF16 rounding, no workspace), with or without a workspace."""
    N, K, M = 4096, 2048, 8
    qw, W = layer(N, K, 4, 128, 37)
    assert tf.gemm_workspace_size(N, K, 4, 128, M) == 0
    xb = synth.make_activations(M, K, 37)
    x = to_dev_bf16(xb)
    ref = tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, 4, 128, K, xb)
    a = to_host_bits(tf.gemm(W, x))
    check_close(a, ref, "gemm M=8 slab GEMV")
    np.testing.assert_array_equal(a, to_host_bits(tf.gemm(W, x, stream_k=False)))


def test_one_workspace_serves_every_layer():
    """Split-K workspaces keep their arrival counters in a fixed region at the
    start, so one zeroed workspace, as large as the largest need, can serve
    layers of any shape in turn: tile GEMV calls (through tf_gemv and
    tf_gemm) and tensor-memory stream-K calls alternate on it and give the
    bits of private workspaces."""
    import torch
    calls = [(tf.gemv, (1024, 768, 4, 32), 1), (tf.gemm, (2048, 768, 8, 0), 4),
             (tf.gemm, (20480, 384, 4, 128), 80), (tf.gemv, (640, 896, 8, 32), 5), (tf.gemm, (1000, 8192, 4, 64), 64)]
    sizes = [(tf.gemv_workspace_size if fn is tf.gemv else tf.gemm_workspace_size)(*shape, M) for fn, shape, M in calls]
    assert all(n > 0 for n in sizes)
    shared = torch.zeros(max(sizes), dtype=torch.uint8, device="cuda")
    layers, want = [], []
    for i, (fn, shape, M) in enumerate(calls):
        _, W = layer(*shape, 40 + i)
        x = to_dev_bf16(synth.make_activations(M, shape[1], 40 + i))
        layers.append((fn, W, x))
        want.append(to_host_bits(fn(W, x)))  # its own cached workspace
    for _ in range(3):
        for (fn, W, x), w in zip(layers, want):
            np.testing.assert_array_equal(to_host_bits(fn(W, x, workspace=shared)), w)
    torch.cuda.synchronize()
    assert int(shared[:16384].view(torch.int32).abs().sum()) == 0, "arrival counters left non-zero"


@pytest.mark.parametrize("M", [128, 200, 256, 300, 640])
def test_gemm_token_tiles(M):
    N, K = 384, 1024
    qw, W = layer(N, K, 4, 128, 33)
    xb = synth.make_activations(M, K, 33, outliers=True)
    y = to_host_bits(tf.gemm(W, to_dev_bf16(xb)))
    ref = tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, 4, 128, K, xb)
    check_close(y, ref, f"gemm M={M}")


def test_gemm_deterministic():
    N, K, M = 1024, 2048, 300
    qw, W = layer(N, K, 4, 64, 35)
    x = to_dev_bf16(synth.make_activations(M, K, 35))
    a = to_host_bits(tf.gemm(W, x))
    b = to_host_bits(tf.gemm(W, x))
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("N,K,bits,group", [(512, 1024, 4, 128), (256, 768, 8, 0), (384 + 128, 640, 4, 64),
                                            (1000, 1016, 4, 0), (256, 512, 4, 32)])
@pytest.mark.parametrize("M", [256, 300, 640, 1000])
def test_gemm_even_blocks(N, K, bits, group, M):
    """Even numbers of 128-row blocks with several ragged 256-token tiles."""
    qw, W = layer(N, K, bits, group, 37)
    xb = synth.make_activations(M, K, 37, outliers=True)
    y = to_host_bits(tf.gemm(W, to_dev_bf16(xb)))
    ref = tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, bits, group, K, xb)
    check_close(y, ref, f"gemm {N}x{K} w{bits} g{group} M={M}")


# Long K: x no longer fits next to a ring at two CTAs per SM, so the slab GEMV
# runs sixteen warps per CTA with x resident (the first three and the last
# two, those with a ring of only two stages); where x does not fit even then
# (M = 8 at K = 16384) the tile GEMV takes the layer.  Sampled output rows:
# the oracle row by row.
LONG_K = [
    (2440, 24576, 4, 32, 1), (2432, 16384, 8, 64, 2), (2432, 32768, 4, 128, 1), (2440, 16384, 4, 128, 8),
    # 128 KB of resident x next to a two-stage ring
    (2440, 8192, 8, 0, 8), (2440, 16384, 4, 128, 4),
]


@pytest.mark.parametrize("N,K,bits,group,M", LONG_K)
def test_gemv_slab_long_k(N, K, bits, group, M):
    qw, W = layer(N, K, bits, group, 27)
    xb = synth.make_activations(M, K, 27)
    y = to_host_bits(tf.gemv(W, to_dev_bf16(xb)))
    rows = np.unique(np.concatenate([np.arange(0, 40), np.arange(N - 40, N),
                                     np.random.default_rng(0).integers(0, N, 64)]))
    ref = tf_oracle.reference_rows(qw.qweight, qw.scales, qw.zeros, bits, group, K, xb, rows)
    check_close(y[:, rows], ref, f"long-K slab gemv {N}x{K} w{bits} g{group} M={M}")


# Shapes whose tiles the tensor-memory GEMM splits along K on a 152-SM GB300
# (M > 8, or per-channel layers with K % 8 != 0, which the GEMV kernels do
# not take): a partial wave over more than one wave of tiles (N = 20480 and
# 19712 rows, a ragged N = 20000 with K % 8 != 0), and every tile split when
# there are few tiles (M = 100 over 3 tiles; M = 1 over 2 tiles of 33
# k-iterations, four CTAs adding into each).
STREAM_K = [
    (20480, 384, 4, 128, 80), (19712, 2048, 4, 128, 300), (20000, 1017, 4, 0, 40),
    (384, 8192, 8, 64, 100), (256, 4097, 8, 0, 1), (2048, 1536, 4, 128, 512),
]


@pytest.mark.parametrize("N,K,bits,group,M", STREAM_K)
def test_gemm_stream_k_and_whole_tiles(N, K, bits, group, M):
    """Both GEMM schedules against the oracle: output tiles split along K across
    SMs (partial sums added in a fixed order), and every tile whole on one SM."""
    import torch
    qw, W = layer(N, K, bits, group, 39)
    if torch.cuda.get_device_properties(0).multi_processor_count == 152 and (N, M) != (2048, 512):
        assert tf.gemm_workspace_size(N, K, bits, group, M) > 0, "expected a K-split schedule"
    xb = synth.make_activations(M, K, 39, outliers=True)
    x = to_dev_bf16(xb)
    ref = tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, bits, group, K, xb)
    y_sk = to_host_bits(tf.gemm(W, x))
    check_close(y_sk, ref, f"stream-K gemm {N}x{K} M={M}")
    if K % 8 == 0:  # else the padded copy of x needs the workspace (whole tiles are not available)
        y_dp = to_host_bits(tf.gemm(W, x, stream_k=False))
        check_close(y_dp, ref, f"whole-tile gemm {N}x{K} M={M}")
    np.testing.assert_array_equal(y_sk, to_host_bits(tf.gemm(W, x)))  # same sums every run
    assert tf.device_error() == 0


def _random_layers(n, seed):
    """Seeded random layer shapes: INT4/INT8, every group kind, ragged N and K, M from 1 to ~700."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        bits = int(rng.choice([4, 8]))
        group = int(rng.choice([0, 32, 64, 128, 256]))
        if group == 0:
            K = int(rng.integers(1, 600)) * 8
        elif group == 256:
            K = int(rng.integers(1, 20)) * 256
        else:
            K = int(rng.integers(1, 40)) * group
        N = int(rng.integers(1, 6000))
        if N * K > 12_000_000:
            N = max(1, 12_000_000 // K)
        M = int(rng.choice([int(rng.integers(1, 9)), int(rng.integers(9, 80)), int(rng.integers(80, 700))]))
        out.append((N, K, bits, group, M))
    return out


@pytest.mark.parametrize("N,K,bits,group,M", _random_layers(16, 2027))
def test_random_layers(N, K, bits, group, M):
    """GEMM (whole tiles or stream-K, TMA or element stores) and, at M <= 8, GEMV on random shapes."""
    qw, W = layer(N, K, bits, group, 43)
    xb = synth.make_activations(M, K, 43, outliers=True)
    x = to_dev_bf16(xb)
    ref = tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, bits, group, K, xb)
    y = to_host_bits(tf.gemm(W, x))
    check_close(y, ref, f"gemm {N}x{K} w{bits} g{group} M={M}")
    np.testing.assert_array_equal(y, to_host_bits(tf.gemm(W, x)))
    if M <= 8:
        check_close(to_host_bits(tf.gemv(W, x)), ref, f"gemv {N}x{K} w{bits} g{group} M={M}")
    assert tf.device_error() == 0


# AWQ checkpoints imported with tf_prepack_awq: the device dequantises exactly
# what the oracle decodes from the AWQ arrays, and both kernels match it.
@pytest.mark.parametrize("N,K,group", [(1032, 1024, 128), (4096, 4096, 128), (2440, 1536, 64), (512, 768, 0)])
def test_awq_import_parity(N, K, group):
    from oracle import awq
    qw = synth.make_weights(N, K, 4, group, 31)
    q = tf_oracle.unpack(qw.qweight, 4, K)
    s16 = (np.random.default_rng([31, 7]).random(qw.scales.shape) * 0.01 + 0.001).astype(np.float16)
    qweight, qzeros, scales = awq.awq_encode(q, qw.zeros, s16)
    W = tf.Weights.upload(tf.prepack_awq(qweight, qzeros, scales, N, K, group))
    qd, sd, zd = awq.awq_decode(qweight, qzeros, scales, N, K, group)
    np.testing.assert_array_equal(to_host_bits(tf.dequant(W)), tf_oracle.dequant_bits(qd, sd, zd, group))
    wd = tf_oracle.dequant(qd, sd, zd, group)
    for M, fn in ((1, tf.gemv), (8, tf.gemv), (64, tf.gemm)):
        xb = synth.make_activations(M, K, 31)
        y = to_host_bits(fn(W, to_dev_bf16(xb)))
        check_close(y, tf_oracle.linear_f64(xb, wd), f"awq {fn.__name__} {N}x{K} g{group} M={M}")


# Bias in the epilogue (tf_gemv_bias / tf_gemm_bias): y = bf16_rne(x W^T + bias).
# The shapes reach every place y is written: slab GEMV, tile GEMV (whole row
# blocks and the split-K last arriver), GEMM TMA-staged whole tiles, GEMM
# element stores (N % 8 != 0) and the GEMM stream-K fixup.
BIAS_CASES = [
    (2440, 1152, 4, 128, 1, "gemv"), (2440, 1152, 8, 0, 3, "gemv"), (200, 192, 4, 64, 8, "gemv"),
    (1000, 1016, 4, 0, 1, "gemv"), (200, 192, 4, 32, 8, "gemv"),  # the last one: tile GEMV
    (384, 4096, 8, 64, 37, "gemm"), (20000, 1016, 4, 0, 40, "gemm"),
    (2048, 1536, 4, 128, 512, "gemm"), (1004, 1016, 4, 0, 300, "gemm"),
]


@pytest.mark.parametrize("N,K,bits,group,M,fn", BIAS_CASES)
def test_bias_epilogue(N, K, bits, group, M, fn):
    import torch
    qw, W = layer(N, K, bits, group, 47)
    xb = synth.make_activations(M, K, 47, outliers=fn == "gemm")
    b16 = (np.random.default_rng([47, N]).standard_normal(N) * 0.5).astype(np.float32)
    bias_bits = tf_oracle.bf16_value_to_bits(tf_oracle.bf16_round(b16.astype(np.float64)))
    bias = to_dev_bf16(bias_bits)
    ref = tf_oracle.reference(qw.qweight, qw.scales, qw.zeros, bits, group, K, xb) \
        + tf_oracle.bf16_bits_to_f64(bias_bits)[None, :]
    call = tf.gemv if fn == "gemv" else tf.gemm
    y = to_host_bits(call(W, to_dev_bf16(xb), bias=bias))
    check_close(y, ref, f"{fn}+bias {N}x{K} w{bits} g{group} M={M}")
    if fn == "gemm":  # every tile whole (no workspace): the other schedule's epilogue
        y2 = to_host_bits(tf.gemm(W, to_dev_bf16(xb), bias=bias, stream_k=False))
        check_close(y2, ref, f"gemm+bias whole tiles {N}x{K} M={M}")
    with pytest.raises(ValueError):
        call(W, to_dev_bf16(xb), bias=bias[:-1])
    torch.cuda.synchronize()


# Symmetric quantisation (no zero-point tensor in the checkpoint) is the
# constant zero point 2^(bits-1): w = (q - 8) * s for INT4, (q - 128) * s for INT8.
@pytest.mark.parametrize("N,K,bits,group", [(2440, 1024, 4, 128), (512, 768, 8, 64), (300, 256, 4, 32)])
def test_symmetric_zero_point(N, K, bits, group):
    qw = synth.make_weights(N, K, bits, group, 53)
    zeros = np.full_like(qw.zeros, 1 << (bits - 1))
    W = tf.Weights.upload(tf.prepack(qw.qweight, qw.scales, zeros, N, K, bits, group))
    q = tf_oracle.unpack(qw.qweight, bits, K)
    np.testing.assert_array_equal(to_host_bits(tf.dequant(W)), tf_oracle.dequant_bits(q, qw.scales, zeros, group))
    for M, fn in ((1, tf.gemv), (24, tf.gemm)):
        xb = synth.make_activations(M, K, 53)
        ref = tf_oracle.reference(qw.qweight, qw.scales, zeros, bits, group, K, xb)
        check_close(to_host_bits(fn(W, to_dev_bf16(xb))), ref, f"symmetric {fn.__name__} {N}x{K} w{bits} M={M}")


# (call, described layer (N, K, bits, group), the other layer's shape, M): both
# layers have the same number of units, so the blob sizes agree and only the
# header can tell them apart.
HEADER_CASES = [
    ("gemv", (1024, 2048, 4, 128), (2048, 1024), 1),   # stream GEMV, one CTA per slab
    ("gemv", (1024, 768, 4, 32), (768, 1024), 1),      # tile GEMV (K < 1024)
    ("gemv", (4096, 2048, 4, 32), (2048, 4096), 1),    # slab GEMV (groups of 32)
    ("gemm", (4096, 11008, 4, 128), (11008, 4096), 64),
    ("gemm", (4096, 11008, 4, 128), (11008, 4096), 300),
    ("gemm_whole", (4096, 11008, 4, 128), (11008, 4096), 300),
    ("dequant", (1024, 2048, 4, 128), (2048, 1024), 0),
]


@pytest.mark.parametrize("call,desc,other,M", HEADER_CASES, ids=[f"{c[0]}-{c[1][0]}x{c[1][1]}g{c[1][3]}-M{c[3]}" for c in HEADER_CASES])
def test_mismatched_header_rejected_on_device(call, desc, other, M):
    """A device blob of another layer with the same size: the kernel reads its
    header, records 0x800 in the device error word and writes nothing (y and
    the stream-K workspace stay as they were)."""
    import torch
    N, K, bits, group = desc
    _, Wo = layer(other[0], other[1], bits, group, 51)
    assert Wo.nbytes == tf.prepack_size(N, K, bits, group)
    wrong = tf.Weights(Wo.blob, N, K, bits, group)
    assert tf.device_error() == 0
    if call == "dequant":
        out = torch.full((N, K), 3.0, dtype=torch.bfloat16, device="cuda")
        tf.dequant(wrong, out=out)
    else:
        x = to_dev_bf16(synth.make_activations(M, K, 51))
        out = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
        if call == "gemv":
            tf.gemv(wrong, x, out)
        else:
            tf.gemm(wrong, x, out, stream_k=(call == "gemm"))
    torch.cuda.synchronize()
    assert tf.device_error() == 0x800
    assert bool((out == 3.0).all()), "a mismatched blob must not be written through"
    if call == "gemm":
        ws = wrong.workspace(M, "gemm")
        assert int(ws.view(torch.uint8).sum()) == 0
