"""AWQ checkpoint import: the oracle's decoder pinned to the layout's definition,
the FP16 -> BF16 scale rounding pinned to hand-derived values, and the C
``tf_prepack_awq`` checked against both (host only, no GPU).
"""

import numpy as np
import pytest

import gemv_tf_prepack_gb300 as tf
from gemv_tf_prepack_gb300 import synth
from oracle import awq, layout, tf_oracle


def _natural_qweight(q: np.ndarray) -> np.ndarray:
    """Codes [N, K] -> natural INT4 words [N, K/8], low nibble first along K."""
    N, K = q.shape
    w = np.zeros((N, K // 8), dtype=np.uint32)
    for i in range(8):
        w |= q[:, i::8].astype(np.uint32) << np.uint32(4 * i)
    return w


def _awq_layer(N, K, group, seed):
    """Synthetic AWQ arrays: codes and zeros from the seeded generator, FP16 scales
    with a full 11-bit significand (so that the BF16 rounding matters)."""
    qw = synth.make_weights(N, K, 4, group, seed)
    q = tf_oracle.unpack(qw.qweight, 4, K)
    rng = np.random.default_rng([seed, 7])
    s16 = (rng.random(qw.scales.shape) * 0.01 + 0.001).astype(np.float16)
    return awq.awq_encode(q, qw.zeros, s16), (q, qw.zeros, s16)


# --- the oracle decoder --------------------------------------------------------

def test_awq_nibble_order_golden():
    # By the definition nibble i holds output column AWQ_ORDER[i] = (0,2,4,6,1,3,5,7)[i].
    # The word 0x76543210 stores the value i in nibble i, so column j receives the i
    # with AWQ_ORDER[i] = j: columns 0..7 read 0, 4, 1, 5, 2, 6, 3, 7 (worked by hand).
    N, K, g = 8, 128, 128
    qweight = np.zeros((K, N // 8), dtype=np.uint32)
    qweight[5, 0] = 0x76543210
    qzeros = np.zeros((1, 1), dtype=np.uint32)
    qzeros[0, 0] = 0xFEDCBA98  # nibble i holds 8 + i
    s16 = np.full((1, N), np.float16(1.0)).view(np.uint16)
    q, s, z = awq.awq_decode(qweight.view(np.int32), qzeros.view(np.int32), s16, N, K, g)
    assert q[:, 5].tolist() == [0, 4, 1, 5, 2, 6, 3, 7]
    assert z[:, 0].tolist() == [8, 12, 9, 13, 10, 14, 11, 15]
    assert np.count_nonzero(q) == 7
    assert (s == 0x3F80).all()


# (FP16 bits, BF16 bits), each worked by hand: BF16 keeps 8 significant bits.
F16_TO_BF16 = [
    (0x3C00, 0x3F80),  # 1.0
    (0x3C01, 0x3F80),  # 1 + 2^-10: below half a BF16 ulp (2^-8) -> 1.0
    (0x3C04, 0x3F80),  # 1 + 2^-8: exactly half an ulp, tie to the even 1.0
    (0x3C05, 0x3F81),  # 1 + 5*2^-10: above half -> 1 + 2^-7
    (0x3C0C, 0x3F82),  # 1 + 3*2^-8: tie between 1 + 2^-7 (odd) and 1 + 2^-6 (even)
    (0xC000, 0xC000),  # -2.0
    (0x0001, 0x3380),  # 2^-24, the smallest FP16 subnormal, exact in BF16
    (0x03FF, 0x3880),  # (1 - 2^-10) * 2^-14 rounds up to 2^-14
    (0x0400, 0x3880),  # 2^-14, the smallest FP16 normal
    (0x7BFF, 0x4780),  # 65504 = (2 - 2^-10) * 2^15 rounds up to 2^16
    (0x7C00, 0x7F80),  # +inf
    (0xFC00, 0xFF80),  # -inf
    (0x8000, 0x8000),  # -0.0
]


def test_oracle_f16_to_bf16_pins():
    for h, b in F16_TO_BF16:
        assert int(awq.f16_bits_to_bf16_bits(np.array([h], dtype=np.uint16))[0]) == b, hex(h)


@pytest.mark.parametrize("group", [128, 64, 32, 0])
def test_awq_encode_decode_round_trip(group):
    (qweight, qzeros, s16), (q, z, s_f16) = _awq_layer(48, 256, group, 3)
    g = 256 if group == 0 else group
    assert qweight.shape == (256, 6) and qweight.dtype == np.int32
    assert qzeros.shape == (256 // g, 6) and s16.shape == (256 // g, 48)
    q2, s2, z2 = awq.awq_decode(qweight, qzeros, s16, 48, 256, group)
    assert np.array_equal(q2, q) and np.array_equal(z2, z)
    want_s = tf_oracle.bf16_value_to_bits(tf_oracle.bf16_round(s_f16.astype(np.float64)))
    assert np.array_equal(s2, want_s)


# --- the C import against the oracle --------------------------------------------

def _c_scales(s16_flat: np.ndarray, N: int, K: int, group: int) -> np.ndarray:
    """BF16 scales [N, K/g] that tf_prepack_awq stores for FP16 scales [K/g, N]."""
    g = K if group == 0 else group
    qweight = np.zeros((K, N // 8), dtype=np.int32)
    qzeros = np.zeros((K // g, N // 8), dtype=np.int32)
    blob = tf.prepack_awq(qweight, qzeros, s16_flat.reshape(K // g, N), N, K, group)
    _, scales, _, *_ = tf.unprepack(blob)
    return scales


def test_c_f16_to_bf16_pins():
    hs = np.array([h for h, _ in F16_TO_BF16] * 2, dtype=np.uint16)[:16]
    got = _c_scales(hs, 16, 128, 0)[:, 0]
    want = np.array([b for _, b in F16_TO_BF16] * 2, dtype=np.uint16)[:16]
    assert got.tolist() == want.tolist()


def test_c_f16_to_bf16_exhaustive():
    # every FP16 bit pattern as one scale of a 256 x 8192 g32 layer (256 groups x 256 rows)
    allh = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = _c_scales(allh, 256, 8192, 32).T.reshape(-1)
    nan = np.isnan(allh.view(np.float16))
    want = awq.f16_bits_to_bf16_bits(np.where(nan, 0, allh).astype(np.uint16))
    assert np.array_equal(got[~nan], want[~nan])
    got_f = tf_oracle.bf16_bits_to_f64(got[nan])
    assert np.isnan(got_f).all() and nan.sum() == 2046


@pytest.mark.parametrize("N,K,group", [(264, 512, 128), (48, 384, 64), (8, 96, 32), (136, 200, 0),
                                       (1032, 1024, 128), (72, 640, 128), (64, 1024, 256), (40, 768, 384)])
def test_awq_blob_equals_natural_blob(N, K, group):
    (qweight, qzeros, s16), _ = _awq_layer(N, K, group, 11)
    blob = tf.prepack_awq(qweight, qzeros, s16, N, K, group)
    q, s, z = awq.awq_decode(qweight, qzeros, s16, N, K, group)
    natural = _natural_qweight(q)
    assert np.array_equal(blob, tf.prepack(natural, s, z, N, K, 4, group))
    assert np.array_equal(blob, layout.prepack(natural, s, z, N, K, 4, group))


def test_awq_golden_word_through_c():
    N, K = 8, 128
    qweight = np.zeros((K, 1), dtype=np.uint32)
    qweight[5, 0] = 0x76543210
    qzeros = np.array([[0xFEDCBA98]], dtype=np.uint32)
    s16 = np.full((1, N), np.float16(1.0))
    blob = tf.prepack_awq(qweight.view(np.int32), qzeros.view(np.int32), s16, N, K, 128)
    qw_nat, scales, zeros, *_ = tf.unprepack(blob)
    q = tf_oracle.unpack(qw_nat, 4, K)
    assert q[:, 5].tolist() == [0, 4, 1, 5, 2, 6, 3, 7]
    assert zeros[:, 0].tolist() == [8, 12, 9, 13, 10, 14, 11, 15]
    assert (scales == 0x3F80).all()


INVALID_ARG, UNSUPPORTED = -1, -2  # TF_ERR_INVALID_ARG, TF_ERR_UNSUPPORTED in include/tf.h


def test_awq_errors():
    L = tf.lib()
    qw = np.zeros((128, 2), dtype=np.int32)
    qz = np.zeros((1, 2), dtype=np.int32)
    s16 = np.zeros((1, 16), dtype=np.uint16)
    out = np.zeros(1 << 20, dtype=np.uint8)
    P = lambda a: a.ctypes.data
    assert L.tf_prepack_awq(P(qw), P(qz), P(s16), 12, 128, 128, P(out), out.size) == INVALID_ARG
    assert L.tf_prepack_awq(None, P(qz), P(s16), 16, 128, 128, P(out), out.size) == INVALID_ARG
    assert L.tf_prepack_awq(P(qw), P(qz), P(s16), 16, 128, 128, P(out), 64) == INVALID_ARG
    assert L.tf_prepack_awq(P(qw), P(qz), P(s16), 16, 128, 96, P(out), out.size) == UNSUPPORTED
    assert L.tf_prepack_awq(P(qw), P(qz), P(s16), 16, 65536, 128, P(out), out.size) == UNSUPPORTED
    assert L.tf_prepack_awq(P(qw), P(qz), P(s16), 16, 128, 128, P(out), out.size) == 0
    with pytest.raises(ValueError):
        tf.prepack_awq(qw, qz, s16, 12, 128, 128)
    with pytest.raises(ValueError):  # float data is not reinterpreted as packed nibbles
        tf.prepack_awq(qw.astype(np.float32), qz, s16, 16, 128, 128)
    with pytest.raises(ValueError):
        tf.prepack_awq(qw, qz, s16.astype(np.float32), 16, 128, 128)
