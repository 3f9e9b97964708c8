"""Pins of the reference blob layout (oracle/layout.py).

The pages fix that the pre-tiling is a pure reordering with the metadata
co-located in each tile (TileFuse, Methodology 2 "Interleaved pre-tiling"),
valid up to 32K.  So: every weight lands on exactly one (byte, nibble), the
round trip is the identity, each unit's metadata follows its weights, the
units of one slab are contiguous, and the padding dequantises to zero.
"""

import numpy as np
import pytest

from gemv_tf_prepack_gb300 import synth
from oracle import layout as L
from oracle import tf_oracle as O


def test_code_coordinates_are_a_bijection_of_the_unit():
    row, col = L.code_coordinates()
    assert row.size == L.UNIT_N * L.UNIT_K
    flat = row * L.UNIT_K + col
    assert np.array_equal(np.sort(flat), np.arange(L.UNIT_N * L.UNIT_K))


def test_fragment_slots_follow_mma_register_order():
    """Hand-checked entries: slot (gr=0,t=0) word 0 holds rows 0/8, cols 0..3."""
    row, col = L.code_coordinates()
    first = list(zip(row[:8].tolist(), col[:8].tolist()))
    # i = 0..7 -> r = i & 3, e = i >> 2: (row, col)
    assert first == [(0, 0), (8, 0), (0, 2), (8, 2), (0, 1), (8, 1), (0, 3), (8, 3)]
    # slot p = 9 -> gr = 2, t = 1; word j = 2 -> cols 16 + 8 = 24..27
    p, j = 9, 2
    idx = (p * 4 + j) * 8
    got = list(zip(row[idx:idx + 8].tolist(), col[idx:idx + 8].tolist()))
    assert got == [(2, 24), (10, 24), (2, 26), (10, 26), (2, 25), (10, 25), (2, 27), (10, 27)]


@pytest.mark.parametrize("N,K,bits,group", [
    (256, 512, 4, 128), (200, 192, 4, 64), (136, 200, 8, 0), (64, 96, 4, 32),
    (130, 256, 8, 128), (8, 8, 4, 0), (128, 1024, 4, 256), (300, 384, 8, 64),
    (200, 1003, 4, 0), (24, 77, 8, 0), (17, 5, 4, 0),  # K % 8 != 0, per channel
])
def test_round_trip_identity(N, K, bits, group):
    qw = synth.make_weights(N, K, bits, group, 1)
    blob = L.prepack(qw.qweight, qw.scales, qw.zeros, N, K, bits, group)
    hd = L.parse_header(blob)
    assert hd["total_bytes"] == blob.size
    assert (hd["N"], hd["K"], hd["bits"], hd["group"]) == (N, K, bits, group)
    r = L.unprepack(blob)
    np.testing.assert_array_equal(r[0], qw.qweight)
    np.testing.assert_array_equal(r[1], qw.scales)
    np.testing.assert_array_equal(r[2], qw.zeros)


def test_every_weight_lands_on_a_distinct_nibble():
    """Exhaustive on a padded 200 x 320 INT4 matrix: tag each weight, find it."""
    N, K = 200, 320
    # q = (n + 3k) mod 16 tags positions; check all (n, k) via unprepack of codes
    q = ((np.arange(N)[:, None] + 3 * np.arange(K)[None, :]) % 16).astype(np.uint8)
    qweight = synth.pack_w4(q)
    s = np.full((N, K // 64), 0x3F80, np.uint16)
    z = np.zeros((N, K // 64), np.uint8)
    blob = L.prepack(qweight, s, z, N, K, 4, 64)
    S, kt, ub, total = L.blob_geometry(N, K, 4, 64)
    row, col = L.code_coordinates()
    seen = np.zeros((S * 16, kt * 128), np.int32)
    for sl in range(S):
        for t in range(kt):
            seen[sl * 16 + row, t * 128 + col] += 1
    assert (seen == 1).all()
    np.testing.assert_array_equal(O.unpack_w4(L.unprepack(blob)[0], K), q)


def test_metadata_is_contiguous_with_its_unit():
    N, K, bits, group = 128, 256, 4, 64
    qw = synth.make_weights(N, K, bits, group, 2)
    blob = L.prepack(qw.qweight, qw.scales, qw.zeros, N, K, bits, group)
    S, kt, ub, _ = L.blob_geometry(N, K, bits, group)
    assert ub == 1024 + 64 + 16
    for sl in (0, 3, 7):
        for t in range(kt):
            base = L.HEADER_BYTES + (sl * kt + t) * ub
            s = blob[base + 1024: base + 1024 + 64].view("<u2").reshape(2, 8, 2)
            z = blob[base + 1088: base + 1104].reshape(2, 8)
            # [gi][gr][e] -> row 16 sl + gr + 8e, group 2t + gi
            for gi in range(2):
                for gr in (0, 5, 7):
                    for e in (0, 1):
                        n = sl * 16 + gr + 8 * e
                        assert s[gi, gr, e] == qw.scales[n, 2 * t + gi]
                        assert (z[gi, gr] >> (4 * e)) & 0xF == qw.zeros[n, 2 * t + gi]


def test_slab_units_are_contiguous():
    """Unit (s, kt + 1) follows unit (s, kt); slab s + 1 follows the last unit of slab s."""
    N, K = 48, 384
    q = np.zeros((N, K), np.uint8)
    q[np.arange(N), (np.arange(N) * 7) % K] = 1 + np.arange(N) % 15  # one tagged code per row
    blob = L.prepack(synth.pack_w4(q), np.full((N, 3), 0x3F80, np.uint16), np.zeros((N, 3), np.uint8),
                     N, K, 4, 128)
    S, kt, ub, total = L.blob_geometry(N, K, 4, 128)
    assert (S, kt, ub) == (8, 3, 1072) and total == 64 + 8 * 3 * 1072
    row, col = L.code_coordinates()
    for n in range(N):
        k = (n * 7) % K
        sl, t = n // 16, k // 128
        base = L.HEADER_BYTES + (sl * kt + t) * ub
        idx = np.flatnonzero((row == n % 16) & (col == k % 128))[0]
        word = int(blob[base + 4 * (idx // 8): base + 4 * (idx // 8) + 4].view("<u4")[0])
        assert (word >> (4 * (idx % 8))) & 0xF == q[n, k]


def test_padding_dequantises_to_zero():
    """Rows >= N and columns >= K contribute exactly zero."""
    N, K = 130, 200
    qw = synth.make_weights(N, K, 8, 0, 4)
    blob = L.prepack(qw.qweight, qw.scales, qw.zeros, N, K, 8, 0)
    S, kt, ub, _ = L.blob_geometry(N, K, 8, 0)
    assert (S, kt, ub) == (16, 2, 2112)
    row, col = L.code_coordinates()
    for sl in range(S):
        for t in range(kt):
            base = L.HEADER_BYTES + (sl * kt + t) * ub
            codes = blob[base: base + 2048]
            sv = blob[base + 2048: base + 2080].view("<u2").reshape(8, 2)
            zv = blob[base + 2080: base + 2096].reshape(8, 2)
            n = sl * 16 + row
            k = t * 128 + col
            grk, ek = row % 8, row // 8
            w = (codes.astype(np.int64) - zv[grk, ek]) * sv[grk, ek].astype(np.int64)
            pad = (n >= N) | (k >= K)
            assert (w[pad] == 0).all()


def test_unit_sizes_are_aligned():
    for bits in (4, 8):
        for group in (32, 64, 128, 0, 256):
            assert L.unit_bytes(bits, group) % 16 == 0
    assert L.unit_bytes(4, 128) == 1072 and L.unit_bytes(8, 0) == 2112
    assert L.unit_bytes(4, 32) == 1024 + 4 * 40 and L.unit_bytes(8, 64) == 2048 + 2 * 48
    for group in (32, 64, 128, 0):  # INT8 halves are 16-byte multiples
        assert L.unit_bytes(8, group) % 32 == 0


def test_32k_geometry():
    S, kt, ub, total = L.blob_geometry(32768, 32768, 4, 128)
    assert (S, kt) == (2048, 256) and total == 64 + 2048 * 256 * 1072


def test_partial_last_word_of_ragged_k():
    """K = 5 per channel: one word per row, codes in its five low nibbles, the
    three high nibbles unused (zero); unpack reads the codes in order, and the
    blob's padding columns k >= 5 carry the row's zero point (exact zeros)."""
    from oracle import tf_oracle
    qweight = np.array([[0x00054321], [0x000FEDCB]], dtype=np.uint32)
    np.testing.assert_array_equal(tf_oracle.unpack_w4(qweight, 5), [[1, 2, 3, 4, 5], [11, 12, 13, 14, 15]])
    scales = np.full((2, 1), 0x3F80, np.uint16)  # 1.0
    zeros = np.array([[3], [9]], np.uint8)
    blob = L.prepack(qweight, scales, zeros, 2, 5, 4, 0)
    r = L.unprepack(blob)
    np.testing.assert_array_equal(r[0], qweight)
    w = tf_oracle.dequant(tf_oracle.unpack_w4(qweight, 5), scales, zeros, 0)
    np.testing.assert_array_equal(w, [[-2, -1, 0, 1, 2], [2, 3, 4, 5, 6]])
