"""Pins of the reference blob layout (oracle/layout.py).

The pages fix that the pre-tiling is a pure reordering with the metadata
co-located in each tile (TileFuse, Methodology 2 "Interleaved pre-tiling"),
valid up to 32K.  So: every weight lands on exactly one (byte, nibble), the
round trip is the identity, each tile's metadata follows its weights, and the
padding dequantises to zero.
"""

import numpy as np
import pytest

from gemv_tf_prepack_gb300 import synth
from oracle import layout as L
from oracle import tf_oracle as O


def test_code_coordinates_are_a_bijection_of_the_tile():
    row, col = L.code_coordinates()
    assert row.size == L.TILE_N * L.TILE_K
    flat = row * L.TILE_K + col
    assert np.array_equal(np.sort(flat), np.arange(L.TILE_N * L.TILE_K))


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
    nb, kt, tb, total = L.blob_geometry(N, K, 4, 64)
    row, col = L.code_coordinates()
    seen = np.zeros((nb * 128, kt * 128), np.int32)
    for b in range(nb):
        for t in range(kt):
            seen[b * 128 + row, t * 128 + col] += 1
    assert (seen == 1).all()
    np.testing.assert_array_equal(O.unpack_w4(L.unprepack(blob)[0], K), q)


def test_metadata_is_contiguous_with_its_tile():
    N, K, bits, group = 128, 256, 4, 64
    qw = synth.make_weights(N, K, bits, group, 2)
    blob = L.prepack(qw.qweight, qw.scales, qw.zeros, N, K, bits, group)
    nb, kt, tb, _ = L.blob_geometry(N, K, bits, group)
    assert tb == 8192 + 512 + 128
    for t in range(kt):
        base = L.HEADER_BYTES + t * tb
        s = blob[base + 8192: base + 8192 + 512].view("<u2").reshape(2, 8, 8, 2)
        # [gi][mb][gr][e] -> scale of row mb*16 + gr + 8e, group 2t + gi
        for gi in range(2):
            for mb in (0, 7):
                for gr in (0, 5):
                    for e in (0, 1):
                        assert s[gi, mb, gr, e] == qw.scales[mb * 16 + gr + 8 * e, 2 * t + gi]


def test_padding_dequantises_to_zero():
    """Rows >= N and columns >= K contribute exactly zero."""
    N, K = 130, 200
    qw = synth.make_weights(N, K, 8, 0, 4)
    blob = L.prepack(qw.qweight, qw.scales, qw.zeros, N, K, 8, 0)
    nb, kt, tb, _ = L.blob_geometry(N, K, 8, 0)
    row, col = L.code_coordinates()
    for b in range(nb):
        for t in range(kt):
            base = L.HEADER_BYTES + (b * kt + t) * tb
            codes = blob[base: base + 16384]
            sv = blob[base + 16384: base + 16384 + 256].view("<u2").reshape(8, 8, 2)
            zv = blob[base + 16384 + 256: base + 16384 + 384].reshape(8, 8, 2)
            n = b * 128 + row
            k = t * 128 + col
            mbk, grk, ek = row // 16, row % 8, (row % 16) // 8
            w = (codes.astype(np.int64) - zv[mbk, grk, ek]) * sv[mbk, grk, ek].astype(np.int64)
            pad = (n >= N) | (k >= K)
            assert (w[pad] == 0).all()


def test_tile_sizes_are_16_byte_multiples():
    for bits in (4, 8):
        for group in (32, 64, 128, 0, 256):
            assert L.tile_bytes(bits, group) % 16 == 0
    assert L.tile_bytes(4, 128) == 8512 and L.tile_bytes(8, 0) == 16768


def test_32k_geometry():
    nb, kt, tb, total = L.blob_geometry(32768, 32768, 4, 128)
    assert (nb, kt) == (256, 256) and total == 64 + 65536 * 8512
