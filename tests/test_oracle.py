"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each ``pin_*`` function takes an oracle namespace (the real ``tf_oracle`` or a
copy with a planted mistake) and raises AssertionError when the namespace
disagrees with the mathematics: hand-worked values, exact rational
arithmetic, closed forms, a second library's BF16 conversion, special cases.
``test_planted_mistakes_are_caught`` checks that plausible mistakes in the
oracle fail at least one pin.
"""

import os
import types
from fractions import Fraction

import numpy as np
import pytest

from gemv_tf_prepack_gb300 import synth
from oracle import tf_oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# independent helpers (exact rational arithmetic)

def frac_bf16_round(v: Fraction) -> Fraction:
    """Round an exact rational to BF16, ties to even (8 significant bits)."""
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (max(e, -126) - 7)
    n = a / quantum
    f = n.numerator // n.denominator
    rem = n - f
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return sign * f * quantum


def bits_to_frac(b: int) -> Fraction:
    """Exact value of a (finite) BF16 bit pattern, decoded field by field."""
    sign = -1 if b & 0x8000 else 1
    exp = (b >> 7) & 0xFF
    man = b & 0x7F
    assert exp != 0xFF
    if exp == 0:
        return sign * Fraction(man, 128) * Fraction(2) ** -126
    return sign * (1 + Fraction(man, 128)) * Fraction(2) ** (exp - 127)


def load_golden(name):
    rec = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            rec[key] = vals
    return rec


# ----------------------------------------------------------------------------
# pins

def pin_bf16_vs_torch(O):
    """Oracle BF16 rounding == torch's float32 -> bfloat16 conversion (RNE)."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(123)
    u = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    # ties and near-ties around 1.0, subnormals, the overflow edge
    extra = np.array([1 + 2**-8, 1 + 3 * 2**-8, 1 + 2**-8 + 2**-20, -(1 + 2**-8), 2**-130,
                      3 * 2**-134, 2**-133, 3.3895314e38, 3.39e38, 0.0, -0.0], dtype=np.float32)
    f = np.concatenate([f, extra])
    got = O.bf16_round(f.astype(np.float64))
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    same = (got == ref) | (np.isinf(got) & np.isinf(ref) & (np.sign(got) == np.sign(ref)))
    assert same.all(), f"{(~same).sum()} mismatches, first {f[~same][:4]}"


def pin_bf16_hand_ties(O):
    """Halfway cases go to the even neighbour (values checked by hand)."""
    v = np.array([1 + 2**-8, 1 + 3 * 2**-8, 1 + 2**-8 + 2**-30, 255.5, 256.5 * 2, 257.0])
    want = np.array([1.0, 1 + 2**-6, 1 + 2**-7, 256.0, 512.0, 256.0])
    np.testing.assert_array_equal(O.bf16_round(v), want)


def pin_unpack_single_nibble(O):
    """A word with one non-zero nibble v at position j decodes to v at k=j only."""
    words = []
    expect = []
    for j in range(8):
        for v in range(16):
            words.append(v << (4 * j))
            row = [0] * 8
            row[j] = v
            expect.append(row)
    q = O.unpack_w4(np.array(words, dtype=np.uint32)[:, None], 8)
    np.testing.assert_array_equal(q, np.array(expect, dtype=np.uint8))
    # two words per row: the second word holds k = 8..15
    q2 = O.unpack_w4(np.array([[0x00000000, 0x0000000F]], dtype=np.uint32), 16)
    assert q2[0, 8] == 15 and q2[0, :8].sum() == 0 and q2[0, 9:].sum() == 0


def pin_dequant_power_of_two_scale(O):
    """s = 2^-6, z = 8: wd = (q - 8) / 64 exactly; W8 s = 2^-10, z = 128."""
    q = np.arange(16, dtype=np.uint8)[None, :]
    wd = O.dequant(q, np.array([[0x3C80]], np.uint16), np.array([[8]], np.uint8), 0)
    np.testing.assert_array_equal(wd[0], (np.arange(16) - 8) / 64.0)
    q8 = np.arange(256, dtype=np.uint8)[None, :]
    wd8 = O.dequant(q8, np.array([[0x3A80]], np.uint16), np.array([[128]], np.uint8), 0)
    np.testing.assert_array_equal(wd8[0], (np.arange(256) - 128) / 1024.0)


def pin_dequant_all_pairs_rational(O):
    """s = bf16(0.0123) = 0x3C4A and every (q, z) pair: exact Fraction + hand RNE."""
    s_bits = 0x3C4A
    s = bits_to_frac(s_bits)
    for Q in (15, 255):
        qs = np.arange(Q + 1)
        zs = np.arange(Q + 1)
        qq, zz = np.meshgrid(qs, zs, indexing="ij")
        q = qq.reshape(-1, 1).astype(np.uint8)
        z = zz.reshape(-1, 1).astype(np.uint8)
        got = O.dequant(q, np.full((q.shape[0], 1), s_bits, np.uint16), z, 0)[:, 0]
        diffs = sorted(set((qq - zz).ravel().tolist()))
        table = {d: float(frac_bf16_round(d * s)) for d in diffs}
        want = np.array([table[d] for d in (qq - zz).ravel()])
        np.testing.assert_array_equal(got, want)


def pin_dequant_groups(O):
    """Two groups of 4 along K with different (s, z): group index is k // g."""
    q = np.array([[1, 2, 3, 4, 5, 6, 7, 8]], np.uint8)
    s = np.array([[0x3F80, 0x4000]], np.uint16)   # 1.0, 2.0
    z = np.array([[1, 5]], np.uint8)
    wd = O.dequant(q, s, z, 4)
    np.testing.assert_array_equal(wd[0], [0, 1, 2, 3, 0, 2, 4, 6])


def pin_golden_worked_example(O):
    g = load_golden("worked_tiny_w4.txt")
    N, K, group = int(g["N"][0]), int(g["K"][0]), int(g["group"][0])
    qweight = np.array([int(v, 16) for v in g["qweight_hex"]], np.uint32).reshape(N, K // 8)
    q = O.unpack_w4(qweight, K)
    np.testing.assert_array_equal(q[0], [int(v) for v in g["q_row0"]])
    np.testing.assert_array_equal(q[1], [int(v) for v in g["q_row1"]])
    scales = np.array([int(v, 16) for v in g["scales_hex"]], np.uint16).reshape(N, 1)
    zeros = np.array([int(v) for v in g["zeros"]], np.uint8).reshape(N, 1)
    wd_bits = O.dequant_bits(q, scales, zeros, group)
    np.testing.assert_array_equal(wd_bits[0], [int(v, 16) for v in g["wd_row0_hex"]])
    np.testing.assert_array_equal(wd_bits[1], [int(v, 16) for v in g["wd_row1_hex"]])
    x = np.array([int(v, 16) for v in g["x_hex"]], np.uint16).reshape(1, K)
    y = O.reference(qweight, scales, zeros, 4, group, K, x)
    np.testing.assert_array_equal(y[0], [float(v) for v in g["y"]])


def pin_closed_forms(O):
    """One-hot x with z = 0, s = 1 returns a column of q; constant q and all-ones x."""
    rng = np.random.default_rng(7)
    N, K = 8, 64
    q = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    qweight = synth.pack_w4(q)
    s = np.full((N, 1), 0x3F80, np.uint16)
    z = np.zeros((N, 1), np.uint8)
    for k in (0, 5, 63):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80
        y = O.reference(qweight, s, z, 4, 0, K, x)
        np.testing.assert_array_equal(y[0], q[:, k].astype(np.float64))
    # constant q = 11, z = 3, s = 0.25, x = ones: y = K * (11 - 3) * 0.25 = 2K
    qc = np.full((N, K), 11, np.uint8)
    y = O.reference(synth.pack_w4(qc), np.full((N, 1), 0x3E80, np.uint16),
                    np.full((N, 1), 3, np.uint8), 4, 0, K, np.full((2, K), 0x3F80, np.uint16))
    np.testing.assert_array_equal(y, np.full((2, N), 2.0 * K))
    # row-dependent constant: y[m, n] depends on n only through row n of W
    qr = np.repeat(np.arange(N, dtype=np.uint8)[:, None], K, axis=1)
    y = O.reference(synth.pack_w4(qr), s, z, 4, 0, K, np.full((1, K), 0x3F80, np.uint16))
    np.testing.assert_array_equal(y[0], K * np.arange(N, dtype=np.float64))


def pin_brute_force_rational(O):
    """Tiny products against exact Fractions (independent RNE for the weights)."""
    rng = np.random.default_rng(11)
    for bits, g, K, M in [(4, 64, 64, 1), (4, 128, 128, 2), (4, 64, 128, 2), (8, 64, 128, 1)]:
        N = 8
        Q = 2**bits - 1
        q = rng.integers(0, Q + 1, size=(N, K)).astype(np.uint8)
        z = rng.integers(0, Q + 1, size=(N, K // g)).astype(np.uint8)
        s = (0x3C00 + rng.integers(0, 0x200, size=(N, K // g))).astype(np.uint16)
        x = synth.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
        qweight = synth.pack_w4(q) if bits == 4 else q
        y = O.reference(qweight, s, z, bits, g, K, x)
        for m in range(M):
            for n in range(N):
                acc = Fraction(0)
                for k in range(K):
                    w = frac_bf16_round((int(q[n, k]) - int(z[n, k // g])) * bits_to_frac(int(s[n, k // g])))
                    acc += bits_to_frac(int(x[m, k])) * w
                ref = float(acc)
                assert abs(y[m, n] - ref) <= 1e-12 * max(1.0, abs(ref)), (bits, g, K, m, n, y[m, n], ref)


def pin_single_nonzero_group(O):
    """W whose only nonzero group is group j of row n: y[:, n] is that group's 128-term dot
    product (exact Fractions), every other output is 0.  A wrong group-to-column map fails."""
    rng = np.random.default_rng(17)
    N, K, g, M = 4, 512, 128, 2
    for n0, j in [(1, 2), (3, 0), (0, 3)]:
        q = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
        s = np.zeros((N, K // g), np.uint16)          # scale 0: the group dequantises to 0
        z = rng.integers(0, 16, size=(N, K // g)).astype(np.uint8)
        s[n0, j] = 0x3F00                              # 0.5
        x = synth.f32_to_bf16_bits(rng.standard_normal((M, K)).astype(np.float32))
        y = O.reference(synth.pack_w4(q), s, z, 4, g, K, x)
        for m in range(M):
            want = sum(bits_to_frac(int(x[m, k])) * (int(q[n0, k]) - int(z[n0, j])) * Fraction(1, 2)
                       for k in range(j * g, (j + 1) * g))
            assert abs(y[m, n0] - float(want)) <= 1e-12 * max(1.0, abs(float(want)))
            assert all(y[m, n] == 0.0 for n in range(N) if n != n0)


def _row_constant_layer(N, K):
    """A W4 layer whose row n is the constant code q_n with zero z_n and a power-of-two
    scale s_n, all three varying with n: with all-ones x, y[n] = K (q_n - z_n) s_n
    exactly, so every output names the row it came from."""
    n = np.arange(N)
    q = (n % 16).astype(np.uint8)
    z = ((n // 16) % 13).astype(np.uint8)                 # periods 208 and 1792 rows: no two
    e = (n // 256) % 7                                     # 2048-row chunks look alike; s_n = 2^(e_n - 4)
    s = (0x3F80 + ((e.astype(np.int64) - 4) << 7)).astype(np.uint16)
    qweight = synth.pack_w4(np.repeat(q[:, None], K, axis=1))
    want = K * (q.astype(np.float64) - z) * np.ldexp(1.0, (e - 4).astype(np.int64))
    return qweight, s[:, None], z[:, None], want


def pin_rows_and_chunks(O):
    """reference() past its 2048-row chunks, and reference_rows() for unsorted, repeated rows
    spread over those chunks: both against the closed form K (q_n - z_n) s_n, and
    reference_rows() on one-hot x against the requested columns of q."""
    N, K = 4200, 64
    qweight, s, z, want = _row_constant_layer(N, K)
    ones = np.full((2, K), 0x3F80, np.uint16)
    y = O.reference(qweight, s, z, 4, 0, K, ones)
    np.testing.assert_array_equal(y, np.broadcast_to(want, (2, N)))
    rows = np.array([4199, 3, 2048, 2047, 3, 4096, 100, 4095, 2049, 0])
    yr = O.reference_rows(qweight, s, z, 4, 0, K, ones, rows)
    np.testing.assert_array_equal(yr, np.broadcast_to(want[rows], (2, rows.size)))
    # one-hot x, z = 0, s = 1: output i is q[rows[i], k]
    rng = np.random.default_rng(29)
    q = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
    for k in (0, 37):
        x = np.zeros((1, K), np.uint16)
        x[0, k] = 0x3F80
        yr = O.reference_rows(synth.pack_w4(q), np.full((N, 1), 0x3F80, np.uint16), np.zeros((N, 1), np.uint8),
                              4, 0, K, x, rows)
        np.testing.assert_array_equal(yr[0], q[rows, k].astype(np.float64))


PINS = [pin_bf16_vs_torch, pin_bf16_hand_ties, pin_unpack_single_nibble,
        pin_dequant_power_of_two_scale, pin_dequant_all_pairs_rational, pin_dequant_groups,
        pin_golden_worked_example, pin_closed_forms, pin_brute_force_rational, pin_single_nonzero_group,
        pin_rows_and_chunks]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(tf_oracle)


# ----------------------------------------------------------------------------
# planted mistakes: each must fail at least one pin

def _mutant(**overrides):
    ns = types.SimpleNamespace(**{k: getattr(tf_oracle, k) for k in tf_oracle.__all__})
    for k, v in overrides.items():
        setattr(ns, k, v)

    # re-bind the composite functions so that they use the mutated parts
    def dequant_bits(q, s, z, g):
        return tf_oracle.bf16_value_to_bits(ns.dequant(q, s, z, g))

    def reference(qweight, s, z, bits, group, K, x, rows_per_chunk=2048):
        q = ns.unpack(qweight, bits, K)
        wd = ns.dequant(q, s, z, group)
        return ns.linear_f64(x, wd)

    def unpack(qweight, bits, K):
        return ns.unpack_w4(qweight, K) if bits == 4 else tf_oracle.unpack_w8(qweight, K)

    if "dequant_bits" not in overrides:
        ns.dequant_bits = dequant_bits
    if "reference" not in overrides:
        ns.reference = reference
    if "unpack" not in overrides:
        ns.unpack = unpack
    return ns


def _bad_unpack_high_first(qweight, K):
    qweight = np.asarray(qweight, dtype=np.uint32)
    k = np.arange(K)
    shifts = (4 * (7 - (k & 7))).astype(np.uint32)
    return ((qweight[:, k >> 3] >> shifts[None, :]) & 0xF).astype(np.uint8)


def _bad_dequant_sign(q, s, z, group):
    n, k = q.shape
    g = k if group == 0 else group
    j = np.arange(k) // g
    return tf_oracle.bf16_round((z.astype(np.int64)[:, j] - q.astype(np.int64))
                                * tf_oracle.bf16_bits_to_f64(s)[:, j])


def _bad_dequant_prescaled_zero(q, s, z, group):
    """q*s - z*s with each product rounded to BF16 first (a common shortcut)."""
    n, k = q.shape
    g = k if group == 0 else group
    j = np.arange(k) // g
    sf = tf_oracle.bf16_bits_to_f64(s)[:, j]
    a = tf_oracle.bf16_round(q.astype(np.float64) * sf)
    b = tf_oracle.bf16_round(z.astype(np.float64)[:, j] * sf)
    return tf_oracle.bf16_round(a - b)


def _bad_dequant_group_index(q, s, z, group):
    n, k = q.shape
    ng = s.shape[1]
    j = np.arange(k) % ng
    return tf_oracle.bf16_round((q.astype(np.int64) - z.astype(np.int64)[:, j])
                                * tf_oracle.bf16_bits_to_f64(s)[:, j])


def _bad_round_truncate(v):
    v = np.asarray(v, dtype=np.float64)
    f = v.astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
    return f.view(np.float32).astype(np.float64)


def _bad_linear_drops_last_k(x_bits, wd, rows_per_chunk=4096):
    x = tf_oracle.bf16_bits_to_f64(x_bits)
    return x[:, :-1] @ np.asarray(wd)[:, :-1].T


def _bad_linear_float32(x_bits, wd, rows_per_chunk=4096):
    x = tf_oracle.bf16_bits_to_f64(x_bits).astype(np.float32)
    return (x @ np.asarray(wd, np.float32).T).astype(np.float64)


def _bad_rows_metadata_by_position(qweight, scales_bits, zeros, bits, group, K, x_bits, rows):
    """Codes taken for the requested rows, scales and zeros by position instead."""
    rows = np.asarray(rows)
    q = tf_oracle.unpack(qweight[rows], bits, K)
    wd = tf_oracle.dequant(q, scales_bits[:rows.size], zeros[:rows.size], group)
    return tf_oracle.linear_f64(x_bits, wd)


def _bad_rows_sorted(qweight, scales_bits, zeros, bits, group, K, x_bits, rows):
    """Outputs in sorted (and de-duplicated) row order rather than the requested one."""
    return tf_oracle.reference_rows(qweight, scales_bits, zeros, bits, group, K, x_bits, np.unique(rows))


def _bad_reference_chunk_metadata(qweight, s, z, bits, group, K, x, rows_per_chunk=2048):
    """Chunked over rows, but every chunk reads the first chunk's scales and zeros."""
    n = qweight.shape[0]
    y = np.empty((x.shape[0], n), dtype=np.float64)
    for r0 in range(0, n, rows_per_chunk):
        r1 = min(n, r0 + rows_per_chunk)
        q = tf_oracle.unpack(qweight[r0:r1], bits, K)
        wd = tf_oracle.dequant(q, s[:r1 - r0], z[:r1 - r0], group)
        y[:, r0:r1] = tf_oracle.linear_f64(x, wd)
    return y


MUTANTS = {
    "rows_metadata_by_position": dict(reference_rows=_bad_rows_metadata_by_position),
    "rows_returned_sorted": dict(reference_rows=_bad_rows_sorted),
    "reference_chunks_reuse_first_metadata": dict(reference=_bad_reference_chunk_metadata),
    "unpack_high_nibble_first": dict(unpack_w4=_bad_unpack_high_first),
    "dequant_sign_flipped": dict(dequant=_bad_dequant_sign),
    "dequant_prescaled_zero": dict(dequant=_bad_dequant_prescaled_zero),
    "dequant_wrong_group_index": dict(dequant=_bad_dequant_group_index),
    "bf16_truncation": dict(bf16_round=_bad_round_truncate),
    "linear_drops_last_k": dict(linear_f64=_bad_linear_drops_last_k),
    "linear_in_float32": dict(linear_f64=_bad_linear_float32),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name):
    overrides = dict(MUTANTS[name])
    if "bf16_round" in overrides:
        bad_round = overrides["bf16_round"]

        def dequant(q, s, z, group, _r=bad_round):
            n, k = q.shape
            g = k if group == 0 else group
            j = np.arange(k) // g
            return _r((q.astype(np.int64) - z.astype(np.int64)[:, j]) * tf_oracle.bf16_bits_to_f64(s)[:, j])
        overrides["dequant"] = dequant
    ns = _mutant(**overrides)
    failed = []
    for pin in PINS:
        try:
            pin(ns)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"planted mistake {name} passed every pin"


# ----------------------------------------------------------------------------
# the generator's quantiser (input preparation) obeys its recipe

@pytest.mark.parametrize("bits,group", [(4, 128), (4, 64), (4, 32), (8, 0), (8, 128), (4, 0)])
def test_quantiser_invariants(bits, group):
    N, K, seed = 64, 512, 3
    rng = np.random.default_rng(seed)
    w = rng.standard_normal((N, K), dtype=np.float32) * np.float32(0.02)
    qw = synth.quantise(w, bits, group)
    Q = 2**bits - 1
    q = tf_oracle.unpack(qw.qweight, bits, K)
    assert q.max() <= Q and qw.zeros.max() <= Q
    g = qw.g
    wd = tf_oracle.dequant(q, qw.scales, qw.zeros, group)
    s = tf_oracle.bf16_bits_to_f64(qw.scales)[:, np.arange(K) // g]
    err = np.abs(w.astype(np.float64) - wd)
    clamped = (q == 0) | (q == Q)
    slack = 2.0**-8 * np.abs(wd) + 1e-9
    assert (err[~clamped] <= 0.5 * s[~clamped] * (1 + 1e-5) + slack[~clamped]).all()
    assert (err[clamped] <= 1.5 * s[clamped] + slack[clamped]).all()
    qg = q.reshape(N, K // g, g)
    assert (qg.min(axis=2) <= 1).all() and (qg.max(axis=2) >= Q - 1).all()


def test_generator_chunking_is_one_stream():
    a = synth.make_weights(40, 256, 4, 128, 9, rows_per_chunk=40)
    b = synth.make_weights(40, 256, 4, 128, 9, rows_per_chunk=16)
    np.testing.assert_array_equal(a.qweight, b.qweight)
    np.testing.assert_array_equal(a.scales, b.scales)
    np.testing.assert_array_equal(a.zeros, b.zeros)


def test_activation_outliers():
    x = synth.make_activations(4, 4096, 7, outliers=True)
    xf = synth.bf16_bits_to_f32(x)
    big = (np.abs(xf) > 6).any(axis=0)
    assert 30 <= big.sum() <= 41  # 41 outlier columns, most of them exceed 6 in some row
