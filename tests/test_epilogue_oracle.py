"""The epilogue oracle pinned to what the mathematics fixes, and the host
pre-tiling of a gate/up pair against the oracle's interleaving (CPU only).

Pins of ``oracle.epilogue``:
* silu: the values the sigmoid takes at 0 and ln 3 (1/2 and 3/4), the
  identity silu(a) - silu(-a) = a, its limits, and scipy's logistic sigmoid
  (expit) as an independent library routine;
* the gate/up row interleaving: written out by hand for F = 16;
* silu_gate: hand-computed values on a tiny layer;
* split_qkv: the three blocks put back side by side give y.
A planted mistake in each (a swapped gate/up role, an off-by-one block, a
sign error in the exponent) fails one of these.
"""

import math

import numpy as np
import pytest

import gemv_tf_prepack_gb300 as tf
from gemv_tf_prepack_gb300 import synth
from oracle import epilogue as E
from oracle import layout as L


def test_silu_closed_forms():
    assert E.silu(0.0) == 0.0
    assert E.silu(math.log(3.0)) == pytest.approx(0.75 * math.log(3.0), rel=1e-15)
    assert E.silu(-math.log(3.0)) == pytest.approx(-0.25 * math.log(3.0), rel=1e-15)
    a = np.linspace(-30, 30, 601)
    np.testing.assert_allclose(E.silu(a) - E.silu(-a), a, rtol=0, atol=1e-12)
    assert E.silu(200.0) == 200.0
    assert E.silu(-800.0) == 0.0  # exp overflows: -800 / inf
    assert np.signbit(E.silu(-800.0))


def test_silu_matches_scipy_expit():
    special = pytest.importorskip("scipy.special")
    a = np.random.default_rng(3).standard_normal(10000) * 8
    np.testing.assert_allclose(E.silu(a), a * special.expit(a), rtol=1e-13, atol=1e-300)


def test_gate_up_interleaving_written_out():
    F = 16
    gate = np.arange(F)
    up = 1000 + np.arange(F)
    want = list(range(0, 8)) + list(range(1000, 1008)) + list(range(8, 16)) + list(range(1008, 1016))
    assert E.interleave_gate_up(gate, up).tolist() == want
    with pytest.raises(ValueError):
        E.interleave_gate_up(np.arange(12), np.arange(12))


def test_silu_gate_hand_values():
    # one token, F = 8: gate row f holds f - 4, up row f holds 2 (biased sums)
    y = np.zeros((1, 16))
    y[0, :8] = np.arange(8) - 4.0
    y[0, 8:] = 2.0
    h = E.silu_gate(y)
    want = [2.0 * (a / (1.0 + math.exp(-a))) for a in range(-4, 4)]
    np.testing.assert_allclose(h[0], want, rtol=1e-15)
    # the roles are not symmetric: exchanging gate and up changes the result
    y2 = np.concatenate([y[:, 8:], y[:, :8]], axis=1)
    assert not np.allclose(E.silu_gate(y2), h)
    with pytest.raises(ValueError):
        E.silu_gate(np.zeros((1, 24)))


def test_split_qkv_blocks():
    y = np.arange(3 * 40).reshape(3, 40)
    q, k, v = E.split_qkv(y, 16, 8)
    assert q.shape == (3, 16) and k.shape == (3, 8) and v.shape == (3, 16)
    np.testing.assert_array_equal(np.concatenate([q, k, v], axis=1), y)
    q, k, v = E.split_qkv(y, 40, 0)
    assert k.shape == (3, 0) and v.shape == (3, 0)
    with pytest.raises(ValueError):
        E.split_qkv(y, 0, 8)
    with pytest.raises(ValueError):
        E.split_qkv(y, 30, 11)


@pytest.mark.parametrize("F,K,bits,group", [(8, 256, 4, 128), (24, 192, 8, 64), (40, 128, 4, 0), (16, 96, 4, 32)])
def test_prepack_gate_up_matches_oracle_interleaving(F, K, bits, group):
    g = synth.make_weights(F, K, bits, group, 61)
    u = synth.make_weights(F, K, bits, group, 62)
    got = tf.prepack_gate_up((g.qweight, g.scales, g.zeros), (u.qweight, u.scales, u.zeros), F, K, bits, group)
    N = 2 * F
    ref = L.prepack(E.interleave_gate_up(g.qweight, u.qweight), E.interleave_gate_up(g.scales, u.scales),
                    E.interleave_gate_up(g.zeros, u.zeros), N, K, bits, group)
    np.testing.assert_array_equal(got, ref)


def test_prepack_gate_up_rejects_bad_f():
    g = synth.make_weights(12, 128, 4, 128, 1)
    with pytest.raises(tf.TFError):
        tf.prepack_gate_up((g.qweight, g.scales, g.zeros), (g.qweight, g.scales, g.zeros), 12, 128, 4, 128)
