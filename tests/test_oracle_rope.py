"""Pins of the rotary-embedding oracle against closed forms (no GPU).

A hand-computed rotation of the rotate-half pairing, norm preservation of
every rotated pair, composition of two rotations into one by the summed
angle (which fixes the sign convention), the identity at angle 0, and the
rows and dims that must stay untouched."""
import math

import numpy as np
import torch

import oracle
from ragged_gqa_attention_gb300 import workloads as W


def _table(angles):
    a = np.asarray(angles, dtype=np.float64)
    return np.concatenate([np.cos(a), np.sin(a)], axis=1)


def test_hand_rotation():
    # D = R = 4: pairs (0, 2) at angle pi/2 and (1, 3) at angle pi
    x = np.array([[[1.0, 2.0, 3.0, 4.0]]])
    cs = np.array([[0.0, -1.0, 1.0, 0.0]])    # cos(pi/2), cos(pi), sin(pi/2), sin(pi)
    np.testing.assert_allclose(oracle.rope(x, cs)[0, 0], [-3.0, -2.0, 1.0, -4.0], atol=0)


def test_pairs_keep_their_norm():
    g = np.random.default_rng(1)
    x = g.standard_normal((5, 3, 16))
    cs = _table(g.uniform(-7, 7, (5, 4)))
    y = oracle.rope(x, cs)
    for i in range(4):
        np.testing.assert_allclose(x[..., i] ** 2 + x[..., i + 4] ** 2,
                                   y[..., i] ** 2 + y[..., i + 4] ** 2, rtol=1e-12)


def test_rotations_compose_by_adding_angles():
    g = np.random.default_rng(2)
    x = g.standard_normal((4, 2, 8))
    a, b = g.uniform(-3, 3, (4, 4)), g.uniform(-3, 3, (4, 4))
    twice = oracle.rope(oracle.rope(x, _table(a)), _table(b))
    np.testing.assert_allclose(twice, oracle.rope(x, _table(a + b)), atol=1e-12)


def test_angle_zero_padding_rows_and_tail_dims():
    g = np.random.default_rng(3)
    x = g.standard_normal((3, 2, 12))
    cs = _table(g.uniform(-3, 3, (3, 4)))     # R = 8 < D = 12
    cs[1] = _table(np.zeros((1, 4)))[0]        # angle 0: identity
    y = oracle.rope(x, cs, positions=np.array([5, 0, -1]))
    np.testing.assert_array_equal(y[1], x[1])
    np.testing.assert_array_equal(y[2], x[2])  # negative position: untouched
    np.testing.assert_array_equal(y[:, :, 8:], x[:, :, 8:])
    assert not np.allclose(y[0, :, :8], x[0, :, :8])


def test_rope_table_helper_angles():
    cs = W.rope_cos_sin([0, 3, -1], 8, base=100.0)
    assert cs.shape == (3, 8) and cs.dtype == torch.float32
    ang = 3 * 100.0 ** (-2.0 * np.arange(4) / 8)
    np.testing.assert_allclose(cs[1].double().numpy(), np.concatenate([np.cos(ang), np.sin(ang)]),
                               rtol=1e-6, atol=1e-7)
    np.testing.assert_array_equal(cs[2].numpy(), [1, 1, 1, 1, 0, 0, 0, 0])
    assert math.isclose(float(cs[0, 0]), 1.0)
