"""Pins of the fp64 sublayer references (oracle/sublayer.py) to facts fixed outside them: values worked by hand,
closed forms of special cases, and invariants of the definitions."""
import numpy as np

from oracle import sublayer


def test_l2norm_hand_values_and_eps():
    np.testing.assert_allclose(sublayer.l2norm([3.0, 4.0], 0.0), [0.6, 0.8], rtol=0, atol=1e-15)
    # eps shrinks the norm to |x| / sqrt(|x|^2 + eps) exactly
    y = sublayer.l2norm([3.0, 4.0], 11.0)
    np.testing.assert_allclose(np.linalg.norm(y), 5.0 / 6.0, rtol=1e-15)
    np.testing.assert_array_equal(sublayer.l2norm(np.zeros(5), 1e-6), np.zeros(5))
    # per row of the last axis, scale-free
    x = np.random.default_rng(1).standard_normal((4, 3, 8))
    np.testing.assert_allclose(sublayer.l2norm(7.5 * x, 0.0), sublayer.l2norm(x, 0.0), rtol=1e-14)
    np.testing.assert_allclose(np.linalg.norm(sublayer.l2norm(x, 0.0), axis=-1), 1.0, rtol=1e-14)


def test_gated_rmsnorm_closed_forms():
    o = np.array([3.0, -3.0, 3.0, -3.0])
    big = np.full(4, 60.0)  # sigmoid = 1 to double precision
    np.testing.assert_allclose(sublayer.gated_rmsnorm(o, big, None, 0.0), [1, -1, 1, -1], rtol=1e-15)
    np.testing.assert_allclose(sublayer.gated_rmsnorm(o, np.zeros(4), None, 0.0), [0.5, -0.5, 0.5, -0.5],
                               rtol=1e-15)
    w = np.array([2.0, 1.0, 0.5, 0.0])
    np.testing.assert_allclose(sublayer.gated_rmsnorm(o, big, w, 0.0), [2, -1, 0.5, 0], rtol=1e-15)
    # rms of [1, 2, 2] is sqrt(3); eps enters under the root
    np.testing.assert_allclose(sublayer.gated_rmsnorm([1.0, 2.0, 2.0], big[:3], None, 1.0), np.array([1, 2, 2]) / 2.0,
                               rtol=1e-15)
    np.testing.assert_allclose(sublayer.sigmoid([0.0, np.log(3.0)]), [0.5, 0.75], rtol=1e-15)
    x = np.random.default_rng(2).standard_normal((5, 16))
    z = np.random.default_rng(3).standard_normal((5, 16))
    np.testing.assert_allclose(sublayer.gated_rmsnorm(4.0 * x, z, None, 0.0), sublayer.gated_rmsnorm(x, z, None, 0.0),
                               rtol=1e-14)


def test_short_conv_impulse_response_and_state_carry():
    rng = np.random.default_rng(4)
    C, W = 3, 4
    w = rng.standard_normal((C, W))
    x = np.zeros((10, C))
    x[2] = 1.0
    y, _ = sublayer.short_conv(x, w, [0, 10])
    for j in range(W):
        np.testing.assert_array_equal(y[2 + j], w[:, j])  # the impulse response is the filter
    assert not y[:2].any() and not y[2 + W:].any()
    # documents do not see each other: the same tokens packed after another document give the same outputs
    xa, xb = rng.standard_normal((7, C)), rng.standard_normal((5, C))
    y_pack, st = sublayer.short_conv(np.concatenate([xa, xb]), w, [0, 7, 12])
    y_b, st_b = sublayer.short_conv(xb, w, [0, 5])
    np.testing.assert_array_equal(y_pack[7:], y_b)
    np.testing.assert_array_equal(st[1], st_b[0])
    np.testing.assert_array_equal(st[0], xa[-(W - 1):])  # the state is the last W - 1 inputs
    # a document split in two with the state carried equals the whole document
    xs = rng.standard_normal((11, C))
    y_all, st_all = sublayer.short_conv(xs, w, [0, 11])
    y1, s1 = sublayer.short_conv(xs[:4], w, [0, 4])
    y2, s2 = sublayer.short_conv(xs[4:], w, [0, 7], state=s1)
    np.testing.assert_allclose(np.concatenate([y1, y2]), y_all, rtol=1e-15, atol=1e-15)
    np.testing.assert_array_equal(s2, st_all)
    # a split shorter than the window keeps older carried entries
    y3, s3 = sublayer.short_conv(xs[4:5], w, [0, 1], state=s1)
    np.testing.assert_array_equal(s3[0], np.concatenate([s1[0][1:], xs[4:5]]))
