"""Pins of the pre/post-op oracle (oracle/prepost.py) against what does not
depend on it: numpy's own convolution, closed forms, impulse responses,
continuation through the history, and small hand-worked values."""
from __future__ import annotations

import numpy as np
import pytest

from oracle import prepost

rng = np.random.default_rng(7)


@pytest.mark.parametrize("W", [1, 2, 3, 4])
def test_conv_matches_numpy_convolve_per_channel(W):
    L, D = 11, 5
    x = rng.standard_normal((L, D))
    w = rng.standard_normal((D, W))
    h0 = rng.standard_normal((1, D, W - 1))
    y, hT = prepost.causal_conv1d(x, w, None, h0, [0, L])
    for c in range(D):
        ext = np.concatenate([h0[0, c], x[:, c]])
        # np.convolve flips its kernel: correlate with w = convolve with w reversed
        ref = np.convolve(ext, w[c, ::-1], mode="valid")
        np.testing.assert_allclose(y[:, c], ref, rtol=0, atol=1e-12)
        np.testing.assert_allclose(hT[0, c], ext[len(ext) - (W - 1):], rtol=0, atol=0)


def test_conv_width_one_is_a_per_channel_scale_with_no_history():
    x = rng.standard_normal((6, 3))
    w = np.array([[2.0], [-1.0], [0.5]])
    b = np.array([0.1, 0.2, 0.3])
    y, hT = prepost.causal_conv1d(x, w, b, None, [0, 6])
    np.testing.assert_allclose(y, x * w[:, 0] + b, rtol=0, atol=1e-15)
    assert hT.shape == (1, 3, 0)


def test_conv_impulse_response_reads_the_weights_backwards():
    W, D, L = 4, 2, 9
    w = rng.standard_normal((D, W))
    x = np.zeros((L, D))
    x[2] = 1.0
    y, _ = prepost.causal_conv1d(x, w, None, None, [0, L])
    for j in range(W):  # y[2 + j] = w[:, W - 1 - j]
        np.testing.assert_allclose(y[2 + j], w[:, W - 1 - j], rtol=0, atol=0)
    assert np.all(y[:2] == 0) and np.all(y[2 + W:] == 0)


def test_conv_history_alone_feeds_the_first_outputs():
    W, D = 4, 3
    w = rng.standard_normal((D, W))
    h0 = rng.standard_normal((1, D, W - 1))
    y, _ = prepost.causal_conv1d(np.zeros((5, D)), w, None, h0, [0, 5])
    # y[0] = w[:,0] h[0] + w[:,1] h[1] + w[:,2] h[2]; y[1] = w[:,0] h[1] + w[:,1] h[2]
    np.testing.assert_allclose(y[0], (w[:, :3] * h0[0]).sum(1), atol=1e-15)
    np.testing.assert_allclose(y[1], w[:, 0] * h0[0, :, 1] + w[:, 1] * h0[0, :, 2], atol=1e-15)
    np.testing.assert_allclose(y[2], w[:, 0] * h0[0, :, 2], atol=1e-15)
    assert np.all(y[3:] == 0)


@pytest.mark.parametrize("split", [1, 2, 5, 9])
def test_conv_continuation_through_the_history(split):
    W, D, L = 4, 4, 10
    x = rng.standard_normal((L, D))
    w = rng.standard_normal((D, W))
    b = rng.standard_normal(D)
    h0 = rng.standard_normal((1, D, W - 1))
    y, hT = prepost.causal_conv1d(x, w, b, h0, [0, L], prepost.ACT_SILU)
    y1, h1 = prepost.causal_conv1d(x[:split], w, b, h0, [0, split], prepost.ACT_SILU)
    y2, h2 = prepost.causal_conv1d(x[split:], w, b, h1, [0, L - split], prepost.ACT_SILU)
    np.testing.assert_allclose(np.concatenate([y1, y2]), y, atol=1e-14)
    np.testing.assert_allclose(h2, hT, atol=0)


def test_conv_short_sequence_keeps_part_of_the_old_history():
    W, D = 4, 2
    h0 = np.arange(6, dtype=float).reshape(1, D, W - 1)
    x = np.array([[10.0, 20.0]])
    _, hT = prepost.causal_conv1d(x, np.ones((D, W)), None, h0, [0, 1])
    np.testing.assert_array_equal(hT[0], [[1.0, 2.0, 10.0], [4.0, 5.0, 20.0]])
    # an empty sequence hands its history back unchanged
    _, hT = prepost.causal_conv1d(np.zeros((0, D)), np.ones((D, W)), None, h0, [0, 0])
    np.testing.assert_array_equal(hT, h0)


def test_conv_packed_sequences_do_not_see_each_other():
    W, D = 3, 2
    x = rng.standard_normal((7, D))
    w = rng.standard_normal((D, W))
    y, _ = prepost.causal_conv1d(x, w, None, None, [0, 3, 3, 7])
    ya, _ = prepost.causal_conv1d(x[:3], w, None, None, [0, 3])
    yb, _ = prepost.causal_conv1d(x[3:], w, None, None, [0, 4])
    np.testing.assert_array_equal(y, np.concatenate([ya, yb]))


def test_silu_values():
    # silu(0) = 0; silu(x) -> x for large x; silu(-x) = silu(x) - x
    y, _ = prepost.causal_conv1d(np.array([[0.0], [30.0], [-2.0], [2.0]]), np.ones((1, 1)), None,
                                 None, [0, 4], prepost.ACT_SILU)
    assert y[0, 0] == 0.0
    assert abs(y[1, 0] - 30.0) < 1e-11
    assert abs(y[2, 0] - (y[3, 0] - 2.0)) < 1e-15
    assert abs(y[3, 0] - 2.0 / (1.0 + np.exp(-2.0))) < 1e-15


def test_l2norm_values():
    y = prepost.l2norm(np.array([[3.0, 4.0], [0.0, 0.0]]), 0.0 + 1e-300)
    np.testing.assert_allclose(y[0], [0.6, 0.8], atol=1e-15)
    assert np.all(y[1] == 0.0)
    x = rng.standard_normal((5, 16))
    np.testing.assert_allclose(np.linalg.norm(prepost.l2norm(x, 0.0), axis=1), 1.0, atol=1e-14)
    # eps enters under the root: a row of norm 1 with eps = 3 halves
    np.testing.assert_allclose(prepost.l2norm(np.array([[1.0, 0.0]]), 3.0), [[0.5, 0.0]])


def test_rmsnorm_gated_values():
    x = np.full((1, 4), 2.0)
    wgt = np.array([1.0, 2.0, 3.0, 4.0])
    # a constant row c has RMS |c|: y = sign(c) * weight (eps = 0)
    np.testing.assert_allclose(prepost.rmsnorm_gated(x, wgt, None, 0.0), [[1, 2, 3, 4]], atol=1e-15)
    # a zero gate silences the row; a large gate passes it
    assert np.all(prepost.rmsnorm_gated(x, wgt, np.zeros((1, 4)), 0.0) == 0.0)
    np.testing.assert_allclose(prepost.rmsnorm_gated(x, wgt, np.full((1, 4), 40.0), 0.0),
                               [[40, 80, 120, 160]], rtol=1e-12)
    # unit weights: every output row has RMS 1 (eps = 0)
    y = prepost.rmsnorm_gated(rng.standard_normal((6, 32)), np.ones(32), None, 0.0)
    np.testing.assert_allclose(np.sqrt((y * y).mean(axis=1)), 1.0, atol=1e-14)
