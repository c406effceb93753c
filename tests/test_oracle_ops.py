"""Pins for the oracle's single-layer operators (CPU only).

Each operator is checked against something other than itself: an independent
library routine (PyTorch CPU float64), a closed form, or brute force.
"""
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import ops
from oracle.decoder import band_rows, output_shape, temporal_upsample
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng(1234)


def t64(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float64))


# ---------------------------------------------------------------- convolution
@pytest.mark.parametrize("shape,cout,k", [((2, 3, 7, 9), 5, 3), ((1, 4, 1, 5), 2, 3),
                                          ((1, 6, 5, 4), 3, 1), ((1, 2, 6, 6), 3, 5)])
def test_conv2d_matches_torch(shape, cout, k):
    x = rng.standard_normal(shape)
    w = rng.standard_normal((cout, shape[1], k, k))
    b = rng.standard_normal(cout)
    ref = F.conv2d(t64(x), t64(w), t64(b), padding=k // 2).numpy()
    np.testing.assert_allclose(ops.conv2d_same(x, w, b), ref, rtol=1e-12, atol=1e-12)


def test_conv2d_asymmetric_padding_matches_torch():
    x = rng.standard_normal((1, 3, 6, 5))
    w = rng.standard_normal((2, 3, 3, 3))
    b = rng.standard_normal(2)
    pad = (0, 2, 1, 1)     # top, bottom, left, right
    ref = F.conv2d(F.pad(t64(x), (pad[2], pad[3], pad[0], pad[1])), t64(w), t64(b)).numpy()
    np.testing.assert_allclose(ops.conv2d(x, w, b, pad), ref, rtol=1e-12, atol=1e-12)


def test_conv2d_delta_kernel_is_identity():
    x = rng.standard_normal((1, 4, 5, 6))
    w = np.zeros((4, 4, 3, 3))
    for c in range(4):
        w[c, c, 1, 1] = 1.0
    np.testing.assert_array_equal(ops.conv2d_same(x, w, np.zeros(4)), x)


@pytest.mark.parametrize("dy,dx", [(0, 1), (2, 1), (1, 0), (1, 2), (0, 0), (2, 2)])
def test_conv2d_shift_kernel_moves_rows_with_zero_edges(dy, dx):
    # A single 1 at tap (dy, dx) reads x[y + dy - 1, x + dx - 1]; outside the
    # image the value is the zero padding.
    h, w_ = 5, 6
    x = rng.standard_normal((1, 1, h, w_))
    w = np.zeros((1, 1, 3, 3))
    w[0, 0, dy, dx] = 1.0
    y = ops.conv2d_same(x, w, np.zeros(1))
    for i in range(h):
        for j in range(w_):
            si, sj = i + dy - 1, j + dx - 1
            exp = x[0, 0, si, sj] if (0 <= si < h and 0 <= sj < w_) else 0.0
            assert y[0, 0, i, j] == exp


def test_causal_conv3d_matches_torch():
    x = rng.standard_normal((1, 3, 4, 5, 6))
    w = rng.standard_normal((2, 3, 3, 3, 3))
    b = rng.standard_normal(2)
    xp = F.pad(t64(x), (1, 1, 1, 1, 2, 0))          # W, H, then T: (2 front, 0 back)
    ref = F.conv3d(xp, t64(w), t64(b)).numpy()
    np.testing.assert_allclose(ops.causal_conv3d(x, w, b), ref, rtol=1e-12, atol=1e-12)


def test_causal_conv3d_is_causal():
    # Changing frame t must not change outputs before t.
    x = rng.standard_normal((1, 2, 5, 3, 3))
    w = rng.standard_normal((2, 2, 3, 3, 3))
    b = np.zeros(2)
    y0 = ops.causal_conv3d(x, w, b)
    x2 = x.copy()
    x2[:, :, 3] += 1.0
    y1 = ops.causal_conv3d(x2, w, b)
    np.testing.assert_array_equal(y0[:, :, :3], y1[:, :, :3])
    assert np.abs(y0[:, :, 3:] - y1[:, :, 3:]).max() > 0


# ---------------------------------------------------------------- pointwise
def test_silu_matches_torch():
    x = rng.standard_normal(1000) * 10
    np.testing.assert_allclose(ops.silu(x), F.silu(t64(x)).numpy(), rtol=1e-14, atol=1e-300)


def test_upsample_matches_torch_and_index_identity():
    x = rng.standard_normal((2, 3, 4, 5))
    y = ops.upsample_nearest2x(x)
    np.testing.assert_array_equal(y, F.interpolate(t64(x), scale_factor=2, mode="nearest").numpy())
    np.testing.assert_array_equal(y, F.interpolate(t64(x), scale_factor=2, mode="nearest-exact").numpy())
    assert y[1, 2, 7, 9] == x[1, 2, 3, 4]


def test_rms_norm_matches_torch_normalize():
    x = rng.standard_normal((2, 6, 3, 4, 5))
    g = rng.standard_normal(6)
    ref = F.normalize(t64(x), dim=1) * np.sqrt(6) * t64(g).view(1, 6, 1, 1, 1)
    np.testing.assert_allclose(ops.rms_norm_channels(x, g), ref.numpy(), rtol=1e-13, atol=1e-13)
    # zero pixels stay zero (eps clamp)
    x[:, :, 0, 0, 0] = 0
    assert np.all(ops.rms_norm_channels(x, g)[:, :, 0, 0, 0] == 0)


# ---------------------------------------------------------------- GroupNorm
@pytest.mark.parametrize("shape,groups", [((2, 8, 5, 7), 4), ((1, 6, 3, 3), 3), ((2, 8, 3, 4, 5), 2)])
def test_group_norm_matches_torch(shape, groups):
    x = rng.standard_normal(shape) * 3 + 1.5
    g = rng.standard_normal(shape[1])
    b = rng.standard_normal(shape[1])
    ref = F.group_norm(t64(x), groups, t64(g), t64(b), eps=1e-6).numpy()
    np.testing.assert_allclose(ops.group_norm(x, groups, g, b, 1e-6), ref, rtol=1e-11, atol=1e-11)


def test_group_norm_of_constant_is_beta():
    x = np.full((1, 4, 3, 3), 7.25)
    beta = np.array([0.5, -1.0, 2.0, 3.0])
    y = ops.group_norm(x, 2, np.ones(4), beta, 1e-6)
    np.testing.assert_allclose(y, np.broadcast_to(beta.reshape(1, 4, 1, 1), y.shape), atol=0)


@pytest.mark.parametrize("rows,offset", [([34, 33, 33], 0.0), ([16] * 4, 0.0), ([1, 1, 5, 1], 0.0),
                                         ([34, 33, 33], 1e4), ([1, 7], 1e4)])
def test_band_moment_merge_equals_whole_tensor(rows, offset):
    # Bands with different means, so a merge that drops the (mean_i - mean)^2
    # term, or weights bands equally instead of by element count, fails.
    h = sum(rows)
    x = rng.standard_normal((2, 8, h, 5)) * 0.01 + offset
    x += np.linspace(0, 3, h)[None, None, :, None]
    n_all, m_all, v_all = ops.group_moments(x, 4)
    parts, y = [], 0
    for r in rows:
        parts.append(ops.group_moments(x[:, :, y:y + r], 4))
        y += r
    n, m, v = ops.merge_moments(parts)
    assert n == n_all
    np.testing.assert_allclose(m, m_all, rtol=1e-12, atol=0)
    np.testing.assert_allclose(v, v_all, rtol=1e-9, atol=0)
    # law of total variance holds and the merged variance exceeds the mean of
    # within-band variances by the between-band term
    within = sum(p[0] / n * p[2] for p in parts)
    assert np.all(v > within)


def test_band_moment_merge_large_offset_is_cancellation_free():
    # mean 1e6, spread 1e-3: E[x^2] - mean^2 in float64 would lose every digit.
    x = 1e6 + rng.standard_normal((1, 2, 30, 4)) * 1e-3
    parts = [ops.group_moments(x[:, :, a:b], 1) for a, b in ((0, 11), (11, 12), (12, 30))]
    _, m, v = ops.merge_moments(parts)
    _, m_all, v_all = ops.group_moments(x, 1)
    np.testing.assert_allclose(v, v_all, rtol=1e-6)


# ---------------------------------------------------------------- attention
def test_sdpa_matches_torch():
    q = rng.standard_normal((7, 16))
    k = rng.standard_normal((11, 16))
    v = rng.standard_normal((11, 16))
    ref = F.scaled_dot_product_attention(t64(q)[None], t64(k)[None], t64(v)[None])[0].numpy()
    np.testing.assert_allclose(ops.sdpa(q, k, v), ref, rtol=1e-12, atol=1e-12)


def test_sdpa_constant_keys_give_mean_value():
    q = rng.standard_normal((5, 8))
    k = np.tile(rng.standard_normal((1, 8)), (9, 1))
    v = rng.standard_normal((9, 8))
    np.testing.assert_allclose(ops.sdpa(q, k, v), np.tile(v.mean(0), (5, 1)), rtol=1e-12, atol=1e-13)


def test_sdpa_dominant_score_selects_value_row():
    d = 4
    k = np.eye(6, d) * 1e3
    v = rng.standard_normal((6, d))
    q = np.zeros((1, d))
    q[0, 2] = 1.0
    np.testing.assert_allclose(ops.sdpa(q, k, v)[0], v[2], rtol=1e-12)


def test_sdpa_row_split_equals_unsplit():
    q = rng.standard_normal((10, 8))
    k = rng.standard_normal((12, 8))
    v = rng.standard_normal((12, 8))
    whole = ops.sdpa(q, k, v)
    parts = np.concatenate([ops.sdpa(q[:3], k, v), ops.sdpa(q[3:], k, v)])
    np.testing.assert_array_equal(whole, parts)


def test_linear_matches_torch():
    x = rng.standard_normal((5, 6))
    w = rng.standard_normal((3, 6))
    b = rng.standard_normal(3)
    np.testing.assert_allclose(ops.linear(x, w, b), F.linear(t64(x), t64(w), t64(b)).numpy(), rtol=1e-13)


# ---------------------------------------------------------------- band plan / shapes
def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_band_rows_golden():
    for parts in _golden_lines("band_rows.txt"):
        h, n, rows = int(parts[0]), int(parts[1]), [int(p) for p in parts[2:]]
        assert band_rows(h, n) == rows


def test_band_rows_properties():
    for h in range(1, 40):
        for n in range(1, h + 1):
            r = band_rows(h, n)
            assert sum(r) == h and len(r) == n and max(r) - min(r) <= 1 and r == sorted(r, reverse=True)
    with pytest.raises(ValueError):
        band_rows(4, 5)
    with pytest.raises(ValueError):
        band_rows(4, 0)


def test_output_shapes_golden():
    for name, lat, out in _golden_lines("output_shapes.txt"):
        w = synth.WORKLOADS[name]
        assert tuple(int(v) for v in lat.split(",")) == w.latent_shape
        assert output_shape(w.arch, w.latent_shape) == tuple(int(v) for v in out.split(","))


# ---------------------------------------------------------------- temporal upsample
def test_temporal_upsample_frames_and_torch():
    c, t = 3, 4
    a = rng.standard_normal((1, c, t, 2, 3))
    w = rng.standard_normal((2 * c, c, 3, 1, 1))
    b = rng.standard_normal(2 * c)
    y = temporal_upsample(a, w, b)
    assert y.shape[2] == 2 * t - 1
    np.testing.assert_array_equal(y[:, :, 0], a[:, :, 0])
    tc = F.conv3d(F.pad(t64(a[:, :, 1:]), (0, 0, 0, 0, 2, 0)), t64(w), t64(b)).numpy()
    for i in range(t - 1):
        np.testing.assert_allclose(y[:, :, 1 + 2 * i], tc[:, :c, i], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(y[:, :, 2 + 2 * i], tc[:, c:, i], rtol=1e-12, atol=1e-12)
    # a single frame passes through unchanged
    np.testing.assert_array_equal(temporal_upsample(a[:, :, :1], w, b), a[:, :, :1])
