"""Pins of the SSIM used as the second quality metric (CPU only): values the definition fixes."""
import numpy as np

from tests.ssim import gaussian_window, ssim_plane, ssim_rgb

C1 = (0.01 * 2.0) ** 2
C2 = (0.03 * 2.0) ** 2


def test_window_is_normalised_and_symmetric():
    g = gaussian_window()
    assert abs(g.sum() - 1.0) < 1e-15 and np.allclose(g, g[::-1]) and g.argmax() == 5


def test_identical_images_score_one():
    x = np.random.default_rng(1).uniform(-1, 1, (32, 40))
    assert abs(ssim_plane(x, x) - 1.0) < 1e-12


def test_constant_images_reduce_to_the_luminance_term():
    # zero variance everywhere: SSIM = (2ab + C1)/(a^2 + b^2 + C1) * (0 + C2)/(0 + C2)
    a, b = 0.3, -0.2
    x = np.full((20, 20), a)
    y = np.full((20, 20), b)
    want = (2 * a * b + C1) / (a * a + b * b + C1)
    assert abs(ssim_plane(x, y) - want) < 1e-12


def test_negated_zero_mean_texture_gives_the_closed_form():
    # y = -x with a zero-mean local texture: the luminance term is 1 and the structure term is
    # (C2 - 2 s)/(2 s + C2) with s the local variance; a +-1 checkerboard has mean 0 in every 11x11
    # window only approximately, so use a texture that is exactly zero-mean under the window: a
    # single-axis alternation whose Gaussian-weighted mean over 11 taps is computed exactly here.
    g = gaussian_window()
    x = np.tile(np.array([1.0, -1.0]), (16, 8))
    y = -x
    m = float(sum(g[j] * (1.0 if j % 2 == 0 else -1.0) for j in range(11)))  # local mean magnitude
    s = 1.0 - m * m                                                      # local variance
    lum = (2 * (m * -m) + C1) / (m * m + m * m + C1)
    # the mean alternates sign between odd and even columns; both give the same product
    want = lum * (2 * (-s) + C2) / (2 * s + C2)
    assert abs(ssim_plane(x, y) - want) < 1e-12


def test_small_noise_lowers_the_score_monotonically():
    rng = np.random.default_rng(2)
    x = rng.uniform(-1, 1, (48, 48))
    scores = [ssim_plane(x, x + e * rng.standard_normal(x.shape)) for e in (1e-3, 1e-2, 1e-1)]
    assert 1.0 > scores[0] > scores[1] > scores[2]


def test_rgb_average_over_channels_and_frames():
    rng = np.random.default_rng(3)
    x = rng.uniform(-1, 1, (2, 24, 24, 3))
    y = x.copy()
    y[1, :, :, 2] = 0.0
    per = [ssim_plane(x[f, :, :, c], y[f, :, :, c]) for f in range(2) for c in range(3)]
    assert abs(ssim_rgb(y, x) - np.mean(per)) < 1e-15
