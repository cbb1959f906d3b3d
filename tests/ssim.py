"""Structural similarity (SSIM) of decoded images, the second quality metric of the decoder path.

Definition (Wang, Bovik, Sheikh, Simoncelli, "Image quality assessment: from error visibility to
structural similarity", IEEE TIP 2004): with local Gaussian-weighted means mu, variances sigma^2 and
covariance sigma_xy (11x11 window, sigma 1.5),

    SSIM(x, y) = ((2 mu_x mu_y + C1)(2 sigma_xy + C2)) / ((mu_x^2 + mu_y^2 + C1)(sigma_x^2 + sigma_y^2 + C2)),

C1 = (0.01 L)^2, C2 = (0.03 L)^2 with L the dynamic range (2 for values in [-1, 1]); the image score is
the mean over the positions whose window lies inside the image, averaged over channels and frames.
Plain numpy in float64; test infrastructure only.
"""
import numpy as np


def gaussian_window(size=11, sigma=1.5):
    r = np.arange(size, dtype=np.float64) - (size - 1) / 2
    g = np.exp(-(r * r) / (2 * sigma * sigma))
    g /= g.sum()
    return g


def _filter_valid(img, g):
    """Separable 'valid' correlation of a 2D image with the 1D window g along both axes."""
    k = len(g)
    H, W = img.shape
    rows = np.zeros((H - k + 1, W))
    for i in range(k):
        rows += g[i] * img[i:i + H - k + 1, :]
    out = np.zeros((H - k + 1, W - k + 1))
    for j in range(k):
        out += g[j] * rows[:, j:j + W - k + 1]
    return out


def ssim_plane(x, y, data_range=2.0, size=11, sigma=1.5):
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    g = gaussian_window(size, sigma)
    c1 = (0.01 * data_range) ** 2
    c2 = (0.03 * data_range) ** 2
    mx, my = _filter_valid(x, g), _filter_valid(y, g)
    sxx = _filter_valid(x * x, g) - mx * mx
    syy = _filter_valid(y * y, g) - my * my
    sxy = _filter_valid(x * y, g) - mx * my
    num = (2 * mx * my + c1) * (2 * sxy + c2)
    den = (mx * mx + my * my + c1) * (sxx + syy + c2)
    return float(np.mean(num / den))


def ssim_rgb(got, ref, data_range=2.0):
    """Mean SSIM over frames and RGB channels of [..., H, W, 3] channels-last images."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    g2 = got.reshape(-1, got.shape[-3], got.shape[-2], got.shape[-1])
    r2 = ref.reshape(g2.shape)
    vals = [ssim_plane(g2[f, :, :, c], r2[f, :, :, c], data_range) for f in range(g2.shape[0]) for c in range(3)]
    return float(np.mean(vals))
