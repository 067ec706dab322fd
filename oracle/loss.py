"""Float64 oracle of the image loss and its gradient (TEST INFRASTRUCTURE).

Only the test suite, the smoke check and the benchmark's CPU legs may import this module.

The loss whose gradient feeds the backward (Odin: Primitive-Level Synchronization for Distributed
Point-Based Neural Rendering, Figure 7: rendering R precedes backward B). The pages name SSIM only
as an evaluation metric (Odin, Figure 15); the reading taken is the 3D Gaussian splatting training
loss L = (1 - lam) mean|x - y| + lam (1 - mean SSIM(x, y)): SSIM (Wang et al.'s structural
similarity) per channel with an 11x11 Gaussian window of standard deviation 1.5 normalised to sum 1,
C1 = 0.01^2, C2 = 0.03^2 and zeros outside the image; the derivative of |x - y| at x = y is 0.
"""
from __future__ import annotations

import numpy as np
from scipy.ndimage import correlate1d

C1, C2 = 0.01 ** 2, 0.03 ** 2


def window(size: int = 11, sigma: float = 1.5) -> np.ndarray:
    d = np.arange(size, dtype=np.float64) - (size - 1) / 2
    w = np.exp(-d * d / (2 * sigma * sigma))
    return w / w.sum()


def windowed(a: np.ndarray) -> np.ndarray:
    """Zero-padded windowed sum over the last two axes (the 2D Gaussian window is the product of two
    1D windows, so rows then columns)."""
    w = window()
    return correlate1d(correlate1d(a, w, axis=-1, mode="constant"), w, axis=-2, mode="constant")


def ssim_terms(x: np.ndarray, y: np.ndarray):
    mx, my = windowed(x), windowed(y)
    sxx, syy, sxy = windowed(x * x) - mx * mx, windowed(y * y) - my * my, windowed(x * y) - mx * my
    A, B = 2 * mx * my + C1, 2 * sxy + C2
    Cc, D = mx * mx + my * my + C1, sxx + syy + C2
    return mx, my, A, B, Cc, D, A * B / (Cc * D)


def loss_l1_dssim(x: np.ndarray, y: np.ndarray, lam: float = 0.2):
    """(loss, dL/dx) for images [3, H, W] in float64."""
    x = np.asarray(x, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    n = x.size
    mx, my, A, B, Cc, D, S = ssim_terms(x, y)
    loss = (1 - lam) * np.abs(x - y).sum() / n + lam * (1 - S.sum() / n)
    # partial derivatives of S with respect to mu_x, E[x^2] and E[x y] (E = windowed sum)
    d_mu = 2 * my * (B - A) / (Cc * D) - 2 * mx * S * (1 / Cc - 1 / D)
    d_xx = -S / D
    d_xy = 2 * A / (Cc * D)
    dsum = windowed(d_mu) + 2 * x * windowed(d_xx) + y * windowed(d_xy)  # the window is symmetric
    return loss, ((1 - lam) * np.sign(x - y) - lam * dsum) / n
