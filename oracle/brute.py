"""Brute-force per-pixel renderer for tiny scenes (numpy, float64).

TEST INFRASTRUCTURE: it pins the tiled oracle renderer. It builds no duplicate list and calls no
sort of keys: for every tile it enumerates the Gaussians whose 3-sigma square covers one of the
tile's pixel indices, by testing each of those indices directly, orders them by (float32 depth,
index), and blends every pixel of the tile front to back with the rules of the rendering phase:
alpha = min(0.99, o exp(power)), skip when power > 0 or alpha < float32(1/255), stop before a
Gaussian that would take T below float32(1e-4).
"""
from __future__ import annotations

import numpy as np


def _covers(centre_minus_half: float, r: int, first_index: int) -> bool:
    idx = np.arange(first_index, first_index + 16, dtype=np.float64)
    return bool(np.any(np.abs(idx - centre_minus_half) <= r))


def render(mean2d, conic, opacity, rgb, depth32, radius, mean2d_f32, width, height, bg):
    """mean2d/conic/opacity/rgb float64 (the values blended); mean2d_f32 and radius decide the
    tile membership, depth32 the order. Returns image [3,H,W], t_final [H,W], n_contrib [H,W]."""
    n = len(radius)
    tx_n, ty_n = (width + 15) // 16, (height + 15) // 16
    image = np.zeros((3, height, width))
    t_final = np.ones((height, width))
    n_contrib = np.zeros((height, width), np.uint32)
    bits = np.asarray(depth32, np.float32).view(np.uint32)
    a_min, t_min = float(np.float32(1.0) / np.float32(255.0)), float(np.float32(1e-4))
    for ty in range(ty_n):
        for tx in range(tx_n):
            cand = [g for g in range(n) if radius[g] > 0
                    and _covers(float(mean2d_f32[g, 0]) - 0.5, int(radius[g]), 16 * tx)
                    and _covers(float(mean2d_f32[g, 1]) - 0.5, int(radius[g]), 16 * ty)]
            cand.sort(key=lambda g: (int(bits[g]), g))
            ys, xs = np.mgrid[16 * ty:min(16 * ty + 16, height), 16 * tx:min(16 * tx + 16, width)]
            ys, xs = ys.ravel(), xs.ravel()
            T = np.ones(len(xs))
            col = np.zeros((3, len(xs)))
            alive = np.ones(len(xs), bool)
            last = np.zeros(len(xs), np.uint32)
            for pos, g in enumerate(cand):
                dx = mean2d[g, 0] - (xs + 0.5)
                dy = mean2d[g, 1] - (ys + 0.5)
                A, B, Cc = conic[g]
                power = -0.5 * (A * dx * dx + Cc * dy * dy) - B * dx * dy
                alpha = np.minimum(0.99, opacity[g] * np.exp(power))
                use = alive & (power <= 0.0) & (alpha >= a_min)
                test_t = T * (1.0 - alpha)
                stop = use & (test_t < t_min)
                alive &= ~stop
                use &= ~stop
                col += np.where(use, rgb[g][:, None] * alpha * T, 0.0)
                T = np.where(use, test_t, T)
                last = np.where(use, pos + 1, last)
            image[:, ys, xs] = col + T[None, :] * np.asarray(bg, np.float64)[:, None]
            t_final[ys, xs] = T
            n_contrib[ys, xs] = last
    return image, t_final, n_contrib
