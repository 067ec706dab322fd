"""Float64 oracle of the training step's update phase: sparse Adam (TEST INFRASTRUCTURE).

Only the test suite, the smoke check and the benchmark's CPU legs may import this module.

What it computes (Odin: Primitive-Level Synchronization for Distributed Point-Based Neural
Rendering): the optimizer update phase U of a training step (Figure 7), with Adam as the optimizer
(Review, item 1), restricted to the primitives the view made visible (Abstract: each view reads
and updates only the visible primitives). The pages give no further detail; the readings are:
Adam with bias correction by the step index t, m = b1 m + (1 - b1) g, v = b2 v + (1 - b2) g^2,
x -= lr (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps); "visible" = radius > 0 in that view;
hidden Gaussians keep parameters and moments; one learning rate per tensor, with the SH
coefficient k = 0 (the view-independent colour) and k >= 1 separate.
"""
from __future__ import annotations

import numpy as np

NAMES = ("mean3d", "log_scale", "quat", "opacity_logit", "sh")


def _lr_array(name: str, shape, lr: dict) -> np.ndarray | float:
    if name == "sh":
        a = np.full(shape[1:], lr["sh_rest"], dtype=np.float64)  # [K, 3]
        a[0, :] = lr["sh_dc"]
        return a
    return {"mean3d": lr["mean3d"], "log_scale": lr["log_scale"], "quat": lr["quat"],
            "opacity_logit": lr["opacity"]}[name]


def adam_step_sparse(params: dict, grads: dict, exp_avg: dict, exp_avg_sq: dict, visible: np.ndarray,
                     lr: dict, step: int, beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-15):
    """Returns (params, exp_avg, exp_avg_sq) after one step, as new float64 arrays."""
    vis = np.asarray(visible, dtype=bool)
    bc1 = 1.0 - beta1 ** step
    bc2 = 1.0 - beta2 ** step
    out_p, out_m, out_v = {}, {}, {}
    for name in NAMES:
        p = np.array(params[name], dtype=np.float64)
        g = np.asarray(grads[name], dtype=np.float64)
        m = np.array(exp_avg[name], dtype=np.float64)
        v = np.array(exp_avg_sq[name], dtype=np.float64)
        m_new = beta1 * m[vis] + (1.0 - beta1) * g[vis]
        v_new = beta2 * v[vis] + (1.0 - beta2) * g[vis] * g[vis]
        step_size = _lr_array(name, p.shape, lr)
        p[vis] = p[vis] - step_size * (m_new / bc1) / (np.sqrt(v_new / bc2) + eps)
        m[vis] = m_new
        v[vis] = v_new
        out_p[name], out_m[name], out_v[name] = p, m, v
    return out_p, out_m, out_v


def densify_stats(radius, grad2d, width: int, height: int, ndc: bool, grad_norm_accum, view_count, max_radius,
                  param_grads: dict | None = None):
    """One view's post-backward statistics (returns new arrays): for Gaussians with radius > 0 the
    2-norm of the 2D-mean gradient (in pixel units, or in normalised device coordinates, whose
    derivative is the pixel one times width / 2 and height / 2) is added to grad_norm_accum, the
    view count grows by one and max_radius keeps the largest radius (the per-view statistics 3D
    Gaussian splatting's densification reads); with param_grads, also every Gaussian's 2-norm of
    all its parameter gradients, the per-primitive magnitude of Odin's post-backward hook (Review,
    item 1), 0 for hidden Gaussians."""
    r = np.asarray(radius)
    vis = r > 0
    sx, sy = (0.5 * width, 0.5 * height) if ndc else (1.0, 1.0)
    g = np.asarray(grad2d, dtype=np.float64)
    norm = np.sqrt((sx * g[:, 0]) ** 2 + (sy * g[:, 1]) ** 2)
    acc = np.array(grad_norm_accum, dtype=np.float64)
    cnt = np.array(view_count, dtype=np.int64)
    mr = np.array(max_radius, dtype=np.int64)
    acc[vis] += norm[vis]
    cnt[vis] += 1
    mr[vis] = np.maximum(mr[vis], r[vis])
    mag = None
    if param_grads is not None:
        ss = np.zeros(len(r), dtype=np.float64)
        for name in NAMES:
            a = np.asarray(param_grads[name], dtype=np.float64).reshape(len(r), -1)
            ss += (a * a).sum(axis=1)
        mag = np.where(vis, np.sqrt(ss), 0.0)
    return acc, cnt, mr, mag
