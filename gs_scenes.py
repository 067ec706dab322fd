"""Seeded synthetic scenes for the tile-based 3D Gaussian splatting training step.

This module only draws random inputs. It holds none of the rasterizer's arithmetic: no
projection, no covariance, no blending. Both the CUDA library's tests and benchmark and the
float64 CPU oracle consume what it returns, so it is the one piece of code they share.

The pages that describe the method (DISTWAR: Fast Differentiable Rendering on Raster-based
Rendering Pipelines, Abstract; ARC: Warp-level Adaptive Atomic Reduction in GPUs to Accelerate
Differentiable Rendering, Abstract) evaluate on real captured scenes that are not available here.
The five recipes below stand in for them: they reproduce the Gaussian counts, image sizes,
depth spreads and per-tile overlap that those workloads have, from a seeded PCG64 stream.

Scene layout (all float32, C-contiguous, row-major):
    mean3d        [N, 3]   world-space centres
    log_scale     [N, 3]   per-axis log standard deviations
    quat          [N, 4]   rotation quaternion (w, x, y, z), unit length
    opacity_logit [N]      pre-sigmoid opacity
    sh            [N, K, 3] spherical-harmonic coefficients, K = (degree + 1)^2, channel last
Cameras: world-to-camera rotation R (row-major 3x3) and translation t (p_cam = R p_world + t),
pinhole focal lengths and principal point in pixels, image size, background colour.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = ["Camera", "Scene", "CONFIGS", "make_scene", "make_target", "scene_summary"]


@dataclasses.dataclass
class Camera:
    R: np.ndarray          # float32 [9], world->camera rotation, row-major
    t: np.ndarray          # float32 [3]
    fx: float
    fy: float
    cx: float
    cy: float
    width: int
    height: int
    bg: np.ndarray         # float32 [3]

    @property
    def tiles_x(self) -> int:
        return (self.width + 15) // 16

    @property
    def tiles_y(self) -> int:
        return (self.height + 15) // 16

    @property
    def n_tiles(self) -> int:
        return self.tiles_x * self.tiles_y

    @property
    def n_pixels(self) -> int:
        return self.width * self.height


@dataclasses.dataclass
class Scene:
    name: str
    mean3d: np.ndarray
    log_scale: np.ndarray
    quat: np.ndarray
    opacity_logit: np.ndarray
    sh: np.ndarray
    sh_degree: int
    cameras: list
    targets: list          # one float32 [3, H, W] target image per camera

    @property
    def n(self) -> int:
        return int(self.mean3d.shape[0])

    @property
    def sh_k(self) -> int:
        return (self.sh_degree + 1) ** 2


# name, N, W, H, fx, SH degree, background, views
CONFIGS = {
    0: dict(name="tiny", n=2_000, width=128, height=128, f=128.0, deg=0, bg=(0.0, 0.0, 0.0), views=1),
    1: dict(name="object", n=100_000, width=800, height=800, f=1111.0, deg=3, bg=(1.0, 1.0, 1.0), views=1),
    2: dict(name="outdoor", n=1_600_000, width=1297, height=840, f=1160.0, deg=3, bg=(0.0, 0.0, 0.0), views=1),
    3: dict(name="large", n=3_000_000, width=1959, height=1090, f=1500.0, deg=3, bg=(0.0, 0.0, 0.0), views=8),
    4: dict(name="contention", n=50_000, width=3840, height=2160, f=1920.0, deg=0, bg=(0.0, 0.0, 0.0), views=1),
}


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _unit_quats(rng, n):
    q = rng.standard_normal((n, 4))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    return q


def _uniform_sphere_dirs(rng, n):
    v = rng.standard_normal((n, 3))
    return v / np.linalg.norm(v, axis=1, keepdims=True)


def _cluster_mixture(rng, n, n_clusters, sigma):
    centres = np.empty((n_clusters, 3))
    centres[:, 0:2] = rng.uniform(-10.0, 10.0, size=(n_clusters, 2))
    centres[:, 2] = rng.uniform(4.0, 24.0, size=n_clusters)
    pick = rng.integers(0, n_clusters, size=n)
    return centres[pick] + sigma * rng.standard_normal((n, 3))


def _sh_coeffs(rng, n, deg):
    k = (deg + 1) ** 2
    sh = np.zeros((n, k, 3))
    if deg == 0:
        # Degree 0 scenes are specified by their colour c ~ U[0,1]; the stored DC coefficient is
        # chosen so that the evaluated colour, DC * Y00 + 0.5 with Y00 = 1 / (2 sqrt(pi)), is c.
        colour = rng.uniform(0.0, 1.0, size=(n, 3))
        sh[:, 0, :] = (colour - 0.5) * (2.0 * math.sqrt(math.pi))
    else:
        sh[:, 0, :] = rng.uniform(0.0, 1.0, size=(n, 3))
        sh[:, 1:, :] = 0.05 * rng.standard_normal((n, k - 1, 3))
    return sh


def _camera(R, t, f, width, height, bg, res_scale=1.0):
    w = max(16, int(round(width * res_scale)))
    h = max(16, int(round(height * res_scale)))
    s = w / width
    return Camera(R=np.asarray(R, np.float32).reshape(9), t=np.asarray(t, np.float32).reshape(3),
                  fx=float(np.float32(f * s)), fy=float(np.float32(f * s)),
                  cx=float(np.float32(w / 2.0)), cy=float(np.float32(h / 2.0)),
                  width=w, height=h, bg=np.asarray(bg, np.float32))


def _view_rotation(yaw, pitch):
    cy_, sy_ = math.cos(yaw), math.sin(yaw)
    cp, sp = math.cos(pitch), math.sin(pitch)
    ryaw = np.array([[cy_, 0.0, sy_], [0.0, 1.0, 0.0], [-sy_, 0.0, cy_]])
    rpitch = np.array([[1.0, 0.0, 0.0], [0.0, cp, -sp], [0.0, sp, cp]])
    return rpitch @ ryaw


def make_target(rng: np.random.Generator, cam: Camera) -> np.ndarray:
    return rng.uniform(0.0, 1.0, size=(3, cam.height, cam.width)).astype(np.float32)


def make_scene(cfg: int, seed: int | None = None, n: int | None = None,
               res_scale: float = 1.0, views: int | None = None) -> Scene:
    """Draw configuration `cfg` (0..4) with PCG64(seed); seed defaults to the config index.

    `n` overrides the Gaussian count and `res_scale` shrinks the image and focal length together
    (the field of view is kept), which gives smaller cases of the same shape for tests.
    """
    c = CONFIGS[cfg]
    seed = cfg if seed is None else seed
    rng = _rng(seed)
    n = c["n"] if n is None else int(n)
    n_views = c["views"] if views is None else int(views)
    f, W, H = c["f"], c["width"], c["height"]
    eye = np.eye(3)

    if cfg == 0:
        mean = np.empty((n, 3))
        mean[:, 0:2] = rng.uniform(-1.0, 1.0, size=(n, 2))
        mean[:, 2] = rng.uniform(2.0, 4.0, size=n)
        log_scale = rng.normal(-3.0, 0.5, size=(n, 3))
        logit = rng.normal(0.0, 1.0, size=n)
        cams = [_camera(eye, (0, 0, 0), f, W, H, c["bg"], res_scale)]
    elif cfg == 1:
        r = 1.3 * rng.uniform(0.0, 1.0, size=n) ** (1.0 / 3.0)
        mean = _uniform_sphere_dirs(rng, n) * r[:, None]
        log_scale = rng.normal(-4.5, 0.6, size=(n, 3))
        logit = rng.normal(0.0, 1.5, size=n)
        # camera centre at (0, 0, -4) looking along +z at the origin
        cams = [_camera(eye, (0, 0, 4.0), f, W, H, c["bg"], res_scale)]
    elif cfg == 2:
        mean = _cluster_mixture(rng, n, 64, 1.5)
        log_scale = rng.normal(-3.5, 1.0, size=(n, 3))
        logit = rng.normal(0.0, 1.5, size=n)
        cams = [_camera(eye, (0, 0, 0), f, W, H, c["bg"], res_scale)]
    elif cfg == 3:
        n_shell = n // 5
        n_clu = n - n_shell
        clu = _cluster_mixture(rng, n_clu, 128, 1.5)
        tanx, tany = (W / 2.0) / f, (H / 2.0) / f
        u = rng.uniform(-1.1 * tanx, 1.1 * tanx, size=n_shell)
        v = rng.uniform(-1.1 * tany, 1.1 * tany, size=n_shell)
        d = np.stack([u, v, np.ones_like(u)], axis=1)
        d /= np.linalg.norm(d, axis=1, keepdims=True)
        shell = d * rng.uniform(30.0, 60.0, size=n_shell)[:, None]
        mean = np.concatenate([clu, shell], axis=0)
        log_scale = rng.normal(-3.0, 1.2, size=(n, 3))
        logit = rng.normal(0.0, 1.5, size=n)
        cams = []
        for _ in range(n_views):
            yaw, pitch = np.deg2rad(rng.uniform(-10.0, 10.0, size=2))
            cams.append(_camera(_view_rotation(yaw, pitch), rng.uniform(-1.0, 1.0, size=3),
                                f, W, H, c["bg"], res_scale))
    elif cfg == 4:
        z = np.cbrt(rng.uniform(20.0 ** 3, 40.0 ** 3, size=n))
        tanx, tany = (W / 2.0) / f, (H / 2.0) / f
        mean = np.stack([z * rng.uniform(-tanx, tanx, size=n), z * rng.uniform(-tany, tany, size=n), z], axis=1)
        log_scale = rng.normal(-1.0, 0.3, size=(n, 3))
        logit = rng.normal(-2.0, 0.5, size=n)
        cams = [_camera(eye, (0, 0, 0), f, W, H, c["bg"], res_scale)]
    else:
        raise ValueError(f"unknown config {cfg}")

    quat = _unit_quats(rng, n)
    sh = _sh_coeffs(rng, n, c["deg"])
    targets = [make_target(rng, cam) for cam in cams]
    f32 = lambda a: np.ascontiguousarray(a, dtype=np.float32)
    return Scene(name=c["name"], mean3d=f32(mean), log_scale=f32(log_scale), quat=f32(quat),
                 opacity_logit=f32(logit), sh=f32(sh), sh_degree=c["deg"], cameras=cams,
                 targets=targets)


def make_scene_random_small(seed: int, n: int, width: int, height: int, f: float, deg: int,
                            depth=(2.0, 4.0), log_scale_mu=-2.5, log_scale_sd=0.5,
                            bg=(0.0, 0.0, 0.0), extent=1.0) -> Scene:
    """Free-form small scene for finite-difference and brute-force checks."""
    rng = _rng(seed)
    mean = np.empty((n, 3))
    mean[:, 0:2] = rng.uniform(-extent, extent, size=(n, 2))
    mean[:, 2] = rng.uniform(depth[0], depth[1], size=n)
    log_scale = rng.normal(log_scale_mu, log_scale_sd, size=(n, 3))
    logit = rng.normal(0.0, 1.0, size=n)
    quat = _unit_quats(rng, n)
    k = (deg + 1) ** 2
    sh = np.zeros((n, k, 3))
    sh[:, 0, :] = rng.uniform(-1.0, 1.0, size=(n, 3))
    if k > 1:
        sh[:, 1:, :] = 0.3 * rng.standard_normal((n, k - 1, 3))
    cam = Camera(R=np.eye(3, dtype=np.float32).reshape(9), t=np.zeros(3, np.float32), fx=float(f),
                 fy=float(f), cx=width / 2.0, cy=height / 2.0, width=width, height=height,
                 bg=np.asarray(bg, np.float32))
    f32 = lambda a: np.ascontiguousarray(a, dtype=np.float32)
    return Scene(name="small", mean3d=f32(mean), log_scale=f32(log_scale), quat=f32(quat),
                 opacity_logit=f32(logit), sh=f32(sh), sh_degree=deg, cameras=[cam],
                 targets=[make_target(rng, cam)])


def scene_summary(s: Scene) -> dict:
    cam = s.cameras[0]
    return dict(name=s.name, n=s.n, width=cam.width, height=cam.height, views=len(s.cameras),
                sh_degree=s.sh_degree, tiles=cam.n_tiles)


# learning rates per tensor of the 3D Gaussian splatting recipe (mean3d scaled by a unit scene extent)
ADAM_LR = {"mean3d": 1.6e-4, "log_scale": 5e-3, "quat": 1e-3, "opacity": 5e-2, "sh_dc": 2.5e-3,
           "sh_rest": 2.5e-3 / 20}


def make_adam_state(n: int, deg: int, seed: int, visible_frac: float = 0.5) -> dict:
    """Seeded float32 inputs of one sparse Adam step: parameters, gradients, both moments (as after
    some earlier steps) and a visibility mask; the gradients of hidden Gaussians are zero, as the
    backward leaves them."""
    rng = _rng(10_000 + seed)
    K = (deg + 1) ** 2
    shapes = {"mean3d": (n, 3), "log_scale": (n, 3), "quat": (n, 4), "opacity_logit": (n,), "sh": (n, K, 3)}
    vis = rng.random(n) < visible_frac
    out = {"visible": vis, "params": {}, "grads": {}, "exp_avg": {}, "exp_avg_sq": {}}
    for k, shp in shapes.items():
        out["params"][k] = rng.normal(0.0, 1.0, shp).astype(np.float32)
        g = (rng.normal(0.0, 1.0, shp) * 10.0 ** rng.uniform(-6, -2, shp)).astype(np.float32)
        g[~vis] = 0.0
        out["grads"][k] = g
        out["exp_avg"][k] = (rng.normal(0.0, 1.0, shp) * 1e-3).astype(np.float32)
        out["exp_avg_sq"][k] = (rng.normal(0.0, 1.0, shp) * 1e-3).astype(np.float32) ** 2
    return out
