"""Pins of the oracle's marginal-decision flags, the machinery that decides which pixels and
Gaussians the parity tests may leave out of their exact comparisons. CPU only.

A decision is marginal when a float32 evaluation could take it the other way: an alpha within its
float32 error of the 1/255 threshold, a transmittance T (1 - alpha) within its error of 1e-4, a
3-sigma radius within its error of an integer (the ceiling), a tile-rectangle boundary within the
projected mean's error of a tile edge. Two properties pin the flags:

* soundness: every decision that an independent float32 evaluation (numpy, written here from the
  arithmetic of the render and preprocess steps, with its exponential perturbed by up to two units
  in the last place to stand for a hardware approximation) takes differently from the float64
  oracle is flagged;
* tightness: decisions farther from their threshold than a small multiple of float32 rounding are
  never flagged, so a band much wider than the float32 error fails, and so does one much narrower
  (its misses show up as unflagged float32 disagreements).

The scenes are crafted so that each pixel's decisions involve only the Gaussians placed on it, at a
known relative distance delta from the threshold (log-uniform from 1e-9 to 1e-2, both signs).
The per-scene bound on the number of flagged pixels of the configuration-shaped cases is checked
here too.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

import gs_scenes
import oracle

pytestmark = pytest.mark.usefixtures("oracle_lib")

F32 = np.float32
A_MIN32 = F32(1.0) / F32(255.0)
T_MIN32 = F32(1e-4)
A_MAX32 = F32(0.99)


def _cam(W, H):
    return gs_scenes.Camera(R=np.eye(3, dtype=np.float32).reshape(9), t=np.zeros(3, np.float32), fx=100.0, fy=100.0,
                            cx=W / 2.0, cy=H / 2.0, width=W, height=H, bg=np.zeros(3, np.float32))


def _conic(sig1, sig2, theta):
    """float32 conic (A, B, C) of a 2D Gaussian with standard deviations sig1, sig2 (px) and
    principal axis at angle theta: the inverse of R diag(sig^2) R^T."""
    c, s = math.cos(theta), math.sin(theta)
    a = c * c * sig1 ** 2 + s * s * sig2 ** 2
    b = c * s * (sig1 ** 2 - sig2 ** 2)
    cc = s * s * sig1 ** 2 + c * c * sig2 ** 2
    det = a * cc - b * b
    return np.array([cc / det, -b / det, a / det], np.float32)


def _power64(mean, conic, px, py):
    dx, dy = float(mean[0]) - (px + 0.5), float(mean[1]) - (py + 0.5)
    A, B, C = (float(v) for v in conic)
    return -0.5 * (A * dx * dx + C * dy * dy) - B * dx * dy


def _crafted_scene(seed=0, W=64, H=64):
    """Pixels (i, j) with i + j even carry decisions; the others stay empty so that no Gaussian
    reaches a neighbouring decision pixel. Alpha pixels: one Gaussian whose alpha at the pixel is
    1/255 (1 + delta). Termination pixels: a stack of Gaussians blended in depth order, the last
    of which brings T (1 - alpha) to 1e-4 (1 + delta). delta is computed in float64 from the
    float32 records actually used."""
    rng = np.random.default_rng(seed)
    means, conics, opac, depth, kind, delta, owner = [], [], [], [], [], [], []
    z = 1.0
    for py in range(H):
        for px in range(W):
            if (px + py) % 2:
                continue
            sgn = 1.0 if rng.random() < 0.5 else -1.0
            d_target = sgn * 10.0 ** rng.uniform(-9, -2)
            pix = py * W + px
            if px % 4 < 2:
                # one Gaussian, alpha = opacity G at the threshold; narrow enough (sigma <= 0.12 px,
                # offset <= 0.4 px) that its alpha at the neighbouring decision pixels is ~1e-6
                off = rng.uniform(-0.4, 0.4, 2)
                cn = _conic(rng.uniform(0.08, 0.12), rng.uniform(0.08, 0.12), rng.uniform(0, math.pi))
                m = np.array([px + 0.5 + off[0], py + 0.5 + off[1]], np.float32)
                G = math.exp(_power64(m, cn, px, py))
                o = F32(float(A_MIN32) * (1.0 + d_target) / G)
                if not (0.0 < o <= 1.0):
                    continue
                alpha = float(o) * G
                means.append(m); conics.append(cn); opac.append(o); depth.append(z); z += 1e-3
                kind.append(0); delta.append(alpha / float(A_MIN32) - 1.0); owner.append(pix)
            else:
                # a stack of k Gaussians at the pixel centre (offset <= 0.05 px, sigma 0.1-0.15 px)
                k = int(rng.integers(8, 13))
                T_end = 10.0 ** rng.uniform(math.log10(1.2e-4), math.log10(5e-4))
                f = np.exp(rng.normal(0, 0.05, k - 1))
                f *= (T_end ** (1.0 / (k - 1))) / np.exp(np.mean(np.log(f)))
                recs = []
                T = 1.0
                for i in range(k):
                    off = rng.uniform(-0.05, 0.05, 2)
                    cn = _conic(rng.uniform(0.1, 0.15), rng.uniform(0.1, 0.15), rng.uniform(0, math.pi))
                    m = np.array([px + 0.5 + off[0], py + 0.5 + off[1]], np.float32)
                    G = math.exp(_power64(m, cn, px, py))
                    a_t = (1.0 - f[i]) if i < k - 1 else 1.0 - float(T_MIN32) * (1.0 + d_target) / T
                    o = F32(a_t / G)
                    if not (0.0 < o <= 1.0):
                        recs = None
                        break
                    a = min(0.99, float(o) * G)
                    recs.append((m, cn, o))
                    if i < k - 1:
                        T *= 1.0 - a
                    else:
                        d_real = T * (1.0 - a) / float(T_MIN32) - 1.0
                if recs is None:
                    continue
                for m, cn, o in recs:
                    means.append(m); conics.append(cn); opac.append(o); depth.append(z); z += 1e-3
                    kind.append(1); delta.append(d_real); owner.append(pix)
    n = len(means)
    mean2d = np.array(means, np.float32)
    radius = np.full(n, 2, np.int32)
    return dict(mean2d=mean2d, conic=np.array(conics, np.float32), opacity=np.array(opac, np.float32),
                rgb=np.full((n, 3), 0.5, np.float32), depth=np.array(depth, np.float32), radius=radius,
                kind=np.array(kind), delta=np.array(delta), owner=np.array(owner), W=W, H=H)


def _f32_blend(sc, exp_ulps: int, plain_form: bool):
    """Number of Gaussians blended at every decision pixel by a float32 evaluation: power from the
    completed square -(A u^2 + D dy^2)/2 with u = dx + (B/A) dy, D = (A C - B^2)/A (or the plain
    quadratic form), exp(power) in float32 scaled by (1 + exp_ulps 2^-23), alpha =
    min(0.99, opacity G), skip below 1/255, stop before T (1 - alpha) < 1e-4."""
    W, H = sc["W"], sc["H"]
    out = np.zeros(W * H, np.int64)
    order = np.argsort(sc["owner"], kind="stable")
    owners, starts = np.unique(sc["owner"][order], return_index=True)
    ends = np.append(starts[1:], len(order))
    pert = F32(1.0) + F32(exp_ulps) * F32(2.0 ** -23)
    for pix, s, e in zip(owners, starts, ends):
        px, py = F32(pix % W), F32(pix // W)
        T = F32(1.0)
        nb = 0
        for g in order[s:e]:
            mx, my = sc["mean2d"][g]
            A, B, C = sc["conic"][g]
            dx = mx - (px + F32(0.5))
            dy = my - (py + F32(0.5))
            if plain_form:
                power = F32(-0.5) * (A * dx * dx + C * dy * dy) - B * dx * dy
            else:
                r = B / A
                u = dx + r * dy
                D = (A * C - B * B) / A
                power = F32(-0.5) * (A * u * u + D * dy * dy)
            G = np.exp(F32(power)) * pert
            alpha = min(A_MAX32, F32(sc["opacity"][g] * G))
            if alpha < A_MIN32:
                continue
            test_T = F32(T * (F32(1.0) - alpha))
            if test_T < T_MIN32:
                break
            T = test_T
            nb += 1
        out[pix] = nb
    return out.reshape(H, W)


@pytest.fixture(scope="module")
def crafted():
    sc = _crafted_scene()
    W, H = sc["W"], sc["H"]
    _, vals, ranges = oracle.bin_and_sort(sc["mean2d"], sc["depth"], sc["radius"], W, H)
    f64 = lambda a: a.astype(np.float64)
    out = oracle.render(f64(sc["mean2d"]), f64(sc["conic"]), f64(sc["opacity"]), f64(sc["rgb"]), vals, ranges,
                        _cam(W, H))
    # the decision each pixel carries and its relative distance from the threshold
    pd = np.full(W * H, np.nan)
    pk = np.full(W * H, -1)
    for g in range(len(sc["owner"])):
        if sc["kind"][g] == 0 or g + 1 == len(sc["owner"]) or sc["owner"][g + 1] != sc["owner"][g]:
            pd[sc["owner"][g]] = sc["delta"][g]
            pk[sc["owner"][g]] = sc["kind"][g]
    return sc, out, pd.reshape(H, W), pk.reshape(H, W)


def test_crafted_decisions_span_the_float32_error_scale(crafted):
    _, _, pd, pk = crafted
    for k in (0, 1):
        d = np.abs(pd[pk == k])
        assert len(d) > 400
        assert (d < 1e-7).sum() > 30 and (d > 1e-3).sum() > 30


@pytest.mark.parametrize("plain_form", [False, True])
def test_flags_cover_every_float32_disagreement(crafted, plain_form):
    """Soundness: wherever a float32 evaluation blends a different number of Gaussians than the
    float64 oracle, the oracle has flagged the pixel."""
    sc, out, pd, pk = crafted
    flagged = out["pix_flags"] != 0
    total_mismatch = 0
    for ulps in (-2, -1, 0, 1, 2):
        nb = _f32_blend(sc, ulps, plain_form)
        mism = (nb != out["n_blended"]) & (pk >= 0)
        total_mismatch += int(mism.sum())
        assert not np.any(mism & ~flagged), (
            f"unflagged float32 disagreement at deltas {pd[mism & ~flagged][:5]}")
    # the crafted deltas reach below float32 resolution, so disagreements do occur
    assert total_mismatch > 10


def test_flags_only_near_thresholds(crafted):
    """Tightness: alpha decisions 1e-4 or more from 1/255 and termination decisions 1e-3 or more
    from 1e-4 (relative) are never flagged; decisions within 1e-8 always are."""
    _, out, pd, pk = crafted
    flagged = out["pix_flags"] != 0
    d = np.abs(pd)
    assert not np.any(flagged & (pk == 0) & (d >= 1e-4))
    assert not np.any(flagged & (pk == 1) & (d >= 1e-3))
    assert np.all(flagged[(pk >= 0) & (d <= 1e-8)])
    # bits: 1 = alpha threshold, 2 = termination
    assert np.all((out["pix_flags"][(pk == 0) & (d <= 1e-8)] & 1) != 0)
    assert np.all((out["pix_flags"][(pk == 1) & (d <= 1e-8)] & 2) != 0)


# --------------------------------------------------------------------------------- preprocess flags

def _on_axis(scales, mean_xy, z=4.0, f=100.0, W=128, H=128):
    """Axis-aligned Gaussians seen by an identity camera: Sigma' = diag((f s_x / z)^2 + 0.3, ...)
    at the optical axis; mean_xy offsets the projected mean by moving the 3D mean sideways."""
    n = len(scales)
    mean3d = np.zeros((n, 3), np.float32)
    mean3d[:, 2] = z
    mean3d[:, :2] = np.asarray(mean_xy, np.float64) * z / f
    log_scale = np.log(np.asarray(scales, np.float64)).astype(np.float32)
    quat = np.tile(np.array([1, 0, 0, 0], np.float32), (n, 1))
    logit = np.zeros(n, np.float32)
    sh = np.zeros((n, 1, 3), np.float32)
    cam = gs_scenes.Camera(R=np.eye(3, dtype=np.float32).reshape(9), t=np.zeros(3, np.float32), fx=f, fy=f,
                           cx=W / 2.0, cy=H / 2.0, width=W, height=H, bg=np.zeros(3, np.float32))
    return (mean3d, log_scale, quat, logit, sh), cam


def _f32_radius(p, cam):
    """3-sigma radius by a float32 evaluation of the on-axis covariance (x/z, y/z clamp inactive)."""
    mean3d, log_scale = p[0], p[1]
    z = mean3d[:, 2].astype(np.float32)
    s = np.exp(log_scale.astype(np.float32))
    a = (F32(cam.fx) * s[:, 0] / z) ** 2 * F32(1.0) + F32(0.3)
    c = (F32(cam.fy) * s[:, 1] / z) ** 2 + F32(0.3)
    m = F32(0.5) * (a + c)
    lam = m + np.sqrt(F32(0.25) * (a - c) ** 2)
    return np.ceil(F32(3.0) * np.sqrt(lam)).astype(np.int64)


def test_radius_flags_sound_and_tight():
    """Radii whose 3 sqrt(lambda) lies within float32 error of an integer are flagged; a float32
    evaluation that rounds to another radius is always flagged; those 1e-3 or more (relative)
    from an integer never are."""
    rng = np.random.default_rng(1)
    n = 4000
    k = rng.integers(3, 40, n).astype(np.float64)
    rel = rng.choice([-1, 1], n) * 10.0 ** rng.uniform(-9, -2, n)
    target = k * (1.0 + rel)                       # 3 sqrt(lambda)
    fs = np.sqrt(np.maximum((target / 3.0) ** 2 - 0.3, 1e-6))  # f s / z
    s = fs * 4.0 / 100.0
    p, cam = _on_axis(np.stack([s, s * 0.5, s * 0.5], 1), np.zeros((n, 2)))
    pre = oracle.preprocess(*p, 0, cam)
    # the distance actually realised by the float32 scale, in float64
    s32 = np.exp(p[1].astype(np.float64))
    real = 3.0 * np.sqrt((100.0 * s32[:, 0] / 4.0) ** 2 + 0.3)
    d = np.abs(real - np.round(real)) / real
    flagged = (pre["flags"] & 2) != 0
    assert not np.any(flagged & (d >= 1e-3))
    assert np.all(flagged[d <= 1e-9])
    r32 = _f32_radius(p, cam)
    mism = r32 != pre["radius"]
    assert mism.sum() > 5 and not np.any(mism & ~flagged)


def test_rectangle_flags_sound_and_tight():
    """Tile-rectangle boundaries: the rectangle starts at tile ceil((x - 0.5 - r - 15) / 16); a mean
    whose boundary lies within float32 error of a tile edge is flagged, one 0.01 px or more from
    it is not."""
    rng = np.random.default_rng(2)
    n = 4000
    r_target = 4  # 3 sqrt(lambda) = 3.5 on the axis, at most about 3.7 at the largest offsets used
    fs = math.sqrt((3.5 / 3.0) ** 2 - 0.3)
    s = fs * 4.0 / 100.0
    edge = 16.0 * rng.integers(2, 6, n) + r_target + 15.5    # boundary position of the projected mean
    off = rng.choice([-1, 1], n) * 10.0 ** rng.uniform(-8, -1, n)
    mx = edge + off - 64.0                                 # relative to the principal point
    p, cam = _on_axis(np.tile([s, s, s], (n, 1)), np.stack([mx, np.zeros(n)], 1))
    pre = oracle.preprocess(*p, 0, cam)
    assert np.all(pre["radius"] == r_target)
    real = pre["mean2d"][:, 0]
    dist = np.abs(real - (np.round((real - r_target - 15.5) / 16.0) * 16.0 + r_target + 15.5))
    flagged = (pre["flags"] & 4) != 0
    assert not np.any(flagged & (dist >= 1e-2))
    assert np.all(flagged[dist <= 1e-6])
    # a float32 projected mean (x / z computed in float32) crossing the edge is flagged
    m32 = (F32(100.0) * (p[0][:, 0] / p[0][:, 2]) + F32(64.0)).astype(np.float64)
    side64 = np.floor((real - 0.5 - r_target - 15.0) / 16.0)
    side32 = np.floor((m32 - 0.5 - r_target - 15.0) / 16.0)
    mism = side32 != side64
    assert mism.sum() > 5 and not np.any(mism & ~flagged)


# --------------------------------------------------------------------------------- scene-level bound

@pytest.mark.parametrize("name", ["tiny", "object", "outdoor", "large", "contention"])
def test_flagged_pixels_are_rare_in_the_configuration_scenes(name):
    """The marginal set is about one pixel per million evaluated (pixel, Gaussian) pairs: the
    oracle flags at most 2e-6 of the evaluated pairs (+3). On the scenes with fewer than 300
    pairs evaluated per pixel that is within 1e-4 of the pixels (+3)."""
    import _cases
    d = _cases.stage_inputs(name)
    f, st = d["fwd"], d["stats"]
    P = f["pix_flags"].size
    nf = int((f["pix_flags"] != 0).sum())
    q = st["pairs_evaluated"]
    assert nf <= 2e-6 * q + 3, (nf, q)
    if q < 300 * P:
        assert nf <= 1e-4 * P + 3, (nf, P)
