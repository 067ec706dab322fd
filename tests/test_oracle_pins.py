"""Pins of the float64 oracle to things other than itself: closed forms, library routines
(scipy spherical harmonics and rotations), Monte Carlo of the exact pinhole projection,
brute-force tile enumeration and sorting, the brute-force renderer, invariants of the blending
recursion, and central finite differences of the whole forward. CPU only.
"""
import math

import numpy as np
import pytest

import gs_scenes
import oracle
from oracle import brute

pytestmark = pytest.mark.usefixtures("oracle_lib")

A_MIN = float(np.float32(1.0) / np.float32(255.0))
T_MIN = float(np.float32(1e-4))


def _cam(width, height, f, R=None, t=None, bg=(0.0, 0.0, 0.0), cx=None, cy=None):
    return gs_scenes.Camera(R=np.eye(3, dtype=np.float32).reshape(9) if R is None else np.asarray(R, np.float32).reshape(9),
                            t=np.zeros(3, np.float32) if t is None else np.asarray(t, np.float32),
                            fx=float(f), fy=float(f), cx=width / 2.0 if cx is None else cx,
                            cy=height / 2.0 if cy is None else cy, width=width, height=height,
                            bg=np.asarray(bg, np.float32))


def _one(mean, log_scale, quat=(1, 0, 0, 0), logit=0.0, colour=(0.5, 0.5, 0.5)):
    sh = np.zeros((1, 1, 3))
    sh[0, 0] = (np.asarray(colour) - 0.5) * 2.0 * math.sqrt(math.pi)
    return (np.asarray([mean], np.float64), np.asarray([log_scale], np.float64),
            np.asarray([quat], np.float64), np.asarray([logit], np.float64), sh)


# ---------------------------------------------------------------- spherical harmonics

def test_sh_dc_constant_closed_form():
    for d in ([0, 0, 1], [1, 2, 3], [-1, 0.2, -0.3]):
        assert oracle.sh_basis(0, d)[0] == pytest.approx(1.0 / (2.0 * math.sqrt(math.pi)), abs=1e-15)


def test_sh_matches_scipy_complex_harmonics():
    from scipy.special import sph_harm_y
    rng = np.random.default_rng(7)
    for _ in range(50):
        v = rng.standard_normal(3)
        v /= np.linalg.norm(v)
        theta = math.acos(v[2])          # polar
        phi = math.atan2(v[1], v[0])     # azimuth
        Y = oracle.sh_basis(3, v)
        for l in range(4):
            for m in range(0, l + 1):
                c = complex(sph_harm_y(l, m, theta, phi))
                if m == 0:
                    assert Y[l * l + l] == pytest.approx(c.real, abs=1e-12)
                else:
                    assert Y[l * l + l + m] == pytest.approx(math.sqrt(2) * c.real, abs=1e-12)
                    assert Y[l * l + l - m] == pytest.approx(math.sqrt(2) * c.imag, abs=1e-12)


def test_sh_orthonormal_by_quadrature():
    zs, wz = np.polynomial.legendre.leggauss(12)
    n_phi = 24
    G = np.zeros((16, 16))
    for z, w in zip(zs, wz):
        s = math.sqrt(1 - z * z)
        for k in range(n_phi):
            phi = 2 * math.pi * k / n_phi
            Y = oracle.sh_basis(3, [s * math.cos(phi), s * math.sin(phi), z])
            G += np.outer(Y, Y) * w * (2 * math.pi / n_phi)
    np.testing.assert_allclose(G, np.eye(16), atol=1e-12)


# ---------------------------------------------------------------- rotations / covariance

def test_quaternion_matches_scipy_rotation():
    from scipy.spatial.transform import Rotation
    rng = np.random.default_rng(3)
    for _ in range(20):
        q = rng.standard_normal(4)
        R = oracle.quat_to_rotmat(q)
        ref = Rotation.from_quat([q[1], q[2], q[3], q[0]]).as_matrix()  # scipy is scalar-last
        np.testing.assert_allclose(R, ref, atol=1e-12)


@pytest.mark.parametrize("z", [2.0, 7.5])
def test_projection_closed_form_on_axis(z):
    f, W, H = 300.0, 64, 48
    sx, sy, sz = 0.05, 0.02, 0.3
    m, ls, q, lg, sh = _one([0, 0, z], np.log([sx, sy, sz]))
    out = oracle.preprocess(m, ls, q, lg, sh, 0, _cam(W, H, f))
    a_ref = (f * sx / z) ** 2 + 0.3
    c_ref = (f * sy / z) ** 2 + 0.3
    np.testing.assert_allclose(out["cov2d"][0], [a_ref, 0.0, c_ref], rtol=1e-6, atol=1e-12)
    np.testing.assert_allclose(out["mean2d"][0], [W / 2, H / 2], atol=1e-12)
    np.testing.assert_allclose(out["conic"][0], [1 / a_ref, 0.0, 1 / c_ref], rtol=1e-6, atol=1e-12)
    assert out["radius"][0] == math.ceil(3 * math.sqrt(max(a_ref, c_ref)))
    assert out["depth"][0] == np.float32(z)
    assert out["opacity"][0] == pytest.approx(0.5)
    np.testing.assert_allclose(out["rgb"][0], [0.5, 0.5, 0.5], atol=1e-7)


def test_projection_rot90_about_z_swaps_axes():
    f, W, H, z = 300.0, 64, 48, 3.0
    sx, sy = 0.05, 0.02
    c45 = math.cos(math.pi / 4)
    m, ls, q, lg, sh = _one([0, 0, z], np.log([sx, sy, 0.1]), quat=(c45, 0, 0, c45))
    out = oracle.preprocess(m, ls, q, lg, sh, 0, _cam(W, H, f))
    a_ref = (f * sy / z) ** 2 + 0.3
    c_ref = (f * sx / z) ** 2 + 0.3
    np.testing.assert_allclose(out["cov2d"][0], [a_ref, 0.0, c_ref], rtol=1e-6, atol=1e-9)


def test_projection_matches_monte_carlo_of_exact_pinhole():
    """The EWA covariance is the covariance of the exactly projected samples of a small Gaussian
    (first order in its size), for a rotated, translated camera and an off-axis, rotated Gaussian."""
    from scipy.spatial.transform import Rotation
    rng = np.random.default_rng(11)
    Rcam = Rotation.from_euler("xyz", [0.2, -0.3, 0.15]).as_matrix().astype(np.float32)
    tcam = np.asarray([0.3, -0.2, 1.0], np.float32)
    cam = _cam(640, 480, 500.0, R=Rcam, t=tcam)
    mean_cam = np.array([0.8, -0.5, 6.0])
    mean = (Rcam.T.astype(np.float64) @ (mean_cam - tcam)).astype(np.float32)
    scales = np.array([0.004, 0.0015, 0.003])
    qv = rng.standard_normal(4)
    qv /= np.linalg.norm(qv)
    m, ls, q, lg, sh = _one(mean, np.log(scales), quat=qv)
    out = oracle.preprocess(m, ls, q, lg, sh, 0, cam, jacobian_clamp=0.0)
    Rq = Rotation.from_quat([qv[1], qv[2], qv[3], qv[0]]).as_matrix()
    n = 400_000
    eps = rng.standard_normal((n, 3)) * np.exp(ls[0].astype(np.float64))
    pw = m[0].astype(np.float64) + eps @ Rq.T
    pc = pw @ Rcam.T.astype(np.float64) + tcam.astype(np.float64)
    uv = np.stack([cam.fx * pc[:, 0] / pc[:, 2] + cam.cx, cam.fy * pc[:, 1] / pc[:, 2] + cam.cy], 1)
    cov = np.cov(uv.T)
    a, b, c = out["cov2d"][0]
    np.testing.assert_allclose([a - 0.3, b, c - 0.3], [cov[0, 0], cov[0, 1], cov[1, 1]],
                               rtol=0.02, atol=0.02 * math.sqrt(cov[0, 0] * cov[1, 1]))
    np.testing.assert_allclose(out["mean2d"][0], uv.mean(0), atol=0.01)


def test_depth_key_is_view_space_depth():
    rng = np.random.default_rng(5)
    from scipy.spatial.transform import Rotation
    R = Rotation.from_euler("xyz", [0.1, 0.2, -0.1]).as_matrix().astype(np.float32)
    t = np.asarray([0.1, 0.2, 0.5], np.float32)
    mean = rng.uniform(-1, 1, (200, 3)).astype(np.float32)
    mean[:, 2] += 4
    n = len(mean)
    out = oracle.preprocess(mean, np.full((n, 3), -3, np.float32), np.tile([1, 0, 0, 0], (n, 1)).astype(np.float32),
                            np.zeros(n, np.float32), np.zeros((n, 1, 3), np.float32), 0, _cam(64, 64, 64, R=R, t=t))
    exact = mean.astype(np.float64) @ R[2].astype(np.float64) + float(t[2])
    assert np.all(np.abs(out["depth"] - exact) <= 2 * np.spacing(np.float32(exact)))
    out0 = oracle.preprocess(mean, np.full((n, 3), -3, np.float32), np.tile([1, 0, 0, 0], (n, 1)).astype(np.float32),
                             np.zeros(n, np.float32), np.zeros((n, 1, 3), np.float32), 0, _cam(64, 64, 64))
    assert np.array_equal(out0["depth"], mean[:, 2])


def test_culling_near_plane_and_behind():
    mean = np.asarray([[0, 0, 0.1], [0, 0, -2.0], [0, 0, 0.25], [50, 0, 1.0]], np.float32)
    n = len(mean)
    out = oracle.preprocess(mean, np.full((n, 3), -4, np.float32), np.tile([1, 0, 0, 0], (n, 1)).astype(np.float32),
                            np.zeros(n, np.float32), np.zeros((n, 1, 3), np.float32), 0, _cam(64, 64, 64))
    assert list(out["radius"] > 0) == [False, False, True, False]
    assert list(out["flags"] & 1) == [1, 1, 0, 1]
    assert out["tiles_touched"][0] == 0 and out["tiles_touched"][2] > 0


# ---------------------------------------------------------------- binning and sort

def _brute_tiles(mx, my, r, W, H):
    TX, TY = (W + 15) // 16, (H + 15) // 16
    xh, yh = float(mx) - 0.5, float(my) - 0.5
    cols = [tx for tx in range(TX) if any(abs(i - xh) <= r for i in range(16 * tx, 16 * tx + 16))]
    rows = [ty for ty in range(TY) if any(abs(j - yh) <= r for j in range(16 * ty, 16 * ty + 16))]
    return [ty * TX + tx for ty in rows for tx in cols]


@pytest.mark.parametrize("W,H", [(64, 48), (77, 35), (16, 16)])
def test_binning_matches_brute_force_enumeration(W, H):
    rng = np.random.default_rng(W * 1000 + H)
    n = 400
    mean2d = np.stack([rng.uniform(-30, W + 30, n), rng.uniform(-30, H + 30, n)], 1).astype(np.float32)
    mean2d[:20] = np.round(mean2d[:20]) + 0.5        # centres exactly on pixel centres
    radius = rng.integers(0, 25, n).astype(np.int32)
    depth = rng.uniform(1, 3, n).astype(np.float32)
    depth[50:80] = depth[50]                          # ties in depth: index order decides
    keys, vals, ranges = oracle.bin_and_sort(mean2d, depth, radius, W, H)
    entries = []
    for g in range(n):
        if radius[g] <= 0:
            continue
        for t in _brute_tiles(mean2d[g, 0], mean2d[g, 1], int(radius[g]), W, H):
            entries.append((t, int(depth[g:g + 1].view(np.uint32)[0]), g))
    entries.sort()
    assert len(entries) == len(vals)
    assert [e[2] for e in entries] == vals.tolist()
    assert [(e[0] << 32) | e[1] for e in entries] == keys.tolist()
    T = ((W + 15) // 16) * ((H + 15) // 16)
    for t in range(T):
        idx = [i for i, e in enumerate(entries) if e[0] == t]
        if idx:
            assert (ranges[t, 0], ranges[t, 1]) == (idx[0], idx[-1] + 1)
        else:
            assert ranges[t, 0] == ranges[t, 1]


# ---------------------------------------------------------------- forward

def _records_2d(n, W, H, rng, depth_ties=False):
    mean2d = np.stack([rng.uniform(-10, W + 10, n), rng.uniform(-10, H + 10, n)], 1)
    L = rng.uniform(0.5, 6.0, (n, 2))
    rho = rng.uniform(-0.8, 0.8, n)
    a, c = L[:, 0] ** 2 + 0.3, L[:, 1] ** 2 + 0.3
    b = rho * L[:, 0] * L[:, 1]
    det = a * c - b * b
    conic = np.stack([c / det, -b / det, a / det], 1)
    radius = np.ceil(3 * np.sqrt(0.5 * (a + c) + np.sqrt(0.25 * (a - c) ** 2 + b * b))).astype(np.int32)
    opacity = rng.uniform(0.05, 1.0, n)
    opacity[: n // 10] = 1.0                      # alpha clamped at 0.99 near their centres
    rgb = rng.uniform(0, 1, (n, 3))
    depth = rng.uniform(1, 5, n).astype(np.float32)
    if depth_ties:
        depth[::3] = depth[0]
    return mean2d, conic, opacity, rgb, depth, radius


@pytest.mark.parametrize("W,H,n,seed", [(48, 32, 150, 0), (37, 29, 300, 1), (64, 64, 600, 2)])
def test_forward_matches_brute_force(W, H, n, seed):
    rng = np.random.default_rng(seed)
    mean2d, conic, opacity, rgb, depth, radius = _records_2d(n, W, H, rng, depth_ties=True)
    m32 = mean2d.astype(np.float32)
    _, vals, ranges = oracle.bin_and_sort(m32, depth, radius, W, H)
    cam = _cam(W, H, 100.0, bg=(0.2, 0.4, 0.6))
    out = oracle.render(m32.astype(np.float64), conic, opacity, rgb, vals, ranges, cam)
    img, tf, nc = brute.render(m32.astype(np.float64), conic, opacity, rgb, depth, radius, m32, W, H, cam.bg)
    np.testing.assert_allclose(out["image"], img, atol=1e-12)
    np.testing.assert_allclose(out["t_final"], tf, atol=1e-12)
    assert np.array_equal(out["n_contrib"], nc)


def test_forward_matches_brute_force_on_tiny_config_subset():
    s = gs_scenes.make_scene(0, n=300, res_scale=0.5)
    cam = s.cameras[0]
    pre = oracle.preprocess(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, 0, cam)
    m32 = pre["mean2d"].astype(np.float32)
    _, vals, ranges = oracle.bin_and_sort(m32, pre["depth"], pre["radius"], cam.width, cam.height)
    out = oracle.render(pre["mean2d"], pre["conic"], pre["opacity"], pre["rgb"], vals, ranges, cam)
    img, tf, nc = brute.render(pre["mean2d"], pre["conic"], pre["opacity"], pre["rgb"], pre["depth"],
                               pre["radius"], m32, cam.width, cam.height, cam.bg)
    np.testing.assert_allclose(out["image"], img, atol=1e-12)
    assert np.array_equal(out["n_contrib"], nc)


def test_blending_weights_and_transmittance_invariants():
    rng = np.random.default_rng(4)
    W, H, n = 64, 48, 800
    mean2d, conic, opacity, _, depth, radius = _records_2d(n, W, H, rng)
    _, vals, ranges = oracle.bin_and_sort(mean2d.astype(np.float32), depth, radius, W, H)
    out = oracle.render(mean2d.astype(np.float32).astype(np.float64), conic, opacity, np.ones((n, 3)), vals,
                        ranges, _cam(W, H, 50.0))
    # sum_i alpha_i T_i + T_final = 1 (the weights of a front-to-back blend of white on black)
    np.testing.assert_allclose(out["image"][0] + out["t_final"], 1.0, atol=1e-12)
    assert np.all(out["t_final"] >= T_MIN) and np.all(out["t_final"] <= 1.0)
    assert np.all((out["n_blended"] > 0) == (out["t_final"] < 1.0))
    assert np.all(out["n_contrib"] >= out["n_blended"])


def _stack_records(n, opacity, W=32, H=32, at=(8.5, 8.5)):
    mean2d = np.tile(np.asarray(at, np.float64), (n, 1))
    conic = np.tile([1e-9, 0.0, 1e-9], (n, 1))
    radius = np.full(n, 40, np.int32)
    depth = (1.0 + np.arange(n)).astype(np.float32)
    return mean2d, conic, np.asarray(opacity, np.float64), depth, radius


def test_termination_closed_form():
    """Stacked Gaussians of alpha 1/2: T after k blends is 2^-k; the 14th would take T below 1e-4,
    so exactly 13 are blended and the contributor count is 13."""
    n = 20
    mean2d, conic, opacity, depth, radius = _stack_records(n, np.full(n, 0.5))
    rgb = np.tile([0.9, 0.5, 0.1], (n, 1))
    _, vals, ranges = oracle.bin_and_sort(mean2d.astype(np.float32), depth, radius, 32, 32)
    cam = _cam(32, 32, 50.0, bg=(0.1, 0.2, 0.3))
    out = oracle.render(mean2d, conic, opacity, rgb, vals, ranges, cam)
    T13 = 0.5 ** 13
    assert out["n_contrib"][8, 8] == 13 and out["n_blended"][8, 8] == 13
    assert out["t_final"][8, 8] == pytest.approx(T13, rel=1e-6)
    np.testing.assert_allclose(out["image"][:, 8, 8], np.array([0.9, 0.5, 0.1]) * (1 - T13) + T13 * cam.bg,
                               rtol=1e-6)


def test_alpha_threshold_and_clamp_closed_form():
    # entry 0: alpha just below 1/255 (skipped), entry 1: just above (blended), entry 2: opacity 1
    # (alpha clamped to 0.99), entry 3 would take T below 1e-4 and is not blended.
    mean2d, conic, _, depth, radius = _stack_records(4, np.zeros(4))
    G = math.exp(-0.5 * 1e-9 * 0.0)  # pixel centre exactly at the mean: G = 1
    opacity = np.array([A_MIN * (1 - 1e-6), A_MIN * (1 + 1e-6), 1.0, 1.0]) / G
    rgb = np.tile([1.0, 1.0, 1.0], (4, 1))
    _, vals, ranges = oracle.bin_and_sort(mean2d.astype(np.float32), depth, radius, 32, 32)
    out = oracle.render(mean2d, conic, opacity, rgb, vals, ranges, _cam(32, 32, 50.0))
    a1 = opacity[1]
    T_after = (1 - a1) * (1 - 0.99)
    assert out["n_contrib"][8, 8] == 3 and out["n_blended"][8, 8] == 2
    assert out["t_final"][8, 8] == pytest.approx(T_after, rel=1e-12)


def test_single_isotropic_gaussian_closed_form():
    """One isotropic Gaussian on the optical axis: sigma^2 = (f s / z)^2 + 0.3 and
    pixel = c alpha(d) + (1 - alpha(d)) bg with alpha(d) = min(0.99, o exp(-d^2 / (2 sigma^2)))
    inside its tile rectangle; and the analytic gradients of sum(g * pixel)."""
    f, W, H, z, s_ = 120.0, 48, 40, 3.0, 0.08
    logit, colour, bg = 1.5, np.array([0.8, 0.3, 0.6]), np.array([0.1, 0.2, 0.05])
    m, ls, q, lg, sh = _one([0, 0, z], np.log([s_] * 3), logit=logit, colour=colour)
    cam = _cam(W, H, f, bg=bg)
    bg = cam.bg.astype(np.float64)          # the camera carries the background in float32
    pre = oracle.preprocess(m, ls, q, lg, sh, 0, cam)
    sig2 = (f * float(np.exp(ls[0, 0])) / z) ** 2 + 0.3
    o = 1 / (1 + math.exp(-float(lg[0])))
    r = math.ceil(3 * math.sqrt(sig2))
    assert pre["radius"][0] == r
    _, vals, ranges = oracle.bin_and_sort(pre["mean2d"].astype(np.float32), pre["depth"], pre["radius"], W, H)
    rng = np.random.default_rng(0)
    g = rng.standard_normal((3, H, W)).astype(np.float32)
    out = oracle.render(pre["mean2d"], pre["conic"], pre["opacity"], pre["rgb"], vals, ranges, cam, dl_dimage=g)
    ys, xs = np.mgrid[0:H, 0:W]
    dx, dy = W / 2 - (xs + 0.5), H / 2 - (ys + 0.5)
    G = np.exp(-(dx * dx + dy * dy) / (2 * sig2))
    alpha = np.minimum(0.99, o * G)
    xh, yh = W / 2 - 0.5, H / 2 - 0.5
    in_rect = ((xs // 16 >= math.ceil((xh - r - 15) / 16)) & (xs // 16 <= math.floor((xh + r) / 16)) &
               (ys // 16 >= math.ceil((yh - r - 15) / 16)) & (ys // 16 <= math.floor((yh + r) / 16)))
    used = in_rect & (alpha >= A_MIN)
    a = np.where(used, alpha, 0.0)
    ref = colour[:, None, None] * a + (1 - a) * bg[:, None, None]
    np.testing.assert_allclose(out["image"], ref, atol=1e-12)
    # gradients: dL/drgb = sum g alpha; dL/do = sum g.(c - bg) G; dL/dmean_x = sum g.(c - bg) o G (-dx / sigma^2)
    unclamped = used & (o * G <= 0.99)
    gcb = np.einsum("chw,c->hw", g.astype(np.float64), colour - bg)
    d_rgb = np.einsum("chw,hw->c", g.astype(np.float64), a)
    d_o = np.sum(np.where(unclamped, gcb * G, 0.0))
    d_mx = np.sum(np.where(unclamped, gcb * o * G * (-dx / sig2), 0.0))
    d_A = np.sum(np.where(unclamped, gcb * o * G * (-0.5 * dx * dx), 0.0))
    g2 = out["grad2d"][0]
    np.testing.assert_allclose(g2[6:9], d_rgb, rtol=1e-9)
    assert g2[5] == pytest.approx(d_o, rel=1e-9)
    assert g2[0] == pytest.approx(d_mx, rel=1e-9, abs=1e-9)
    assert g2[2] == pytest.approx(d_A, rel=1e-9)


# ---------------------------------------------------------------- finite differences

def _loss_2d(mean2d, conic, opacity, rgb, vals, ranges, cam, g):
    out = oracle.render(mean2d, conic, opacity, rgb, vals, ranges, cam)
    return float(np.sum(out["image"] * g)), out["pix_sig"], out["n_contrib"]


def test_raster_backward_matches_central_differences():
    rng = np.random.default_rng(21)
    W, H, n = 32, 32, 40
    mean2d, conic, opacity, rgb, depth, radius = _records_2d(n, W, H, rng)
    mean2d = mean2d.astype(np.float32).astype(np.float64)
    _, vals, ranges = oracle.bin_and_sort(mean2d.astype(np.float32), depth, radius, W, H)
    cam = _cam(W, H, 50.0, bg=(0.3, 0.1, 0.7))
    g = rng.standard_normal((3, H, W)).astype(np.float32)
    an = oracle.render(mean2d, conic, opacity, rgb, vals, ranges, cam, dl_dimage=g)["grad2d"]
    base_sig = oracle.render(mean2d, conic, opacity, rgb, vals, ranges, cam)["pix_sig"]
    fields = [(mean2d, 0), (mean2d, 1), (conic, 0), (conic, 1), (conic, 2), (opacity, None),
              (rgb, 0), (rgb, 1), (rgb, 2)]
    checked = skipped = 0
    for gi in range(n):
        for j, (arr, col) in enumerate(fields):
            idx = (gi,) if col is None else (gi, col)
            x0 = arr[idx]
            h = 1e-6 * max(abs(x0), 1e-2)
            arr[idx] = x0 + h
            lp, sp, _ = _loss_2d(mean2d, conic, opacity, rgb, vals, ranges, cam, g)
            arr[idx] = x0 - h
            lm, sm, _ = _loss_2d(mean2d, conic, opacity, rgb, vals, ranges, cam, g)
            arr[idx] = x0
            if not (np.array_equal(sp, base_sig) and np.array_equal(sm, base_sig)):
                skipped += 1
                continue
            fd = (lp - lm) / (2 * h)
            assert abs(fd - an[gi, j]) <= 1e-6 * max(1.0, abs(an[gi, j])) + 1e-6 * np.abs(an[:, j]).max(), \
                (gi, j, fd, an[gi, j])
            checked += 1
    assert checked > 0.9 * (checked + skipped)


def _chain(s, cam):
    pre = oracle.preprocess(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, s.sh_degree, cam)
    m32 = pre["mean2d"].astype(np.float32)
    _, vals, ranges = oracle.bin_and_sort(m32, pre["depth"], pre["radius"], cam.width, cam.height)
    out = oracle.render(pre["mean2d"], pre["conic"], pre["opacity"], pre["rgb"], vals, ranges, cam)
    return pre, vals, ranges, out


@pytest.mark.parametrize("deg", [0, 3])
def test_end_to_end_gradients_match_central_differences(deg):
    """Central differences of sum(g * image) through preprocess, binning and render, in float64,
    against the preprocess backward applied to the render backward."""
    s = gs_scenes.make_scene_random_small(seed=100 + deg, n=25, width=32, height=32, f=40.0, deg=deg,
                                          log_scale_mu=-2.3, bg=(0.2, 0.3, 0.1))
    for name in ("mean3d", "log_scale", "quat", "opacity_logit", "sh"):
        setattr(s, name, getattr(s, name).astype(np.float64))
    cam = s.cameras[0]
    rng = np.random.default_rng(9)
    g = rng.standard_normal((3, cam.height, cam.width)).astype(np.float32)
    pre, vals, ranges, out = _chain(s, cam)
    bwd = oracle.render(pre["mean2d"], pre["conic"], pre["opacity"], pre["rgb"], vals, ranges, cam, dl_dimage=g)
    gr = oracle.preprocess_bwd(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, s.sh_degree, cam, bwd["grad2d"])
    base = (pre["radius"].copy(), out["pix_sig"].copy(), vals.copy())
    params = [("mean3d", "d_mean3d"), ("log_scale", "d_log_scale"), ("quat", "d_quat"),
              ("opacity_logit", "d_opacity_logit"), ("sh", "d_sh")]
    checked = skipped = 0
    for pname, gname in params:
        flat = getattr(s, pname).reshape(-1)
        an_all = gr[gname].reshape(-1)
        scale = np.abs(an_all).max()
        for k in range(flat.size):
            x0 = float(flat[k])
            h = 1e-6 * max(abs(x0), 1e-2)
            flat[k] = x0 + h
            pp, rp, _, op = _chain(s, cam)
            flat[k] = x0 - h
            pm, rm, _, om = _chain(s, cam)
            flat[k] = x0
            same = all(np.array_equal(a, b) for a, b in
                       [(pp["radius"], base[0]), (pm["radius"], base[0]), (op["pix_sig"], base[1]),
                        (om["pix_sig"], base[1]), (rp, base[2]), (rm, base[2])])
            if not same:
                skipped += 1
                continue
            fd = (float(np.sum(op["image"] * g)) - float(np.sum(om["image"] * g))) / (2 * h)
            assert abs(fd - an_all[k]) <= 1e-6 * abs(an_all[k]) + 1e-7 * scale + 1e-9, (pname, k, fd, an_all[k])
            checked += 1
    assert checked > 0.9 * (checked + skipped)


def test_backward_sums_do_not_depend_on_the_thread_count():
    """Per-Gaussian gradient sums are formed per tile and added in tile order: the same bits with
    one, three or eight threads."""
    rng = np.random.default_rng(7)
    W, H, n = 96, 80, 700
    mean2d, conic, opacity, rgb, depth, radius = _records_2d(n, W, H, rng)
    m32 = mean2d.astype(np.float32)
    _, vals, ranges = oracle.bin_and_sort(m32, depth, radius, W, H)
    g = rng.standard_normal((3, H, W)).astype(np.float32)
    outs = [oracle.render(m32.astype(np.float64), conic, opacity, rgb, vals, ranges, _cam(W, H, 50.0), dl_dimage=g,
                          threads=t)["grad2d"] for t in (1, 3, 8)]
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])
