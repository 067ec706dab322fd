"""Pins of the oracle's surfel (2D Gaussian splatting) functions, independent of their formulas:
closed forms for a splat facing the camera, the ray-plane intersection against a direct ray cast,
the bounding box against Monte Carlo projection of the 3-sigma circle, and end-to-end central
finite differences from the 3D parameters."""
import numpy as np
import pytest

import gs_scenes
import oracle


def _single(mean, log_scale, quat, f=100.0, w=64, h=48, logit=0.0, deg=0):
    s = gs_scenes.make_scene_random_small(seed=1, n=1, width=w, height=h, f=f, deg=deg)
    s.mean3d = np.asarray([mean], np.float64)
    s.log_scale = np.asarray([log_scale], np.float64)
    s.quat = np.asarray([quat], np.float64)
    s.opacity_logit = np.asarray([logit], np.float64)
    s.sh = s.sh.astype(np.float64)
    return s


def test_facing_splat_closed_forms():
    z, su, sv = 3.0, 0.05, 0.02
    s = _single([0.0, 0.0, z], [np.log(su), np.log(sv), 0.0], [1.0, 0.0, 0.0, 0.0])
    cam = s.cameras[0]
    pre = oracle.preprocess2d(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, 0, cam)
    r = pre["rec2d"][0]
    f = cam.fx
    assert np.allclose(r[:9], [su * f, 0, 0, 0, sv * f, 0, cam.cx, cam.cy, z], rtol=1e-14, atol=1e-14)
    assert np.allclose(r[9:11], [cam.cx, cam.cy], rtol=1e-14)  # the box is centred on the projection
    assert np.allclose(pre["half"][0], [3 * f * su / z, 3 * f * sv / z], rtol=1e-12)
    # the render: one surfel, every pixel's weight is max(disk Gaussian, screen filter)
    out = oracle.view_step2d(s)
    img = out["fwd"]["image"][0]
    o = 1 / (1 + np.exp(-0.0))
    c0 = (s.sh[0, 0, 0] * 0.28209479177387814 + 0.5)
    ys, xs = np.mgrid[0:cam.height, 0:cam.width] + 0.5
    sx, sy = f * su / z, f * sv / z
    p3 = -0.5 * (((xs - cam.cx) / sx) ** 2 + ((ys - cam.cy) / sy) ** 2)
    plp = -((xs - cam.cx) ** 2 + (ys - cam.cy) ** 2)
    a = np.minimum(0.99, o * np.exp(np.maximum(p3, plp)))
    a = np.where(a >= np.float32(1 / 255), a, 0.0)
    # pixels of the tiles that list the surfel (the binning is pinned with the 3D rasterizer)
    listed = (out["ranges"][:, 1] > out["ranges"][:, 0]).reshape((cam.height + 15) // 16, (cam.width + 15) // 16)
    inside = np.kron(listed, np.ones((16, 16), bool))[:cam.height, :cam.width]
    assert inside.sum() >= 256 and pre["radius"][0] == 5
    assert np.allclose(img, np.where(inside, a * max(c0, 0.0), 0.0), atol=1e-12)


def test_ray_plane_intersection_matches_a_direct_ray_cast():
    rng = np.random.default_rng(4)
    for trial in range(20):
        mean = np.array([rng.uniform(-0.5, 0.5), rng.uniform(-0.4, 0.4), rng.uniform(2, 5)])
        q = rng.normal(size=4)
        ls = np.log(rng.uniform(0.03, 0.2, 3))
        s = _single(mean, ls, q)
        cam = s.cameras[0]
        pre = oracle.preprocess2d(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, 0, cam)
        if pre["radius"][0] == 0:
            continue
        R = oracle.quat_to_rotmat(q / np.linalg.norm(q))
        tu, tv = R[:, 0] * np.exp(ls[0]), R[:, 1] * np.exp(ls[1])
        rec = pre["rec2d"][:1].copy()
        vals = np.zeros(1, np.uint32)
        ranges = np.zeros((((cam.height + 15) // 16) * ((cam.width + 15) // 16), 2), np.uint32)
        ranges[:, 1] = 1  # every tile lists the surfel
        rec[0, 11] = 0.5  # opacity
        rec[0, 12:15] = 1.0
        img = oracle.render2d(rec, vals, ranges, cam)["image"][0]
        for _ in range(30):
            px, py = rng.integers(0, cam.width), rng.integers(0, cam.height)
            d = np.array([(px + 0.5 - cam.cx) / cam.fx, (py + 0.5 - cam.cy) / cam.fy, 1.0])  # camera ray
            # mean + u tu + v tv = t d  ->  [tu, tv, -d] (u, v, t) = -mean
            u, v, _ = np.linalg.solve(np.stack([tu, tv, -d], axis=1), -mean)
            p3 = -0.5 * (u * u + v * v)
            cxb, cyb = pre["mean2d"][0]
            plp = -((px + 0.5 - cxb) ** 2 + (py + 0.5 - cyb) ** 2)
            a = min(0.99, 0.5 * np.exp(max(p3, plp)))
            expect = a if a >= np.float32(1 / 255) else 0.0
            assert abs(img[py, px] - expect) < 1e-9, (trial, px, py)


def test_bounding_box_is_the_projection_of_the_3_sigma_circle():
    rng = np.random.default_rng(5)
    th = np.linspace(0, 2 * np.pi, 200001)
    for trial in range(10):
        mean = np.array([rng.uniform(-0.3, 0.3), rng.uniform(-0.3, 0.3), rng.uniform(2, 4)])
        q = rng.normal(size=4)
        ls = np.log(rng.uniform(0.05, 0.3, 3))
        s = _single(mean, ls, q)
        cam = s.cameras[0]
        pre = oracle.preprocess2d(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, 0, cam)
        if pre["radius"][0] == 0:
            continue
        R = oracle.quat_to_rotmat(q / np.linalg.norm(q))
        P = mean[:, None] + 3 * (np.exp(ls[0]) * R[:, :1] * np.cos(th) + np.exp(ls[1]) * R[:, 1:2] * np.sin(th))
        x = cam.fx * P[0] / P[2] + cam.cx
        y = cam.fy * P[1] / P[2] + cam.cy
        c, hf = pre["mean2d"][0], pre["half"][0]
        assert np.allclose([x.min(), x.max()], [c[0] - hf[0], c[0] + hf[0]], atol=1e-6 * (1 + hf[0]))
        assert np.allclose([y.min(), y.max()], [c[1] - hf[1], c[1] + hf[1]], atol=1e-6 * (1 + hf[1]))


def _chain2d(s, cam, g=None):
    pre = oracle.preprocess2d(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, s.sh_degree, cam)
    _, vals, ranges = oracle.bin_and_sort(pre["mean2d"].astype(np.float32), pre["depth"], pre["radius"], cam.width,
                                          cam.height)
    out = oracle.render2d(pre["rec2d"], vals, ranges, cam, g)
    return pre, vals, out


@pytest.mark.parametrize("deg", [0, 3])
def test_surfel_end_to_end_gradients_match_central_differences(deg):
    s = gs_scenes.make_scene_random_small(seed=200 + deg, n=25, width=32, height=32, f=40.0, deg=deg,
                                          log_scale_mu=-2.0, bg=(0.2, 0.3, 0.1))
    for name in ("mean3d", "log_scale", "quat", "opacity_logit", "sh"):
        setattr(s, name, getattr(s, name).astype(np.float64))
    cam = s.cameras[0]
    g = np.random.default_rng(9).standard_normal((3, cam.height, cam.width)).astype(np.float32)
    pre, vals, out = _chain2d(s, cam, g)
    gr = oracle.preprocess2d_bwd(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, s.sh_degree, cam, out["grad"])
    base = (pre["radius"].copy(), out["pix_sig"].copy(), vals.copy())
    checked = skipped = 0
    for pname, gname in [("mean3d", "d_mean3d"), ("log_scale", "d_log_scale"), ("quat", "d_quat"),
                         ("opacity_logit", "d_opacity_logit"), ("sh", "d_sh")]:
        flat = getattr(s, pname).reshape(-1)
        an_all = gr[gname].reshape(-1)
        scale = np.abs(an_all).max()
        for k in range(flat.size):
            x0 = float(flat[k])
            # step: rounding noise of the 3 x 32 x 32 sum / h against curvature error ~ h^2
            h = 1e-5 * max(abs(x0), 1e-2)
            flat[k] = x0 + h
            pp, vp, op = _chain2d(s, cam)
            flat[k] = x0 - h
            pm, vm, om = _chain2d(s, cam)
            flat[k] = x0
            same = all(np.array_equal(a, b) for a, b in [(pp["radius"], base[0]), (pm["radius"], base[0]),
                                                         (op["pix_sig"], base[1]), (om["pix_sig"], base[1]),
                                                         (vp, base[2]), (vm, base[2])])
            if not same:
                skipped += 1
                continue
            fd = (float(np.sum(op["image"] * g)) - float(np.sum(om["image"] * g))) / (2 * h)
            assert abs(fd - an_all[k]) <= 1e-6 * abs(an_all[k]) + 1e-7 * scale + 1e-9, (pname, k, fd, an_all[k])
            checked += 1
    assert checked > 0.9 * (checked + skipped)
    assert np.all(gr["d_log_scale"][:, 2] == 0)  # the third scale has no role for a surfel
