"""Single-Gaussian cases with closed forms (tests/golden/one_gaussian.json, written from the float64
oracle by tests/golden/make_golden.py).

Derivations (3D Gaussian splatting's projection and blending as the library and the oracle
implement them; the pages give the pipeline, DISTWAR: Fast Differentiable Rendering on Raster-based
Rendering Pipelines, Abstract):
  * Isotropic Gaussian, scale s, on the optical axis at depth z, camera R = I, t = 0: the
    projection Jacobian at the mean is diag(f/z, f/z) (x/z = y/z = 0, no clamp), so the 2D
    covariance is ((f s / z)^2 + lowpass) I: conic (1/a, 0, 1/a), a = (f s / z)^2 + 0.3, radius
    ceil(3 sqrt(a)), mean2d = (cx, cy), depth z. With f = 64, s = 1/4, z = 4: a = 16.3, radius 13;
    the mean (32.5, 32.5) is the centre of pixel (32, 32), so tiles 1..2 in x and y (4 tiles).
    Opacity sigmoid(0) = 1/2; colour (degree 0) 1/2 + Y00 c, Y00 = 1 / (2 sqrt(pi)).
    Pixel (x, y) at offset d from the mean: alpha = 1/2 exp(-(dx^2 + dy^2) / (2 a)), blended when
    >= 1/255; T = 1 - alpha; image = colour alpha + background T. By the mirror symmetry of the
    blended pixels about the mean (the support lies inside the image), dL/dmean_x = dL/dmean_y = 0,
    dL/dlog s_x = dL/dlog s_y, and dL/dquat = 0 (an isotropic Gaussian ignores its rotation); the
    depth scale s_z never reaches the projection (the Jacobian's third column vanishes on the axis),
    so dL/dlog s_z = 0.
  * One-pixel image whose centre is the projected mean (f = 1, cx = cy = 1/2, mean (0, 0, 2),
    s = 1/2): alpha = o = sigmoid(logit) (< 0.99, no clamp), I_c = rgb_c o + bg_c (1 - o). With
    L = 1/2 sum_c (I_c - t_c)^2: dL/dlogit = sum_c (I_c - t_c)(rgb_c - bg_c) o (1 - o),
    dL/dsh_c = (I_c - t_c) o Y00 (rgb unclamped), and every geometric gradient is 0 (the power's
    derivatives vanish at the mean).
The inputs are float32 (the stored log-scales and logits are rounded), so the closed forms are
evaluated from the float32 inputs in float64.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
DATA = json.load(open(os.path.join(HERE, "golden", "one_gaussian.json")))
Y00 = 0.5 / math.sqrt(math.pi)
f32 = lambda v: float(np.float32(v))


def _scene(name):
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(HERE, "golden", "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    return mg.scene_of(DATA["cases"][name]["inputs"])


def test_axis_isotropic_closed_forms():
    c = DATA["cases"]["axis_isotropic"]
    inp, o = c["inputs"], c["oracle"]
    s = math.exp(f32(inp["log_scale"][0][0]))
    a = (64.0 * s / 4.0) ** 2 + 0.3
    assert o["mean2d"][0] == pytest.approx([32.5, 32.5], abs=1e-12)
    assert o["conic"][0] == pytest.approx([1.0 / a, 0.0, 1.0 / a], rel=1e-12, abs=1e-15)
    assert o["radius"] == [math.ceil(3.0 * math.sqrt(a))] == [13]
    assert o["tiles_touched"] == [4] and o["depth"] == [4.0]
    assert o["opacity"] == [0.5]
    rgb = [0.5 + Y00 * f32(v) for v in inp["sh"][0][0]]
    assert o["rgb"][0] == pytest.approx(rgb, rel=1e-12)
    for (x, y), img, t, nc in zip(o["pixels"], o["image"], o["t_final"], o["n_contrib"]):
        dx, dy = 32.5 - (x + 0.5), 32.5 - (y + 0.5)
        alpha = 0.5 * math.exp(-(dx * dx + dy * dy) / (2.0 * a))
        blended = alpha >= 1.0 / 255.0
        assert nc == (1 if blended else 0), (x, y)
        T = 1.0 - alpha if blended else 1.0
        assert t == pytest.approx(T, rel=1e-12), (x, y)
        assert img == pytest.approx([cc * (alpha if blended else 0.0) for cc in rgb], rel=1e-12, abs=1e-15)
    # symmetry of the gradients
    dm, dls, dq = o["d_mean3d"][0], o["d_log_scale"][0], o["d_quat"][0]
    assert abs(dm[0]) <= 1e-12 * abs(dm[2]) and abs(dm[1]) <= 1e-12 * abs(dm[2]) and abs(dm[2]) > 1.0
    assert dls[0] == pytest.approx(dls[1], rel=1e-12) and dls[2] == 0.0
    assert dq == [0.0, 0.0, 0.0, 0.0]


def test_one_pixel_closed_forms():
    c = DATA["cases"]["one_pixel"]
    inp, o = c["inputs"], c["oracle"]
    s = math.exp(f32(inp["log_scale"][0][0]))
    a = (1.0 * s / 2.0) ** 2 + 0.3
    assert o["conic"][0] == pytest.approx([1.0 / a, 0.0, 1.0 / a], rel=1e-12, abs=1e-15)
    assert o["radius"] == [math.ceil(3.0 * math.sqrt(a))] == [2] and o["tiles_touched"] == [1]
    op = 1.0 / (1.0 + math.exp(-f32(inp["opacity_logit"][0])))
    assert o["opacity"][0] == pytest.approx(op, rel=1e-14)
    rgb = [0.5 + Y00 * f32(v) for v in inp["sh"][0][0]]
    bg = [f32(v) for v in inp["camera"]["bg"]]
    tgt = [f32(v) for v in inp["target_value"]]
    I = [rgb[k] * op + bg[k] * (1.0 - op) for k in range(3)]
    assert o["image"][0] == pytest.approx(I, rel=1e-12)
    assert o["t_final"] == [pytest.approx(1.0 - op, rel=1e-12)] and o["n_contrib"] == [1]
    # the oracle's upstream gradient is image - target rounded to float32
    r = [f32(I[k] - tgt[k]) for k in range(3)]
    dlogit = sum(r[k] * (rgb[k] - bg[k]) for k in range(3)) * op * (1.0 - op)
    assert o["d_opacity_logit"][0] == pytest.approx(dlogit, rel=1e-12)
    assert o["d_sh"][0][0] == pytest.approx([r[k] * op * Y00 for k in range(3)], rel=1e-12)
    assert o["d_mean3d"][0] == [0.0, 0.0, 0.0] and o["d_log_scale"][0] == [0.0, 0.0, 0.0]
    assert o["d_quat"][0] == [0.0, 0.0, 0.0, 0.0]


@pytest.mark.parametrize("name", sorted(DATA["cases"]))
def test_oracle_reproduces_the_stored_values(name):
    """Regression: the oracle's arithmetic as it stands gives the stored outputs (a change to it
    must come with a regenerated file and the reason in its commit)."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(HERE, "golden", "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    got = mg.oracle_outputs(DATA["cases"][name]["inputs"])
    want = DATA["cases"][name]["oracle"]
    for k, v in want.items():
        assert np.allclose(np.asarray(got[k], np.float64), np.asarray(v, np.float64), rtol=1e-13, atol=1e-300), k


@pytest.mark.gpu
@pytest.mark.parametrize("name", sorted(DATA["cases"]))
def test_library_matches_the_closed_form_cases(name):
    """The CUDA library's whole step on the same inputs, against the stored values: float32 work,
    so within 1e-6 relative (+1e-7 absolute) for the records, image and transmittance, 1e-5 relative
    for the non-zero gradients, and below 1e-5 of the largest gradient of the case where the stored
    value is (about) 0."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from differentiable_gaussian_splatting_gs_gb300 import _abi, api
    s = _scene(name)
    want = DATA["cases"][name]["oracle"]
    dev = torch.device("cuda:0")
    params = {k: torch.from_numpy(np.ascontiguousarray(getattr(s, k))).to(dev)
              for k in ("mean3d", "log_scale", "quat", "opacity_logit", "sh")}
    opt = api.make_options(s.sh_degree)
    cam = s.cameras[0]
    target = torch.from_numpy(s.targets[0]).to(dev)
    proj = api.gs_preprocess(params, cam, opt)
    b = api.gs_bin_and_sort(proj, cam, opt)
    image, t_final, n_contrib = api.gs_render_fwd(proj, b.vals, b.ranges, cam, opt)
    g2 = api.gs_render_bwd_sqerr(proj, b.vals, b.ranges, cam, opt, image, target, t_final, n_contrib)
    grads = api.gs_preprocess_bwd(params, cam, opt, proj, g2)
    rec = proj.rec.cpu().numpy().reshape(-1, 12)
    close = lambda got, w: np.allclose(np.asarray(got, np.float64), np.asarray(w, np.float64), rtol=1e-6, atol=1e-7)
    assert close(rec[:, 0:2], want["mean2d"]) and close(rec[:, 2:5], want["conic"])
    assert close(rec[:, 5], want["opacity"]) and close(rec[:, 6:9], want["rgb"])
    assert proj.radius.cpu().tolist() == want["radius"]
    im, tf, nc = image.cpu().numpy(), t_final.cpu().numpy(), n_contrib.cpu().numpy()
    for (x, y), img, t, n in zip(want["pixels"], want["image"], want["t_final"], want["n_contrib"]):
        assert close(im[:, y, x], img) and close(tf[y, x], t) and int(nc[y, x]) == n, (x, y)
    pairs = (("d_mean3d", "mean3d"), ("d_log_scale", "log_scale"), ("d_quat", "quat"),
             ("d_opacity_logit", "opacity_logit"), ("d_sh", "sh"))
    gscale = max(np.abs(np.asarray(want[key], np.float64)).max() for key, _ in pairs)  # the largest gradient
    for key, pk in pairs:
        got = grads[pk].cpu().numpy().reshape(-1)
        w = np.asarray(want[key], np.float64).reshape(-1)
        err = np.abs(got - w)
        ok = np.where(np.abs(w) > 1e-6 * gscale, err <= 1e-5 * np.abs(w) + 1e-7, err <= 1e-5 * gscale)
        assert ok.all(), (key, got, w)
    assert api.gs_device_error() == _abi.GS_OK
