"""GPU parity of the surfel (2D Gaussian splatting) path against the float64 oracle, stage by stage
as for the 3D path: each stage gets the oracle's previous outputs rounded to float32.

Tolerances: the step's bars, as for the 3D path: pixels within 1e-5 where the oracle flags no
alpha or termination decision within 1e-4 of its threshold, and every gradient tensor within 1e-4
of its largest magnitude, with the upstream gradient zeroed on flagged pixels (a decision that
legitimately differs moves every gradient of its pixel). Record fields are products and quotients
of a few float32 values: 2e-6 of each field's largest magnitude over the scene; the box centre is
the projected mean plus a quotient of dual-conic entries and enters only through the tile
rectangle and the screen filter: 1e-3 px.
"""
import functools

import numpy as np
import pytest
import torch

import gs_scenes
import oracle

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from differentiable_gaussian_splatting_gs_gb300 import api  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")

# the last case is the 1.6M-surfel 1297x840 scene at full size, in the launch configuration the
# benchmark's surfel step uses
CASES2D = {"tiny": (0, None, 1.0), "object": (1, 20_000, 1.0), "outdoor": (2, 100_000, 0.5),
           "outdoor_full": (2, None, 1.0)}


@functools.lru_cache(maxsize=None)
def _case(name):
    cfg, n, rs = CASES2D[name]
    s = gs_scenes.make_scene(cfg, n=n, res_scale=rs)
    cam = s.cameras[0]
    pre = oracle.preprocess2d(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, s.sh_degree, cam)
    rec32 = pre["rec2d"].astype(np.float32)
    c32 = pre["mean2d"].astype(np.float32)
    _, vals, ranges = oracle.bin_and_sort(c32, pre["depth"], pre["radius"], cam.width, cam.height)
    fwd = oracle.render2d(rec32.astype(np.float64), vals, ranges, cam)
    dl = (fwd["image"] - s.targets[0]).astype(np.float32)
    dl_m = np.where(fwd["pix_flags"][None] != 0, 0.0, dl).astype(np.float32)
    bwd_m = oracle.render2d(rec32.astype(np.float64), vals, ranges, cam, dl_m)
    g32 = bwd_m["grad"].astype(np.float32)
    g3 = oracle.preprocess2d_bwd(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, s.sh_degree, cam, g32)
    return s, cam, pre, rec32, c32, vals, ranges, fwd, dl_m, bwd_m, g32, g3


def _params(s):
    return {k: torch.from_numpy(np.ascontiguousarray(getattr(s, k))).to(DEV) for k in
            ("mean3d", "log_scale", "quat", "opacity_logit", "sh")}


def _ranges_dev(ranges):
    return torch.from_numpy(ranges.astype(np.int32)).to(DEV)


@pytest.mark.parametrize("name", list(CASES2D))
def test_surfel_preprocess_matches_oracle(name):
    s, cam, pre, *_ = _case(name)
    proj, rec2d = api.gs_preprocess2d(_params(s), cam, api.make_options(s.sh_degree))
    torch.cuda.synchronize()
    r = rec2d.cpu().numpy().astype(np.float64)
    rad = proj.radius.cpu().numpy()
    depth = proj.depth.cpu().numpy()
    assert np.array_equal(depth, pre["depth"])
    half = pre["half"]
    hm = np.maximum(half.max(axis=1), 3 * np.sqrt(0.5))
    marginal = np.abs(hm - np.round(hm)) < 1e-4 * np.maximum(hm, 1)  # ceil boundary of the radius
    ok = ~marginal
    assert np.array_equal(rad[ok], pre["radius"][ok]), (rad[ok] != pre["radius"][ok]).sum()
    vis = (pre["radius"] > 0) & (rad > 0) & ok
    o = pre["rec2d"]
    for f in range(9):  # A, B, C (u, v), m, z
        scale = np.abs(o[vis, f]).max()
        assert np.abs(r[vis, f] - o[vis, f]).max() <= 2e-6 * scale, (name, f)
    assert np.abs(r[vis, 9:11] - o[vis, 9:11]).max() <= 1e-3  # box centre (px)
    assert np.allclose(r[vis, 11:15], o[vis, 11:15], rtol=1e-5, atol=1e-6)  # opacity, colour
    assert api.gs_device_error() == 0


@pytest.mark.parametrize("name", list(CASES2D))
def test_surfel_render_forward_matches_oracle(name):
    s, cam, pre, rec32, c32, vals, ranges, fwd, *_ = _case(name)
    image, t_final, n_contrib = api.gs_render2d_fwd(torch.from_numpy(rec32).to(DEV),
                                                    torch.from_numpy(vals.astype(np.int32)).to(DEV),
                                                    _ranges_dev(ranges), cam, api.make_options(s.sh_degree))
    torch.cuda.synchronize()
    # the pixel value is continuous where the two exponents cross (flag 4): only the alpha and
    # termination decisions (flags 1, 2) can move a pixel by more than rounding
    ok = (fwd["pix_flags"] & 3) == 0
    assert (~ok).sum() <= max(3, 1e-2 * ok.size)
    err = np.abs(image.cpu().numpy() - fwd["image"])
    assert err[:, ok].max() <= 1e-5, err[:, ok].max()
    assert np.array_equal(n_contrib.cpu().numpy().astype(np.uint32)[ok], fwd["n_contrib"][ok])
    assert api.gs_device_error() == 0


@pytest.mark.parametrize("name", list(CASES2D))
@pytest.mark.parametrize("mode", ["adaptive", "direct", "warp"])
def test_surfel_render_backward_matches_oracle(name, mode):
    s, cam, pre, rec32, c32, vals, ranges, fwd, dl_m, bwd_m, *_ = _case(name)
    opt = api.make_options(s.sh_degree, bwd_mode=mode)
    r = torch.from_numpy(rec32).to(DEV)
    v = torch.from_numpy(vals.astype(np.int32)).to(DEV)
    rg = _ranges_dev(ranges)
    _, t_final, n_contrib = api.gs_render2d_fwd(r, v, rg, cam, opt)
    grad = api.gs_render2d_bwd(r, v, rg, cam, opt, torch.from_numpy(dl_m).to(DEV), t_final, n_contrib)
    torch.cuda.synchronize()
    g = grad.cpu().numpy().astype(np.float64)
    ref = bwd_m["grad"]
    for lo, hi in [(0, 3), (3, 6), (6, 8), (8, 9), (9, 11), (11, 12), (12, 15)]:
        scale = np.abs(ref[:, lo:hi]).max()
        err = np.abs(g[:, lo:hi] - ref[:, lo:hi]).max()
        assert err <= 1e-4 * scale + 1e-12, (name, mode, lo, err / max(scale, 1e-30))
    assert np.all(g[:, 15] == 0)
    assert api.gs_device_error() == 0


@pytest.mark.parametrize("name", list(CASES2D))
def test_surfel_preprocess_backward_matches_oracle(name):
    s, cam, pre, rec32, c32, vals, ranges, fwd, dl_m, bwd_m, g32, g3 = _case(name)
    params = _params(s)
    opt = api.make_options(s.sh_degree)
    proj, _ = api.gs_preprocess2d(params, cam, opt)
    # both sides see the oracle's visibility (the GPU's may differ on marginal radii only)
    proj.radius.copy_(torch.from_numpy(pre["radius"]))
    out = api.gs_preprocess2d_bwd(params, cam, opt, proj, torch.from_numpy(g32).to(DEV))
    torch.cuda.synchronize()
    for k, ok in [("mean3d", "d_mean3d"), ("log_scale", "d_log_scale"), ("quat", "d_quat"),
                  ("opacity_logit", "d_opacity_logit"), ("sh", "d_sh")]:
        a = out[k].cpu().numpy().astype(np.float64)
        b = g3[ok]
        scale = np.abs(b).max()
        assert np.abs(a - b).max() <= 1e-4 * scale + 1e-12, (name, k, np.abs(a - b).max() / max(scale, 1e-30))
    assert api.gs_device_error() == 0


def test_surfel_empty_and_all_culled():
    opt = api.make_options(0)
    cam = gs_scenes.make_scene(0).cameras[0]
    empty = {k: torch.empty((0,) + shp, dtype=torch.float32, device=DEV)
             for k, shp in (("mean3d", (3,)), ("log_scale", (3,)), ("quat", (4,)), ("opacity_logit", ()),
                            ("sh", (1, 3)))}
    proj, rec2d = api.gs_preprocess2d(empty, cam, opt)
    assert proj.n == 0 and rec2d.shape == (0, 16)
    s = gs_scenes.make_scene(0, n=500)
    s.mean3d[:, 2] = -1.0  # everything behind the camera
    params = _params(s)
    proj, rec2d = api.gs_preprocess2d(params, cam, opt)
    assert int(proj.radius.max()) == 0 and int(proj.tiles_touched.max()) == 0
    assert float(rec2d.abs().max()) == 0.0
    b = api.gs_bin_and_sort(proj, cam, opt)
    assert b.n_dup == 0 and int(b.ranges.abs().max()) == 0
    img, tf, nc = api.gs_render2d_fwd(rec2d, b.vals, b.ranges, cam, opt)
    bg = torch.tensor(cam.bg, dtype=torch.float32, device=DEV)[:, None, None].expand_as(img)
    assert torch.equal(img, bg) and float(tf.min()) == 1.0 and int(nc.max()) == 0
    grad = api.gs_render2d_bwd(rec2d, b.vals, b.ranges, cam, opt, torch.ones_like(img), tf, nc)
    assert float(grad.abs().max()) == 0.0
    out = api.gs_preprocess2d_bwd(params, cam, opt, proj, grad)
    assert all(float(t.abs().max()) == 0.0 for t in out.values())
    assert api.gs_device_error() == 0


def test_surfel_backward_rejects_shared_memory_mode():
    s, cam, pre, rec32, c32, vals, ranges, fwd, dl_m, *_ = _case("tiny")
    opt = api.make_options(s.sh_degree, bwd_mode="sm")
    r = torch.from_numpy(rec32).to(DEV)
    v = torch.from_numpy(vals.astype(np.int32)).to(DEV)
    _, t_final, n_contrib = api.gs_render2d_fwd(r, v, _ranges_dev(ranges), cam, opt)
    with pytest.raises(api.GsError, match="GS_BWD_SM"):
        api.gs_render2d_bwd(r, v, _ranges_dev(ranges), cam, opt, torch.from_numpy(dl_m).to(DEV), t_final, n_contrib)


def test_surfel_preprocess_backward_accumulates_views():
    """Two views of the multi-view scene: the second call with accumulate adds to the first; the
    sum equals the sum of the oracle's per-view gradients."""
    s = gs_scenes.make_scene(3, n=20_000, res_scale=0.25, views=2)
    params = _params(s)
    opt = api.make_options(s.sh_degree)
    grads, want = None, None
    for v, cam in enumerate(s.cameras):
        pre = oracle.preprocess2d(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, s.sh_degree, cam)
        _, vals, ranges = oracle.bin_and_sort(pre["mean2d"].astype(np.float32), pre["depth"], pre["radius"],
                                              cam.width, cam.height)
        rec = pre["rec2d"].astype(np.float32).astype(np.float64)
        fwd = oracle.render2d(rec, vals, ranges, cam)
        dl = np.where(fwd["pix_flags"][None] != 0, 0.0, fwd["image"] - s.targets[v]).astype(np.float32)
        g32 = oracle.render2d(rec, vals, ranges, cam, dl)["grad"].astype(np.float32)
        proj, _ = api.gs_preprocess2d(params, cam, opt)
        proj.radius.copy_(torch.from_numpy(pre["radius"]))
        grads = api.gs_preprocess2d_bwd(params, cam, opt, proj, torch.from_numpy(g32).to(DEV), out=grads,
                                        accumulate=v > 0)
        o = oracle.preprocess2d_bwd(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, s.sh_degree, cam, g32)
        want = o if want is None else {k: want[k] + o[k] for k in o}
    torch.cuda.synchronize()
    for k, ok in [("mean3d", "d_mean3d"), ("log_scale", "d_log_scale"), ("quat", "d_quat"),
                  ("opacity_logit", "d_opacity_logit"), ("sh", "d_sh")]:
        a = grads[k].cpu().numpy().astype(np.float64)
        b = want[ok]
        assert np.abs(a - b).max() <= 1e-4 * np.abs(b).max() + 1e-12, k
    assert api.gs_device_error() == 0
