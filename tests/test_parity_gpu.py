"""Parity of the CUDA library (through its C ABI) with the float64 oracle, stage by stage and end
to end, on seeded scenes shaped like the five configurations (smaller sizes that span many tiles
and a ragged image edge) plus edge cases. The full-size configurations are in
test_full_size_gpu.py.

Bars: bit-exact for depth keys, duplicate counts, sorted (tile, depth, index) lists, tile ranges
and contributor counts (outside the oracle's marginal decisions); 1e-5 max abs error on pixels;
1e-4 of max|grad| per gradient tensor. The oracle flags at most 5e-6 of the evaluated (pixel,
Gaussian) pairs as marginal (+3), and at most 1e-4 of the pixels (+3) on scenes with fewer than
300 evaluated pairs per pixel.
"""
from __future__ import annotations

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import gs_scenes  # noqa: E402
import oracle  # noqa: E402
from differentiable_gaussian_splatting_gs_gb300 import _abi, api, step  # noqa: E402

import _gpu_checks as gc  # noqa: E402
from _cases import (CASES, GRAD2D_GROUPS, GRAD_KEYS, PARAM_NAMES, grad_close, grad_close_mag, scene,  # noqa: E402
                    stage_inputs)

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
MODES = ["direct", "warp", "adaptive", "sm"]
STAGINGS = [_abi.GS_STAGE_BULK, _abi.GS_STAGE_LOADS]


def u32(t):
    return t.detach().cpu().numpy().view(np.uint32)


def dev_params(s):
    return {k: torch.from_numpy(np.ascontiguousarray(getattr(s, k))).to(DEV) for k in PARAM_NAMES}


def dev_proj(rec):
    return api.proj_from_arrays(rec["mean2d"], rec["conic"], rec["opacity"], rec["rgb"], rec["depth"], rec["radius"],
                                DEV)


@pytest.fixture(autouse=True)
def _no_device_errors():
    yield
    assert api.gs_device_error() == _abi.GS_OK, "device error word set"


# --------------------------------------------------------------------------------- bounded wait

def test_bounded_wait_gives_up_and_reports_timeout():
    lib = _abi.load()
    assert lib.gs_selftest_timeout(64, None) == 0
    assert api.gs_device_error() == _abi.GS_ERR_TIMEOUT
    assert api.gs_device_error() == _abi.GS_OK  # cleared, context still usable
    x = torch.arange(10, device=DEV).sum().item()
    assert x == 45


@pytest.mark.parametrize("spin", [1, 64])
def test_sort_lookback_gives_up_and_reports_timeout(spin):
    """The depth sort's look-back, with a predecessor block that never publishes, gives up after
    `spin` polls: the device error word reports GS_ERR_TIMEOUT, the block still places its items
    (within its buffers), and the next sort is exact."""
    lib = _abi.load()
    ws = torch.full((_abi.GS_SELFTEST_SORT_WORKSPACE_BYTES // 4,), 7, dtype=torch.int32, device=DEV)
    assert lib.gs_selftest_sort_timeout(ws.data_ptr(), ws.numel() * 4, spin, None) == 0
    assert api.gs_device_error() == _abi.GS_ERR_TIMEOUT
    assert api.gs_device_error() == _abi.GS_OK
    # the block's 4096 items (keys 0, values 4096..8191 in order) landed at positions 0..4095
    vals_out = ws[2 * 8192: 3 * 8192].cpu().numpy()
    assert np.array_equal(vals_out[:4096], np.arange(4096, 8192))
    # too small a workspace is rejected on the host
    assert lib.gs_selftest_sort_timeout(ws.data_ptr(), 1024, spin, None) == _abi.GS_ERR_ARG
    d = stage_inputs("tiny")
    b = api.gs_bin_and_sort(dev_proj(d["rec"]), d["cam"], api.make_options(0))
    assert np.array_equal(u32(b.vals), d["vals"])


# --------------------------------------------------------------------------------- preprocess

@pytest.mark.parametrize("name", list(CASES))
def test_preprocess_matches_oracle(name):
    d = stage_inputs(name)
    gc.check_preprocess(d["scene"], d["cam"], d["pre"])


def test_preprocess_empty_and_all_culled():
    opt = api.make_options(0)
    cam = gs_scenes.make_scene(0).cameras[0]
    empty = {k: torch.empty((0,) + shp, dtype=torch.float32, device=DEV)
             for k, shp in (("mean3d", (3,)), ("log_scale", (3,)), ("quat", (4,)), ("opacity_logit", ()),
                            ("sh", (1, 3)))}
    proj = api.gs_preprocess(empty, cam, opt)
    assert proj.n == 0
    s = gs_scenes.make_scene(0, n=500)
    s.mean3d[:, 2] = -1.0  # everything behind the camera
    proj = api.gs_preprocess(dev_params(s), cam, opt)
    assert int(proj.radius.max()) == 0 and int(proj.tiles_touched.max()) == 0
    b = api.gs_bin_and_sort(proj, cam, opt)
    assert b.n_dup == 0 and int(b.ranges.abs().max()) == 0
    img, tf, nc = api.gs_render_fwd(proj, b.vals, b.ranges, cam, opt)
    assert float(img.abs().max()) == 0.0 and float(tf.min()) == 1.0 and int(nc.max()) == 0


# --------------------------------------------------------------------------------- binning / sort

def _check_bin(rec, cam, b):
    keys, vals, ranges = oracle.bin_and_sort(rec["mean2d"], rec["depth"], rec["radius"], cam.width, cam.height)
    assert b.n_dup == len(vals)
    assert np.array_equal(u32(b.vals), vals)
    if b.keys is not None:
        assert np.array_equal(b.keys.cpu().numpy().view(np.uint64), keys)
    assert np.array_equal(u32(b.ranges), ranges)


@pytest.mark.parametrize("name", list(CASES))
def test_bin_and_sort_bit_exact(name):
    d = stage_inputs(name)
    proj = dev_proj(d["rec"])
    b = api.gs_bin_and_sort(proj, d["cam"], api.make_options(d["scene"].sh_degree))
    assert b.n_dup == len(d["vals"])
    assert np.array_equal(u32(b.vals), d["vals"])
    assert np.array_equal(b.keys.cpu().numpy().view(np.uint64), d["keys"])
    assert np.array_equal(u32(b.ranges), d["ranges"])


@pytest.mark.parametrize("W,H,n", [(16, 16, 300), (17, 9, 200), (200, 120, 3000), (4112, 4112, 400)])
def test_bin_and_sort_tile_pass_counts_and_ties(W, H, n):
    """Single tile (no tile pass), ragged edges, one and two passes, and > 65536 tiles (three
    passes); a third of the depths tie exactly, so index order decides."""
    rng = np.random.default_rng(W * 7 + H)
    mean2d = np.stack([rng.uniform(-40, W + 40, n), rng.uniform(-40, H + 40, n)], 1).astype(np.float32)
    mean2d[: n // 10] = np.floor(mean2d[: n // 10]) + 0.5
    radius = rng.integers(0, min(60, 2 * max(W, H)), n).astype(np.int32)
    depth = rng.uniform(1, 3, n).astype(np.float32)
    depth[::3] = depth[0]
    rec = dict(mean2d=mean2d, conic=np.tile([0.1, 0.0, 0.1], (n, 1)), opacity=np.full(n, 0.5),
               rgb=np.full((n, 3), 0.5), depth=depth, radius=radius)
    cam = gs_scenes.Camera(R=np.eye(3, dtype=np.float32).reshape(9), t=np.zeros(3, np.float32), fx=100.0, fy=100.0,
                           cx=W / 2, cy=H / 2, width=W, height=H, bg=np.zeros(3, np.float32))
    b = api.gs_bin_and_sort(dev_proj(rec), cam, api.make_options(0))
    _check_bin(rec, cam, b)


def test_bin_and_sort_capacity_error_reports_required_size():
    d = stage_inputs("tiny")
    proj = dev_proj(d["rec"])
    with pytest.raises(_abi.GsError) as ei:
        api.gs_bin_and_sort(proj, d["cam"], api.make_options(0), capacity=10)
    assert ei.value.status == _abi.GS_ERR_CAPACITY
    b = api.gs_bin_and_sort(proj, d["cam"], api.make_options(0), capacity=len(d["vals"]))
    assert np.array_equal(u32(b.vals), d["vals"])


def test_bin_and_sort_without_keys():
    d = stage_inputs("object")
    b = api.gs_bin_and_sort(dev_proj(d["rec"]), d["cam"], api.make_options(3), want_keys=False)
    assert b.keys is None and np.array_equal(u32(b.vals), d["vals"])


# --------------------------------------------------------------------------------- forward

def _fwd(d, staging):
    proj = dev_proj(d["rec"])
    opt = api.make_options(d["scene"].sh_degree, staging=staging)
    b = api.gs_bin_and_sort(proj, d["cam"], opt)
    img, tf, nc = api.gs_render_fwd(proj, b.vals, b.ranges, d["cam"], opt)
    return proj, b, opt, img, tf, nc


@pytest.mark.parametrize("staging", STAGINGS)
@pytest.mark.parametrize("name", list(CASES))
def test_render_fwd_matches_oracle(name, staging):
    d = stage_inputs(name)
    _, _, _, img, tf, nc = _fwd(d, staging)
    f = d["fwd"]
    ok = f["pix_flags"] == 0
    gc.check_flag_count(f["pix_flags"], d["stats"]["pairs_evaluated"])
    if d["stats"]["pairs_evaluated"] < 300 * ok.size:
        assert (~ok).sum() <= 1e-4 * ok.size + 3, f"{(~ok).sum()} marginal pixels"
    err = np.abs(img.cpu().numpy() - f["image"])
    assert err[:, ok].max() <= 1e-5, err[:, ok].max()
    assert np.array_equal(u32(nc)[ok], f["n_contrib"][ok])
    assert np.allclose(tf.cpu().numpy()[ok], f["t_final"][ok], rtol=1e-4, atol=1e-7)
    # marginal pixels differ at most by the last Gaussian's contribution
    assert err.max() <= 0.02


# --------------------------------------------------------------------------------- backward

@pytest.mark.parametrize("staging", STAGINGS)
@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("name", list(CASES))
def test_render_bwd_matches_oracle(name, mode, staging):
    d = stage_inputs(name)
    proj, b, _, img, tf, nc = _fwd(d, staging)
    opt = api.make_options(d["scene"].sh_degree, bwd_mode=mode, staging=staging)
    # upstream gradient zero on the oracle's marginal pixels: the 1e-4 bar
    g2 = api.gs_render_bwd(proj, b.vals, b.ranges, d["cam"], opt, torch.from_numpy(d["dl_masked"]).to(DEV), tf, nc)
    got = g2.cpu().numpy()
    assert np.all(got[:, 9:] == 0.0)
    for group, cols in GRAD2D_GROUPS.items():
        ok, err, tol = grad_close(got[:, cols], d["grad2d_masked"][:, cols])
        assert ok, f"{group}: error {err:.3g} > {tol:.3g}"
    # full upstream gradient: marginal pixels may move sums a little more
    got = api.gs_render_bwd(proj, b.vals, b.ranges, d["cam"], opt, torch.from_numpy(d["dl"]).to(DEV), tf,
                            nc).cpu().numpy()
    for group, cols in GRAD2D_GROUPS.items():
        ok, err, tol = grad_close(got[:, cols], d["grad2d"][:, cols], rel=1e-2)
        assert ok, f"unmasked {group}: error {err:.3g} > {tol:.3g}"


@pytest.mark.parametrize("mode", ["adaptive", "direct"])
@pytest.mark.parametrize("name", list(CASES))
def test_render_bwd_sqerr_matches_oracle(name, mode):
    """The backward that forms dL/dimage = image - target itself: given the oracle's image (rounded
    to float32) and the target, with the target set to the image on the flagged pixels (zero
    gradient there), it matches the oracle's backward at 1e-4 of max and reports the loss
    0.5 sum (image - target)^2 within 1e-5 relative."""
    d = stage_inputs(name)
    proj, b, _, img, tf, nc = _fwd(d, _abi.GS_STAGE_BULK)
    image32 = d["fwd"]["image"].astype(np.float32)
    target = np.where(d["fwd"]["pix_flags"][None] != 0, image32, d["scene"].targets[d["view"]]).astype(np.float32)
    loss = torch.zeros(1, device=DEV)
    g2 = api.gs_render_bwd_sqerr(proj, b.vals, b.ranges, d["cam"], api.make_options(d["scene"].sh_degree, bwd_mode=mode),
                                 torch.from_numpy(image32).to(DEV), torch.from_numpy(target).to(DEV), tf, nc,
                                 loss=loss).cpu().numpy()
    for group, cols in GRAD2D_GROUPS.items():
        ok, err, tol = grad_close(g2[:, cols], d["grad2d_masked"][:, cols])
        assert ok, f"{group}: error {err:.3g} > {tol:.3g}"
    want = 0.5 * float(((image32.astype(np.float64) - target) ** 2).sum())
    assert float(loss.item()) == pytest.approx(want, rel=1e-5)


@pytest.mark.parametrize("thr", [1, 16, 33])
def test_adaptive_threshold_extremes(thr):
    d = stage_inputs("contention")
    proj, b, _, img, tf, nc = _fwd(d, _abi.GS_STAGE_BULK)
    for mode in ("adaptive", "sm"):
        opt = api.make_options(0, bwd_mode=mode, adaptive_threshold=thr)
        got = api.gs_render_bwd(proj, b.vals, b.ranges, d["cam"], opt, torch.from_numpy(d["dl_masked"]).to(DEV), tf,
                                nc).cpu().numpy()
        for group, cols in GRAD2D_GROUPS.items():
            ok, err, tol = grad_close(got[:, cols], d["grad2d_masked"][:, cols])
            assert ok, f"{mode}/{thr}/{group}: {err:.3g} > {tol:.3g}"


# --------------------------------------------------------------------------------- preprocess backward

@pytest.mark.parametrize("name", list(CASES))
def test_preprocess_bwd_matches_oracle(name):
    d = stage_inputs(name)
    gc.check_preprocess_bwd(d["scene"], d["cam"], d["pre"], d["grad2d32"], d["grads"])


def test_preprocess_bwd_accumulates_views():
    s, _ = scene("large")
    params = dev_params(s)
    opt = api.make_options(s.sh_degree)
    grads = api.alloc_param_grads(params)
    want = None
    for v, cam in enumerate(s.cameras):
        g2n = np.random.default_rng(v).standard_normal((s.n, 9)).astype(np.float32)
        proj = api.gs_preprocess(params, cam, opt)
        g2 = torch.zeros((s.n, 12), dtype=torch.float32, device=DEV)
        g2[:, :9] = torch.from_numpy(g2n).to(DEV)
        api.gs_preprocess_bwd(params, cam, opt, proj, g2, out=grads, accumulate=v > 0)
        o = oracle.preprocess_bwd(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, s.sh_degree, cam, g2n)
        o.pop("mag")
        want = o if want is None else {k: want[k] + o[k] for k in o}
    for name_p in PARAM_NAMES:
        got = grads[name_p].cpu().numpy().reshape(s.n, -1)
        ok, err, tol = grad_close(got, want[GRAD_KEYS[name_p]].reshape(s.n, -1))
        assert ok, f"{name_p}: {err:.3g} > {tol:.3g}"


def _offset_copy(t):
    """A contiguous copy of t whose data starts 4 bytes past a 16-byte boundary."""
    buf = torch.zeros(t.numel() + 4, dtype=t.dtype, device=t.device)
    v = buf[1:1 + t.numel()].view(t.shape)
    v.copy_(t)
    assert v.data_ptr() % 16 == 4
    return v


@pytest.mark.parametrize("deg", [0, 1, 2, 3])
def test_preprocess_sh_layouts_match_oracle(deg):
    """Every SH degree, with the SH arrays 16-byte aligned (for degrees 1 and 3 the rows then move
    through the bulk-copy engine, and the gradient rows back by bulk copies or bulk additions) and
    4 bytes past a 16-byte boundary (coalesced 4-byte copies). Both layouts against the oracle and
    against each other: depths bit for bit, radii exactly off the oracle's marginal Gaussians, the
    records and the gradients of one view within 1e-5 of each field's largest magnitude (the
    kernels may contract different multiply-adds), and a second, accumulated view doubling every
    gradient exactly. A seventh of the Gaussians sit behind the camera (culled: no SH row is read,
    their gradient rows are written as zeros)."""
    s = gs_scenes.make_scene_random_small(40 + deg, 3000, 200, 136, 180.0, deg)
    s.mean3d[::7, 2] = -1.0
    cam = s.cameras[0]
    pre = oracle.preprocess(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, deg, cam)
    assert 0 < int((pre["radius"] > 0).sum()) < s.n
    g2n = np.random.default_rng(deg).standard_normal((s.n, 9)).astype(np.float32)
    want = oracle.preprocess_bwd(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, deg, cam, g2n)
    opt = api.make_options(deg)
    res = {}
    for layout in ("aligned", "offset"):
        params = dev_params(s)
        if layout == "offset":
            params["sh"] = _offset_copy(params["sh"])
        gc.check_preprocess(s, cam, pre, params=params)
        gc.check_preprocess_bwd(s, cam, pre, g2n, want, params=params)
        proj = api.gs_preprocess(params, cam, opt)
        g2 = torch.zeros((s.n, 12), dtype=torch.float32, device=DEV)
        g2[:, :9] = torch.from_numpy(g2n).to(DEV)
        grads = api.alloc_param_grads(params)
        if layout == "offset":
            grads["sh"] = _offset_copy(grads["sh"])
        api.gs_preprocess_bwd(params, cam, opt, proj, g2, out=grads)
        once = {k: v.clone() for k, v in grads.items()}
        api.gs_preprocess_bwd(params, cam, opt, proj, g2, out=grads, accumulate=True)
        res[layout] = ((proj.rec.clone(), proj.depth.clone(), proj.radius.clone()), once, grads)
    (ra, oa, ga), (rb, ob, gb) = res["aligned"], res["offset"]
    steady = torch.from_numpy((pre["flags"] & oracle.MARGINAL) == 0).to(DEV)
    assert torch.equal(ra[1], rb[1]) and torch.equal(ra[2][steady], rb[2][steady])
    rec_a, rec_b = ra[0].reshape(s.n, -1), rb[0].reshape(s.n, -1)
    assert bool(((rec_a - rec_b).abs() <= 1e-5 * rec_a.abs().amax(0)).all())
    culled = torch.from_numpy(pre["radius"] == 0).to(DEV)
    for k in PARAM_NAMES:
        assert float((oa[k] - ob[k]).abs().max()) <= 1e-5 * float(oa[k].abs().max()), k
        for once, acc in ((oa, ga), (ob, gb)):
            assert torch.equal(acc[k], 2 * once[k]), k
            assert int(once[k][culled].count_nonzero()) == 0, k


@pytest.mark.parametrize("n", [1, 31, 33, 4097])
def test_preprocess_bulk_rows_ragged_sizes_and_all_culled(n):
    """The bulk-copy preprocess kernels (degree 3, aligned arrays, persistent grids) on group counts
    that are not multiples of the grid, a last group of 1..31 Gaussians, and a scene with every
    Gaussian behind the camera (no row is copied, every gradient row is written as zeros, and
    accumulating adds nothing)."""
    s = gs_scenes.make_scene_random_small(70 + n, n, 96, 80, 90.0, 3)
    cam = s.cameras[0]
    pre = oracle.preprocess(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, 3, cam)
    g2n = np.random.default_rng(n).standard_normal((s.n, 9)).astype(np.float32)
    want = oracle.preprocess_bwd(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, 3, cam, g2n)
    gc.check_preprocess(s, cam, pre)
    gc.check_preprocess_bwd(s, cam, pre, g2n, want)
    s.mean3d[:, 2] = -1.0  # everything culled
    params = dev_params(s)
    opt = api.make_options(3)
    proj = api.gs_preprocess(params, cam, opt)
    assert int(proj.radius.abs().max()) == 0 and float(proj.rec.abs().max()) == 0.0
    g2 = torch.from_numpy(np.pad(g2n, ((0, 0), (0, 3)))).to(DEV)
    grads = {k: torch.full_like(v, 7.0) for k, v in params.items()}
    api.gs_preprocess_bwd(params, cam, opt, proj, g2, out=grads)
    assert all(float(v.abs().max()) == 0.0 for v in grads.values())
    api.gs_preprocess_bwd(params, cam, opt, proj, g2, out=grads, accumulate=True)
    assert all(float(v.abs().max()) == 0.0 for v in grads.values())


# --------------------------------------------------------------------------------- end to end

@pytest.mark.parametrize("mode", ["adaptive", "direct"])
@pytest.mark.parametrize("name", list(CASES))
def test_end_to_end_matches_oracle(name, mode):
    s, view = scene(name)
    gc.end_to_end(s, view, mode=mode)


def test_large_scene_views_accumulate_like_the_oracle():
    """The large scene's step renders 8 views whose parameter gradients are summed (reduced
    scene): the library's multi-view step (eager and as one captured graph) against the sum of
    the oracle's per-view steps, each view with its own marginal masking."""
    s = gs_scenes.make_scene(3, n=60_000, res_scale=0.25)
    assert len(s.cameras) == 8
    refs = [oracle.view_step(s, view=v, mask_marginal=True) for v in range(8)]
    want = {k: sum(r["grads"][k] for r in refs) for k in refs[0]["grads"] if k != "mag"}
    mags = {k: sum(r["grads"]["mag"][k] for r in refs) for k in refs[0]["grads"]["mag"]}
    flagged = np.zeros(s.n, bool)
    for r in refs:
        flagged |= (r["pre"]["flags"] & oracle.MARGINAL) != 0
    params = gc.dev_params(s)
    opt = api.make_options(s.sh_degree)
    ups = [torch.from_numpy(r["dl_dimage"]).to(DEV) for r in refs]
    cap = max(int(r["pre"]["tiles_touched"].sum(dtype=np.int64)) for r in refs) + 4096
    for graph in (False, True):
        grads = api.alloc_param_grads(params)
        bufs = step.StepBuffers(s.n, DEV)
        if graph:
            g = step.GraphedStep(params, s.cameras, [None] * 8, opt, grads, bufs, cap, upstream=ups)
            g.replay()
        else:
            n_dup = torch.zeros(8, dtype=torch.int64, device=DEV)
            step.train_step_async(params, s.cameras, [None] * 8, opt, grads, bufs, cap, n_dup, upstream=ups)
        torch.cuda.synchronize()
        for name_p in PARAM_NAMES:
            got = grads[name_p].cpu().numpy().reshape(s.n, -1)
            okg, ratio = grad_close_mag(got, want[GRAD_KEYS[name_p]].reshape(s.n, -1),
                                        mags[GRAD_KEYS[name_p]].reshape(s.n, -1), rel_mag=1e-4, mask=~flagged)
            assert okg, f"graph={graph} {name_p}: error {ratio:.3g} x allowance"
