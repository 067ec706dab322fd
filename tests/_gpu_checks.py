"""GPU-side comparisons against the oracle shared by the parity test files: each runs a stage (or
the whole step) of the CUDA library through its C ABI and checks it at the parity bars.

Bars: bit-exact depth keys, duplicate counts, sorted (tile, depth, index) lists, tile ranges and
contributor counts (outside the oracle's marginal decisions); 1e-5 max abs error on pixels; 1e-4
of max|grad| per gradient tensor. The flagged (marginal) pixels are bounded by 5e-6 of the
evaluated (pixel, Gaussian) pairs plus 3: about one flag per million decisions is what a sound
float32 error bound gives (measured up to 3.1e-6 on the full-size scenes).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from differentiable_gaussian_splatting_gs_gb300 import api, step

from _cases import GRAD2D_GROUPS, GRAD_KEYS, PARAM_NAMES, grad_close, grad_close_mag

DEV = torch.device("cuda:0")
FLAGS_PER_PAIR = 5e-6


def u32(t):
    return t.detach().cpu().numpy().view(np.uint32)


def dev_params(s):
    return {k: torch.from_numpy(np.ascontiguousarray(getattr(s, k))).to(DEV) for k in PARAM_NAMES}


def dev_proj(rec):
    return api.proj_from_arrays(rec["mean2d"], rec["conic"], rec["opacity"], rec["rgb"], rec["depth"], rec["radius"],
                                DEV)


def check_flag_count(pix_flags, pairs_evaluated):
    nf = int((pix_flags != 0).sum())
    assert nf <= FLAGS_PER_PAIR * pairs_evaluated + 3, f"{nf} flagged pixels for {pairs_evaluated} evaluated pairs"


def check_preprocess(s, cam, pre, params=None):
    """gs_preprocess of the scene against the oracle's: depth keys bit-exact, radius and tiles
    touched exact off the flagged Gaussians, the mean, opacity and colour within 1e-5 relative
    (+1e-6 of the field's largest magnitude), each conic entry within the larger of 1e-5 and the
    oracle's float32 conditioning bound of the Gaussian's projection, relative to the entry's
    scale (|A|, |C|, sqrt(A C) for B). The flagged Gaussians number at most 4e-3 of the visible
    ones plus 1e-4 of their summed radii plus 3 (four tile edges within 1e-3 px, a radius within
    its relative bound of an integer; measured 2.6e-3 and 6e-5 at the outdoor scene)."""
    params = params if params is not None else dev_params(s)
    proj = api.gs_preprocess(params, cam, api.make_options(s.sh_degree))
    rec = proj.rec.cpu().numpy()
    radius = proj.radius.cpu().numpy()
    tt = u32(proj.tiles_touched)
    depth = proj.depth.cpu().numpy()
    assert np.array_equal(depth.view(np.uint32), pre["depth"].view(np.uint32)), "depth keys differ"
    marginal = (pre["flags"] & oracle.MARGINAL) != 0
    ok = ~marginal
    assert np.array_equal(radius[ok], pre["radius"][ok])
    assert np.array_equal(tt[ok], pre["tiles_touched"][ok])
    live = ok & (pre["radius"] > 0)
    for cols, ref in ((slice(0, 2), pre["mean2d"]), (slice(5, 6), pre["opacity"][:, None]), (slice(6, 9), pre["rgb"])):
        got, want = rec[live, cols].astype(np.float64), ref[live]
        err = np.abs(got - want)
        bound = 1e-5 * np.abs(want) + 1e-6 * np.abs(want).max(axis=0)
        assert np.all(err <= bound), f"cols {cols}: worst {(err / np.maximum(bound, 1e-30)).max():.3g} x bound"
    want = pre["conic"][live]
    err = np.abs(rec[live, 2:5].astype(np.float64) - want)
    scale = np.stack([np.abs(want[:, 0]), np.sqrt(np.abs(want[:, 0] * want[:, 2])), np.abs(want[:, 2])], 1)
    bound = np.maximum(1e-5, pre["conic_tol"][live])[:, None] * scale
    assert np.all(err <= bound), f"conic: worst {(err / np.maximum(bound, 1e-30)).max():.3g} x bound"
    assert np.all(rec[~(radius > 0)] == 0.0)
    vis = pre["radius"] > 0
    allowed = 4e-3 * vis.sum() + 1e-4 * pre["radius"][vis].astype(np.float64).sum() + 3
    assert marginal.sum() <= allowed, (int(marginal.sum()), allowed)
    return proj


def check_bin(proj, cam, opt, vals, ranges, want_keys=False, keys=None):
    """gs_bin_and_sort on the given records: D, the sorted list and the ranges bit-exact."""
    b = api.gs_bin_and_sort(proj, cam, opt, want_keys=want_keys)
    assert b.n_dup == len(vals), (b.n_dup, len(vals))
    assert np.array_equal(u32(b.vals), vals)
    if want_keys:
        assert np.array_equal(b.keys.cpu().numpy().view(np.uint64), keys)
    assert np.array_equal(u32(b.ranges), ranges)
    return b


def check_fwd(proj, b, cam, opt, fwd, pairs_evaluated):
    """gs_render_fwd against the oracle's forward on the same records."""
    img, tf, nc = api.gs_render_fwd(proj, b.vals, b.ranges, cam, opt)
    ok = fwd["pix_flags"] == 0
    check_flag_count(fwd["pix_flags"], pairs_evaluated)
    err = np.abs(img.cpu().numpy() - fwd["image"])
    assert err[:, ok].max() <= 1e-5, err[:, ok].max()
    assert np.array_equal(u32(nc)[ok], fwd["n_contrib"][ok])
    assert np.allclose(tf.cpu().numpy()[ok], fwd["t_final"][ok], rtol=1e-4, atol=1e-7)
    # marginal pixels differ at most by one Gaussian's contribution
    assert err.max() <= 0.02
    return img, tf, nc


def check_bwd(proj, b, cam, opt, tf, nc, dl_masked, grad2d_masked):
    """gs_render_bwd with the upstream gradient zeroed on the flagged pixels: 1e-4 of max per
    group of 2D gradient columns."""
    g2 = api.gs_render_bwd(proj, b.vals, b.ranges, cam, opt, torch.from_numpy(dl_masked).to(DEV), tf, nc)
    got = g2.cpu().numpy()
    assert np.all(got[:, 9:] == 0.0)
    for group, cols in GRAD2D_GROUPS.items():
        okg, err, tol = grad_close(got[:, cols], grad2d_masked[:, cols])
        assert okg, f"{group}: error {err:.3g} > {tol:.3g}"
    return g2


def check_preprocess_bwd(s, cam, pre, grad2d32, want, params=None, proj=None):
    params = params if params is not None else dev_params(s)
    opt = api.make_options(s.sh_degree)
    if proj is None:
        proj = api.gs_preprocess(params, cam, opt)
    g2 = torch.zeros((s.n, 12), dtype=torch.float32, device=DEV)
    g2[:, :9] = torch.from_numpy(grad2d32).to(DEV)
    grads = api.gs_preprocess_bwd(params, cam, opt, proj, g2)
    ok_rows = (pre["flags"] & oracle.MARGINAL) == 0
    # 1e-4 of the tensor's largest magnitude, plus 1e-5 of the Gaussian's own chain-rule terms where
    # they cancel (float32 evaluates each term to a few units in the last place)
    for name_p in PARAM_NAMES:
        got = grads[name_p].cpu().numpy().reshape(s.n, -1)
        w = want[GRAD_KEYS[name_p]].reshape(s.n, -1)
        mag = want["mag"][GRAD_KEYS[name_p]].reshape(s.n, -1)
        okg, ratio = grad_close_mag(got, w, mag, rel_mag=1e-5, mask=ok_rows)
        assert okg, f"{name_p}: error {ratio:.3g} x allowance"


def tile_entries(vals, ranges):
    """(tile id, Gaussian index) of every entry of a sorted list, in list order."""
    lens = (ranges[:, 1].astype(np.int64) - ranges[:, 0].astype(np.int64))
    tiles = np.repeat(np.arange(len(ranges)), lens)
    starts = ranges[lens > 0, 0].astype(np.int64)
    if lens.sum() == 0:
        return tiles, np.zeros(0, np.uint32)
    # positions of every entry: each non-empty tile's run, in tile order
    offs = np.repeat(starts - np.concatenate([[0], np.cumsum(lens[lens > 0])[:-1]]), lens[lens > 0])
    order = np.arange(int(lens.sum()), dtype=np.int64) + offs
    return tiles, vals[order]


def check_end_to_end(ref, b, img, nc, grads, s, flagged):
    """A whole step of the library (each side computes its own float32 / float64 records) against
    the oracle's view step with marginal masking (`ref` from oracle.view_step(mask_marginal=True))."""
    pre = ref["pre"]
    # sorted lists: identical after removing the entries of Gaussians with a marginal radius or
    # rectangle; so is the duplicate count once their entries are taken off on both sides
    gv_all, ov_all = u32(b.vals)[: b.n_dup], ref["vals"]
    gt, gv = tile_entries(gv_all, u32(b.ranges))
    ot, ov = tile_entries(ov_all, ref["ranges"])
    kg, ko = ~flagged[gv], ~flagged[ov]
    assert np.array_equal(gt[kg], ot[ko]) and np.array_equal(gv[kg], ov[ko])
    assert int(kg.sum()) == int(ko.sum())
    ok = ~ref["marginal"]
    err = np.abs(img.cpu().numpy() - ref["fwd"]["image"])
    # each side computes its own records here, so the 1e-5 bar is widened by the oracle's bound on
    # the colour change those record differences can cause (alpha bounds propagated per pixel)
    bound = 1e-5 + ref["fwd"]["pix_err"]
    assert np.all(err[:, ok] <= bound[None][:, ok]), (err - bound[None])[:, ok].max()
    assert np.median(ref["fwd"]["pix_err"][ok]) < 5e-4, "the propagated bound is not informative"
    assert np.mean(err[:, ok] <= 1e-5) > 0.99, "more than 1% of the pixels above 1e-5"
    assert np.array_equal(u32(nc)[ok], ref["fwd"]["n_contrib"][ok])
    # 3D gradients: 1e-4 of max, plus 1e-4 of the Gaussian's own chain-rule terms (each side's 2D
    # gradient carries the rounding of its own records, which the chain rule of a needle-like
    # Gaussian amplifies where its terms cancel). The 2D gradients themselves are checked at 1e-4
    # of max on identical records by the stage tests.
    for name_p in PARAM_NAMES:
        got = grads[name_p].cpu().numpy().reshape(s.n, -1)
        want = ref["grads"][GRAD_KEYS[name_p]].reshape(s.n, -1)
        mag = ref["grads"]["mag"][GRAD_KEYS[name_p]].reshape(s.n, -1)
        okg, ratio = grad_close_mag(got, want, mag, rel_mag=1e-4, mask=~flagged)
        assert okg, f"{name_p}: error {ratio:.3g} x allowance"


def end_to_end(s, view, mode="adaptive", staging=0, pre=None, bins=None, graph=False):
    """The library's step of one view (default: the benchmark's launch configuration, ADAPTIVE
    accumulation with bulk staging) against oracle.view_step with marginal masking. With `graph`
    the step is the captured CUDA graph of step.GraphedStep, replayed twice, with the oracle's
    masked upstream gradient as its dL/dimage."""
    cam = s.cameras[view]
    params = dev_params(s)
    opt = api.make_options(s.sh_degree, bwd_mode=mode, staging=staging)
    ref = oracle.view_step(s, view=view, mask_marginal=True, pre=pre, bins=bins)
    dl = torch.from_numpy(ref["dl_dimage"]).to(DEV)
    bufs = step.StepBuffers(s.n, DEV)
    if graph:
        grads = api.alloc_param_grads(params)
        cap = int(ref["pre"]["tiles_touched"].sum(dtype=np.int64)) + 4096
        g = step.GraphedStep(params, [cam], [None], opt, grads, bufs, cap, upstream=[dl])
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        D = int(g.n_dup[0].item())
        img, tf, nc, _, ranges = bufs.image_buffers(cam.width, cam.height)
        b = api.BinResult(keys=None, vals=bufs.sort.vals[:D], ranges=ranges, n_dup=D)
    else:
        proj = api.gs_preprocess(params, cam, opt, out=bufs.proj)
        b = api.gs_bin_and_sort(proj, cam, opt, buffers=bufs.sort, want_keys=False)
        img, tf, nc = api.gs_render_fwd(proj, b.vals, b.ranges, cam, opt)
        g2 = api.gs_render_bwd(proj, b.vals, b.ranges, cam, opt, dl, tf, nc)
        grads = api.gs_preprocess_bwd(params, cam, opt, proj, g2)
    flagged = (ref["pre"]["flags"] & oracle.MARGINAL) != 0
    check_end_to_end(ref, b, img, nc, grads, s, flagged)
    return ref, b
