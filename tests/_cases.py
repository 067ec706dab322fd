"""Shared cases for the GPU parity tests: seeded scenes and the oracle's results on them.

Every oracle input comes from the seeded scene generator or from the oracle itself; nothing the
CUDA library produces is fed to the oracle.
"""
from __future__ import annotations

import functools

import numpy as np

import gs_scenes
import oracle

# name -> (config, n, res_scale, view)
CASES = {
    "tiny": (0, None, 1.0, 0),
    "object": (1, 20_000, 1.0, 0),
    "outdoor": (2, 100_000, 0.5, 0),
    "large": (3, 60_000, 0.25, 1),
    "contention": (4, 3_000, 0.25, 0),
}

PARAM_NAMES = ("mean3d", "log_scale", "quat", "opacity_logit", "sh")
GRAD_KEYS = {"mean3d": "d_mean3d", "log_scale": "d_log_scale", "quat": "d_quat", "opacity_logit": "d_opacity_logit",
             "sh": "d_sh"}
# column groups of grad2d compared as separate tensors
GRAD2D_GROUPS = {"mean2d": slice(0, 2), "conic": slice(2, 5), "opacity": slice(5, 6), "rgb": slice(6, 9)}


@functools.lru_cache(maxsize=None)
def scene(name: str):
    cfg, n, rs, view = CASES[name]
    views = None if cfg != 3 else 2
    return gs_scenes.make_scene(cfg, n=n, res_scale=rs, views=views), view


@functools.lru_cache(maxsize=None)
def stage_inputs(name: str):
    """Oracle preprocess of the case; its outputs rounded to float32 are the projected-Gaussian
    inputs of the later stages, for the oracle and the CUDA library alike."""
    s, view = scene(name)
    cam = s.cameras[view]
    pre = oracle.preprocess(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, s.sh_degree, cam)
    rec = dict(mean2d=pre["mean2d"].astype(np.float32), conic=pre["conic"].astype(np.float32),
               opacity=pre["opacity"].astype(np.float32), rgb=pre["rgb"].astype(np.float32),
               depth=pre["depth"], radius=pre["radius"])
    keys, vals, ranges = oracle.bin_and_sort(rec["mean2d"], rec["depth"], rec["radius"], cam.width, cam.height)
    f64 = lambda a: a.astype(np.float64)
    fwd = oracle.render(f64(rec["mean2d"]), f64(rec["conic"]), f64(rec["opacity"]), f64(rec["rgb"]), vals, ranges, cam)
    dl = (fwd["image"] - s.targets[view]).astype(np.float32)
    bwd = oracle.render(f64(rec["mean2d"]), f64(rec["conic"]), f64(rec["opacity"]), f64(rec["rgb"]), vals, ranges,
                        cam, dl_dimage=dl)
    # the same upstream gradient with the marginal pixels zeroed: their float32 decisions may
    # legitimately differ from float64 ones, which moves every gradient they feed
    dl_m = np.where(fwd["pix_flags"][None] != 0, 0.0, dl).astype(np.float32)
    bwd_m = oracle.render(f64(rec["mean2d"]), f64(rec["conic"]), f64(rec["opacity"]), f64(rec["rgb"]), vals, ranges,
                          cam, dl_dimage=dl_m)
    grad2d32 = bwd["grad2d"].astype(np.float32)
    g3 = oracle.preprocess_bwd(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, s.sh_degree, cam, grad2d32)
    return dict(scene=s, cam=cam, view=view, pre=pre, rec=rec, keys=keys, vals=vals, ranges=ranges, fwd=fwd,
                dl=dl, grad2d=bwd["grad2d"], dl_masked=dl_m, grad2d_masked=bwd_m["grad2d"], grad2d32=grad2d32,
                grads=g3, stats=bwd["stats"])


@functools.lru_cache(maxsize=None)
def full_size(cfg: int):
    """One view of a configuration at its full size (the benchmark's workload for that
    configuration), computed once by the oracle: preprocess of the scene, the binning of its
    float32-rounded outputs, and the stagewise forward and backward on those float32 records (the
    inputs both sides take in the stage tests). The upstream gradient of the backward is
    oracle image - target with the flagged pixels zeroed. The 64-bit keys are not kept."""
    s = gs_scenes.make_scene(cfg, views=1 if cfg == 3 else None)
    cam = s.cameras[0]
    pre = oracle.preprocess(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, s.sh_degree, cam)
    rec = dict(mean2d=pre["mean2d"].astype(np.float32), conic=pre["conic"].astype(np.float32),
               opacity=pre["opacity"].astype(np.float32), rgb=pre["rgb"].astype(np.float32),
               depth=pre["depth"], radius=pre["radius"])
    _, vals, ranges = oracle.bin_and_sort(rec["mean2d"], rec["depth"], rec["radius"], cam.width, cam.height,
                                          capacity=int(pre["tiles_touched"].sum(dtype=np.int64)))
    bins = (None, vals, ranges)
    f64 = lambda a: a.astype(np.float64)
    args = (f64(rec["mean2d"]), f64(rec["conic"]), f64(rec["opacity"]), f64(rec["rgb"]), vals, ranges, cam)
    fwd = oracle.render(*args)
    dl = (fwd["image"] - s.targets[0]).astype(np.float32)
    dl_m = np.where(fwd["pix_flags"][None] != 0, 0.0, dl).astype(np.float32)
    bwd = oracle.render(*args, dl_dimage=dl_m)
    grad2d32 = bwd["grad2d"].astype(np.float32)
    g3 = oracle.preprocess_bwd(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, s.sh_degree, cam, grad2d32)
    return dict(scene=s, cam=cam, pre=pre, rec=rec, bins=bins, vals=vals, ranges=ranges, fwd=fwd, dl_masked=dl_m,
                grad2d_masked=bwd["grad2d"], grad2d32=grad2d32, grads=g3, stats=fwd["stats"])


def grad_close_mag(got: np.ndarray, want: np.ndarray, mag: np.ndarray, rel: float = 1e-4, rel_mag: float = 1e-5,
                   mask=None) -> tuple[bool, float]:
    """|got - want| <= rel * max|want| + rel_mag * mag elementwise, where mag is the oracle's sum of
    the magnitudes of the chain-rule terms each gradient adds up (it exceeds |want| where they
    cancel). Returns (ok, worst ratio of error to allowance)."""
    if mask is not None:
        got, want, mag = got[mask], want[mask], mag[mask]
    if not want.size:
        return True, 0.0
    allow = rel * float(np.abs(want).max()) + rel_mag * mag + 1e-30
    ratio = float((np.abs(got.astype(np.float64) - want) / allow).max())
    return ratio <= 1.0, ratio


def grad_close(got: np.ndarray, want: np.ndarray, rel: float = 1e-4, mask=None) -> tuple[bool, float, float]:
    """|got - want| <= rel * max|want| over the tensor (rows restricted by mask)."""
    if mask is not None:
        got, want = got[mask], want[mask]
    scale = float(np.abs(want).max()) if want.size else 0.0
    err = float(np.abs(got.astype(np.float64) - want).max()) if want.size else 0.0
    return err <= rel * scale + 1e-30, err, rel * scale
