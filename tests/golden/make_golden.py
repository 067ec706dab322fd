"""Writes tests/golden/one_gaussian.json: two single-Gaussian cases whose results have closed
forms (derived in tests/test_golden.py), with the float64 oracle's outputs on them.

    python tests/golden/make_golden.py

Only the oracle computes the stored outputs; the inputs are written here by hand. The file is a
regression fixture for the oracle (a change of its arithmetic shows up as a diff of this file)
and the reference values of the GPU check in tests/test_golden.py.
"""
from __future__ import annotations

import json
import math
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import gs_scenes  # noqa: E402
import oracle  # noqa: E402


def cases() -> dict:
    """The two scenes (inputs only), as plain lists."""
    eye = [1.0, 0.0, 0.0, 0.0, 1.0, 0.0, 0.0, 0.0, 1.0]
    return {
        # an isotropic Gaussian on the optical axis, its mean on the centre of pixel (32, 32)
        "axis_isotropic": dict(
            camera=dict(R=eye, t=[0.0, 0.0, 0.0], fx=64.0, fy=64.0, cx=32.5, cy=32.5, width=64, height=64,
                        bg=[0.0, 0.0, 0.0]),
            mean3d=[[0.0, 0.0, 4.0]], log_scale=[[math.log(0.25)] * 3], quat=[[1.0, 0.0, 0.0, 0.0]],
            opacity_logit=[0.0], sh=[[[0.4, -0.2, 1.0]]], sh_degree=0,
            target_value=[0.25, 0.5, 0.75]),
        # a one-pixel image whose pixel centre is the projected mean
        "one_pixel": dict(
            camera=dict(R=eye, t=[0.0, 0.0, 0.0], fx=1.0, fy=1.0, cx=0.5, cy=0.5, width=1, height=1,
                        bg=[0.1, 0.2, 0.3]),
            mean3d=[[0.0, 0.0, 2.0]], log_scale=[[math.log(0.5)] * 3], quat=[[1.0, 0.0, 0.0, 0.0]],
            opacity_logit=[0.3], sh=[[[0.2, 0.1, -0.1]]], sh_degree=0,
            target_value=[0.9, 0.1, 0.4]),
    }


def scene_of(c: dict) -> gs_scenes.Scene:
    cam = c["camera"]
    camera = gs_scenes.Camera(R=np.asarray(cam["R"], np.float32), t=np.asarray(cam["t"], np.float32),
                              fx=cam["fx"], fy=cam["fy"], cx=cam["cx"], cy=cam["cy"], width=cam["width"],
                              height=cam["height"], bg=np.asarray(cam["bg"], np.float32))
    f32 = lambda a: np.asarray(a, np.float32)
    target = np.broadcast_to(f32(c["target_value"])[:, None, None], (3, cam["height"], cam["width"])).copy()
    return gs_scenes.Scene(name="golden", mean3d=f32(c["mean3d"]), log_scale=f32(c["log_scale"]),
                           quat=f32(c["quat"]), opacity_logit=f32(c["opacity_logit"]), sh=f32(c["sh"]),
                           sh_degree=c["sh_degree"], cameras=[camera], targets=[target])


# pixels (x, y) whose image, transmittance and contributor count are stored
SAMPLES = [(32, 32), (33, 32), (32, 34), (29, 36), (44, 32), (45, 32), (0, 0), (63, 63)]


def oracle_outputs(c: dict) -> dict:
    s = scene_of(c)
    out = oracle.view_step(s)
    pre, fwd, g = out["pre"], out["fwd"], out["grads"]
    lst = lambda a: np.asarray(a, np.float64).tolist()
    W, H = c["camera"]["width"], c["camera"]["height"]
    px = [(x, y) for x, y in SAMPLES if x < W and y < H]
    return dict(mean2d=lst(pre["mean2d"]), conic=lst(pre["conic"]), opacity=lst(pre["opacity"]),
                rgb=lst(pre["rgb"]), depth=lst(pre["depth"]), radius=np.asarray(pre["radius"]).tolist(),
                tiles_touched=np.asarray(pre["tiles_touched"]).tolist(), pixels=px,
                image=[lst(fwd["image"][:, y, x]) for x, y in px], t_final=[float(fwd["t_final"][y, x]) for x, y in px],
                n_contrib=[int(fwd["n_contrib"][y, x]) for x, y in px],
                d_mean3d=lst(g["d_mean3d"]), d_log_scale=lst(g["d_log_scale"]), d_quat=lst(g["d_quat"]),
                d_opacity_logit=lst(g["d_opacity_logit"]), d_sh=lst(g["d_sh"]))


def main():
    cs = cases()
    data = {"about": "single-Gaussian cases with closed forms (tests/test_golden.py derives them); outputs "
                     "written by tests/golden/make_golden.py from the float64 oracle only",
            "cases": {name: dict(inputs=c, oracle=oracle_outputs(c)) for name, c in cs.items()}}
    with open(os.path.join(HERE, "one_gaussian.json"), "w") as f:
        json.dump(data, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
