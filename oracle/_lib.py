"""ctypes binding of the float64 CPU oracle (oracle/gs_oracle.cpp).

TEST INFRASTRUCTURE: only the test suite, the smoke check and the benchmark's CPU-baseline leg
use this module. The CUDA library never imports it.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gs_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


# Gaussian flags of preprocess(): bit 0 culled; these three mark a Gaussian whose float32 projection
# may legitimately differ from this oracle's (radius at a ceiling boundary, tile rectangle at a tile
# edge, projection ill-conditioned in float32)
MARGINAL = 2 | 4 | 8


class OrCamera(C.Structure):
    _fields_ = [("R", C.c_float * 9), ("t", C.c_float * 3), ("fx", C.c_float), ("fy", C.c_float),
                ("cx", C.c_float), ("cy", C.c_float), ("width", C.c_int32), ("height", C.c_int32),
                ("bg", C.c_float * 3)]


class OrOptions(C.Structure):
    _fields_ = [("near_z", C.c_double), ("lowpass", C.c_double), ("jacobian_clamp", C.c_double),
                ("sh_degree", C.c_int32), ("threads", C.c_int32)]


class OrRenderStats(C.Structure):
    _fields_ = [("pairs_evaluated", C.c_int64), ("pairs_blended", C.c_int64),
                ("marginal_pixels", C.c_int64), ("warp_gauss_active", C.c_int64),
                ("tile_gauss_active", C.c_int64), ("lane_hist", C.c_int64 * 33)]


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (float64, OpenMP, no floating-point contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = C.CDLL(build())
            P = C.c_void_p
            _lib.or_preprocess.argtypes = [C.c_int64] + [P] * 5 + [P, P] + [P] * 11
            _lib.or_preprocess.restype = C.c_int
            _lib.or_bin.argtypes = [C.c_int64, P, P, P, C.c_int32, C.c_int32, P, P, C.c_int64, P]
            _lib.or_bin.restype = C.c_int64
            _lib.or_render.argtypes = ([C.c_int64] + [P] * 6 + [P] + [P] * 8 + [P, C.c_int] +
                                        [P, C.c_double, P, C.c_double, P])
            _lib.or_render.restype = C.c_int
            _lib.or_preprocess_bwd.argtypes = [C.c_int64] + [P] * 5 + [P, P] + [P] * 7
            _lib.or_preprocess_bwd.restype = C.c_int
            _lib.or_preprocess2d.argtypes = [C.c_int64] + [P] * 5 + [P, P] + [P] * 6
            _lib.or_preprocess2d.restype = C.c_int
            _lib.or_render2d.argtypes = [C.c_int64, P, P, P, P, P, P, P, P, P, P, P, C.c_int]
            _lib.or_render2d.restype = C.c_int
            _lib.or_preprocess2d_bwd.argtypes = [C.c_int64] + [P] * 5 + [P, P] + [P] * 6
            _lib.or_preprocess2d_bwd.restype = C.c_int
            _lib.or_sh_basis.argtypes = [C.c_int, P, P]
            _lib.or_quat_to_rotmat.argtypes = [P, P]
        return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def camera(cam, bg=None) -> OrCamera:
    c = OrCamera()
    c.R[:] = [float(v) for v in np.asarray(cam.R, np.float32).reshape(9)]
    c.t[:] = [float(v) for v in np.asarray(cam.t, np.float32).reshape(3)]
    c.fx, c.fy, c.cx, c.cy = float(cam.fx), float(cam.fy), float(cam.cx), float(cam.cy)
    c.width, c.height = int(cam.width), int(cam.height)
    c.bg[:] = [float(v) for v in np.asarray(cam.bg if bg is None else bg, np.float32).reshape(3)]
    return c


def options(sh_degree, near_z=0.2, lowpass=0.3, jacobian_clamp=1.3, threads=0) -> OrOptions:
    return OrOptions(near_z=float(np.float32(near_z)), lowpass=lowpass, jacobian_clamp=jacobian_clamp,
                     sh_degree=int(sh_degree), threads=int(threads))


def sh_basis(deg: int, direction) -> np.ndarray:
    d = _c(direction, np.float64)
    out = np.zeros(16, np.float64)
    lib().or_sh_basis(deg, _p(d), _p(out))
    return out[: (deg + 1) ** 2]


def quat_to_rotmat(q) -> np.ndarray:
    qq = _c(q, np.float64)
    out = np.zeros(9, np.float64)
    lib().or_quat_to_rotmat(_p(qq), _p(out))
    return out.reshape(3, 3)


def preprocess(mean3d, log_scale, quat, opacity_logit, sh, sh_degree, cam, threads=0, **opt):
    n = int(np.asarray(mean3d).shape[0])
    m, ls, q, lg, sh = (_c(mean3d, np.float64), _c(log_scale, np.float64), _c(quat, np.float64),
                        _c(opacity_logit, np.float64), _c(sh, np.float64))
    out = dict(mean2d=np.zeros((n, 2)), conic=np.zeros((n, 3)), opacity=np.zeros(n), rgb=np.zeros((n, 3)),
               depth=np.zeros(n, np.float32), radius=np.zeros(n, np.int32),
               tiles_touched=np.zeros(n, np.uint32), flags=np.zeros(n, np.uint8), cov2d=np.zeros((n, 3)),
               mean_tol=np.zeros(n), conic_tol=np.zeros(n))
    c, o = camera(cam), options(sh_degree, threads=threads, **opt)
    rc = lib().or_preprocess(n, _p(m), _p(ls), _p(q), _p(lg), _p(sh), C.byref(c), C.byref(o),
                             _p(out["mean2d"]), _p(out["conic"]), _p(out["opacity"]), _p(out["rgb"]),
                             _p(out["depth"]), _p(out["radius"]), _p(out["tiles_touched"]),
                             _p(out["flags"]), _p(out["cov2d"]), _p(out["mean_tol"]), _p(out["conic_tol"]))
    assert rc == 0
    return out


def bin_and_sort(mean2d_f32, depth_f32, radius, width, height, capacity=None):
    """Returns (keys u64[D], vals u32[D], ranges u32[T, 2])."""
    n = int(np.asarray(radius).shape[0])
    m, d, r = _c(mean2d_f32, np.float32), _c(depth_f32, np.float32), _c(radius, np.int32)
    T = ((width + 15) // 16) * ((height + 15) // 16)
    ranges = np.zeros((T, 2), np.uint32)
    cap = 0 if capacity is None else int(capacity)
    while True:
        keys = np.zeros(max(cap, 1), np.uint64)
        vals = np.zeros(max(cap, 1), np.uint32)
        D = lib().or_bin(n, _p(m), _p(d), _p(r), int(width), int(height), _p(keys), _p(vals), cap, _p(ranges))
        if D <= cap:
            return keys[:D], vals[:D], ranges
        cap = int(D)


def render(mean2d, conic, opacity, rgb, vals, ranges, cam, dl_dimage=None, threads=0, bg=None, record_tol=None):
    """record_tol = (mean_tol [N] px, conic_rel, opacity_rel, conic_scale_tol [N] or None) widens
    the marginal-decision bands by how much another implementation's records may differ from
    these (None: same records): means within mean_tol px, the conic's quadratic form within a
    relative conic_rel, opacities within a relative opacity_rel, and where conic_scale_tol > 0
    each conic entry within that fraction of its scale (|A|, |C|, sqrt(A C) for B)."""
    n = int(np.asarray(opacity).shape[0])
    W, H = int(cam.width), int(cam.height)
    m, cn, op, cl = (_c(mean2d, np.float64), _c(conic, np.float64), _c(opacity, np.float64),
                     _c(rgb, np.float64))
    v, rg = _c(vals, np.uint32), _c(ranges, np.uint32)
    dl = None if dl_dimage is None else _c(dl_dimage, np.float32)
    out = dict(image=np.zeros((3, H, W)), t_final=np.zeros((H, W)), n_contrib=np.zeros((H, W), np.uint32),
               n_blended=np.zeros((H, W), np.uint32), pix_flags=np.zeros((H, W), np.uint8),
               pix_sig=np.zeros((H, W), np.uint64), pix_err=np.zeros((H, W)))
    grad = np.zeros((n, 9)) if dl is not None else None
    st = OrRenderStats()
    c = camera(cam, bg)
    mt, crel, orel, cst = (None, 0.0, 0.0, None) if record_tol is None else record_tol
    mt = None if mt is None else _c(mt, np.float64)
    cst = None if cst is None else _c(cst, np.float64)
    rc = lib().or_render(n, _p(m), _p(cn), _p(op), _p(cl), _p(v), _p(rg), C.byref(c), _p(dl),
                         _p(out["image"]), _p(out["t_final"]), _p(out["n_contrib"]), _p(out["n_blended"]),
                         _p(out["pix_flags"]), _p(out["pix_sig"]), _p(grad), C.byref(st), int(threads),
                         _p(mt), float(crel), _p(cst), float(orel), _p(out["pix_err"]))
    assert rc == 0
    out["grad2d"] = grad
    out["stats"] = dict(pairs_evaluated=st.pairs_evaluated, pairs_blended=st.pairs_blended,
                        marginal_pixels=st.marginal_pixels, warp_gauss_active=st.warp_gauss_active,
                        tile_gauss_active=st.tile_gauss_active, lane_hist=list(st.lane_hist))
    return out


def preprocess_bwd(mean3d, log_scale, quat, opacity_logit, sh, sh_degree, cam, grad2d, threads=0, **opt):
    n = int(np.asarray(mean3d).shape[0])
    K = (sh_degree + 1) ** 2
    m, ls, q, lg, shc = (_c(mean3d, np.float64), _c(log_scale, np.float64), _c(quat, np.float64),
                         _c(opacity_logit, np.float64), _c(sh, np.float64))
    g2 = _c(grad2d, np.float64)
    out = dict(d_mean3d=np.zeros((n, 3)), d_log_scale=np.zeros((n, 3)), d_quat=np.zeros((n, 4)),
               d_opacity_logit=np.zeros(n), d_sh=np.zeros((n, K, 3)))
    mag = np.zeros((n, 11))
    c, o = camera(cam), options(sh_degree, threads=threads, **opt)
    rc = lib().or_preprocess_bwd(n, _p(m), _p(ls), _p(q), _p(lg), _p(shc), C.byref(c), C.byref(o), _p(g2),
                                 _p(out["d_mean3d"]), _p(out["d_log_scale"]), _p(out["d_quat"]),
                                 _p(out["d_opacity_logit"]), _p(out["d_sh"]), _p(mag))
    assert rc == 0
    # magnitudes of the terms each gradient sums (the SH gradients are single terms)
    out["mag"] = dict(d_mean3d=mag[:, 0:3], d_log_scale=mag[:, 3:6], d_quat=mag[:, 6:10], d_opacity_logit=mag[:, 10],
                      d_sh=np.abs(out["d_sh"]))
    return out


def preprocess2d(mean3d, log_scale, quat, opacity_logit, sh, sh_degree, cam, threads=0, **opt):
    """Surfel (2D Gaussian splatting) preprocessing: rec2d [N, 16] = (A_u, B_u, C_u, A_v, B_v, C_v,
    m_x, m_y, z_c, c_x, c_y, opacity, r, g, b, 0), mean2d = bounding-box centre (for the binning),
    depth, radius, tiles_touched, half extents."""
    n = int(np.asarray(mean3d).shape[0])
    m, ls, q, lg, sh = (_c(mean3d, np.float64), _c(log_scale, np.float64), _c(quat, np.float64),
                        _c(opacity_logit, np.float64), _c(sh, np.float64))
    out = dict(rec2d=np.zeros((n, 16)), mean2d=np.zeros((n, 2)), depth=np.zeros(n, np.float32),
               radius=np.zeros(n, np.int32), tiles_touched=np.zeros(n, np.uint32), half=np.zeros((n, 2)))
    c, o = camera(cam), options(sh_degree, threads=threads, **opt)
    rc = lib().or_preprocess2d(n, _p(m), _p(ls), _p(q), _p(lg), _p(sh), C.byref(c), C.byref(o), _p(out["rec2d"]),
                               _p(out["mean2d"]), _p(out["depth"]), _p(out["radius"]), _p(out["tiles_touched"]),
                               _p(out["half"]))
    assert rc == 0
    return out


def render2d(rec2d, vals, ranges, cam, dl_dimage=None, threads=0, bg=None):
    """Surfel render forward (+ backward: grad [N, 16] = dL/d rec2d fields 0..14)."""
    n = int(np.asarray(rec2d).shape[0])
    W, H = int(cam.width), int(cam.height)
    r, v, rg = _c(rec2d, np.float64), _c(vals, np.uint32), _c(ranges, np.uint32)
    dl = None if dl_dimage is None else _c(dl_dimage, np.float32)
    out = dict(image=np.zeros((3, H, W)), t_final=np.zeros((H, W)), n_contrib=np.zeros((H, W), np.uint32),
               pix_flags=np.zeros((H, W), np.uint8), pix_sig=np.zeros((H, W), np.uint64))
    grad = np.zeros((n, 16)) if dl is not None else None
    c = camera(cam, bg)
    rc = lib().or_render2d(n, _p(r), _p(v), _p(rg), C.byref(c), _p(dl), _p(out["image"]), _p(out["t_final"]),
                           _p(out["n_contrib"]), _p(out["pix_flags"]), _p(out["pix_sig"]), _p(grad), int(threads))
    assert rc == 0
    out["grad"] = grad
    return out


def preprocess2d_bwd(mean3d, log_scale, quat, opacity_logit, sh, sh_degree, cam, grad, threads=0, **opt):
    n = int(np.asarray(mean3d).shape[0])
    K = (sh_degree + 1) ** 2
    m, ls, q, lg, shc = (_c(mean3d, np.float64), _c(log_scale, np.float64), _c(quat, np.float64),
                         _c(opacity_logit, np.float64), _c(sh, np.float64))
    g = _c(grad, np.float64)
    out = dict(d_mean3d=np.zeros((n, 3)), d_log_scale=np.zeros((n, 3)), d_quat=np.zeros((n, 4)),
               d_opacity_logit=np.zeros(n), d_sh=np.zeros((n, K, 3)))
    c, o = camera(cam), options(sh_degree, threads=threads, **opt)
    rc = lib().or_preprocess2d_bwd(n, _p(m), _p(ls), _p(q), _p(lg), _p(shc), C.byref(c), C.byref(o), _p(g),
                                   _p(out["d_mean3d"]), _p(out["d_log_scale"]), _p(out["d_quat"]),
                                   _p(out["d_opacity_logit"]), _p(out["d_sh"]))
    assert rc == 0
    return out


def view_step2d(scene, view=0, dl_dimage=None, threads=0):
    """Surfel training step of one view in float64: preprocess, binning (the same tile sort on the
    bounding-box centres), render forward, and with dl_dimage the backward to the parameters."""
    cam = scene.cameras[view]
    pre = preprocess2d(scene.mean3d, scene.log_scale, scene.quat, scene.opacity_logit, scene.sh, scene.sh_degree,
                       cam, threads=threads)
    keys, vals, ranges = bin_and_sort(pre["mean2d"].astype(np.float32), pre["depth"], pre["radius"], cam.width,
                                      cam.height, capacity=int(pre["tiles_touched"].sum(dtype=np.int64)))
    fwd = render2d(pre["rec2d"], vals, ranges, cam, dl_dimage, threads=threads)
    out = dict(pre=pre, keys=keys, vals=vals, ranges=ranges, fwd=fwd)
    if dl_dimage is not None:
        out["bwd"] = preprocess2d_bwd(scene.mean3d, scene.log_scale, scene.quat, scene.opacity_logit, scene.sh,
                                      scene.sh_degree, cam, fwd["grad"], threads=threads)
    return out


def marginal_mask(pre, fwd, cam):
    """Pixels whose float32 result may legitimately differ from this float64 oracle: pixels with a
    marginal decision, and the pixels of every tile a Gaussian with a marginal radius or tile
    rectangle may gain or lose: the tiles of its rectangle at radius r + 1 that are not in its
    rectangle at radius r - 1 (one pixel of radius covers more than the mean's float32 error).
    Returns a bool [H, W] array (True = marginal)."""
    mask = fwd["pix_flags"] != 0
    flagged = np.nonzero((pre["flags"] & MARGINAL) != 0)[0]
    T = ((cam.width + 15) // 16) * ((cam.height + 15) // 16)
    ring = np.zeros(T, bool)
    m32 = pre["mean2d"].astype(np.float32)
    for g in flagged:
        r = int(pre["radius"][g]) if pre["radius"][g] > 0 else int(np.ceil(3.0 * np.sqrt(
            0.5 * (pre["cov2d"][g, 0] + pre["cov2d"][g, 2]) +
            np.sqrt(0.25 * (pre["cov2d"][g, 0] - pre["cov2d"][g, 2]) ** 2 + pre["cov2d"][g, 1] ** 2))))
        tiles = []
        for rr in (r + 1, max(r - 1, 0)):
            _, _, rg = bin_and_sort(m32[g:g + 1], pre["depth"][g:g + 1], np.array([rr], np.int32),
                                    cam.width, cam.height)
            tiles.append(rg[:, 1] > rg[:, 0])
        ring |= tiles[0] & ~tiles[1]
    if ring.any():
        hit = ring.reshape((cam.height + 15) // 16, (cam.width + 15) // 16)
        mask |= np.kron(hit, np.ones((16, 16), bool))[: cam.height, : cam.width]
    return mask


def view_step(scene, view=0, dl_dimage=None, with_backward=True, threads=0, mask_marginal=False, pre=None,
              bins=None, **opt):
    """Whole training step of one view: preprocess, binning and sort, render, and (when
    `with_backward`) the gradient computation and the preprocess backward.

    The upstream gradient defaults to dL/dimage = image - target (the squared-error loss
    0.5 |image - target|^2), with the target image of the view; the oracle's own float64 image
    is used, rounded to float32. With `mask_marginal` it is zeroed on `marginal_mask` pixels.
    `pre` and `bins` = (keys, vals, ranges) may pass in this view's preprocess and binning results
    computed earlier by this module (they are then not recomputed).
    """
    cam = scene.cameras[view]
    if pre is None:
        pre = preprocess(scene.mean3d, scene.log_scale, scene.quat, scene.opacity_logit, scene.sh,
                         scene.sh_degree, cam, threads=threads, **opt)
    m32 = pre["mean2d"].astype(np.float32)
    if bins is None:
        bins = bin_and_sort(m32, pre["depth"], pre["radius"], cam.width, cam.height,
                            capacity=int(pre["tiles_touched"].sum(dtype=np.int64)))
    keys, vals, ranges = bins
    # In mask_marginal mode the decision bands also cover a float32 preprocess of the same scene
    # (means within mean_tol, the conic's quadratic form within 1e-5 and opacities within 1e-6
    # relative: several times what a float32 preprocess was measured to differ by; and for the
    # Gaussians whose projection is ill-conditioned in float32 (flag 8), each conic entry within
    # the oracle's conditioning bound conic_tol of its scale).
    ill = (pre["flags"] & 8) != 0
    rt = (pre["mean_tol"], 1e-5, 1e-6, np.where(ill, pre["conic_tol"], 0.0)) if mask_marginal else None
    fwd = render(pre["mean2d"], pre["conic"], pre["opacity"], pre["rgb"], vals, ranges, cam, threads=threads,
                 record_tol=rt)
    out = dict(pre=pre, keys=keys, vals=vals, ranges=ranges, fwd=fwd)
    if not with_backward:
        return out
    if dl_dimage is None:
        dl_dimage = (fwd["image"] - scene.targets[view]).astype(np.float32)
    if mask_marginal:
        # pixels where a float32 implementation may decide differently get no upstream gradient
        out["marginal"] = marginal_mask(pre, fwd, cam)
        dl_dimage = np.where(out["marginal"][None], 0.0, dl_dimage).astype(np.float32)
    bwd = render(pre["mean2d"], pre["conic"], pre["opacity"], pre["rgb"], vals, ranges, cam,
                 dl_dimage=dl_dimage, threads=threads)
    g3 = preprocess_bwd(scene.mean3d, scene.log_scale, scene.quat, scene.opacity_logit, scene.sh,
                        scene.sh_degree, cam, bwd["grad2d"], threads=threads, **opt)
    out.update(dl_dimage=dl_dimage, grad2d=bwd["grad2d"], grads=g3, bwd_stats=bwd["stats"])
    return out
