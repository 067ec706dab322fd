"""Python binding of the library's C ABI, with torch tensors for device memory and streams.

The functions carry the C entry points' names (gs_preprocess, gs_bin_and_sort, gs_render_fwd,
gs_render_bwd, gs_preprocess_bwd). They allocate outputs with torch when the caller passes none,
marshal pointers and the current CUDA stream, and raise GsError on a non-zero status. All
arithmetic runs in libgs_gb300.so.

Dtypes: arrays the C ABI declares as uint32 (vals, tile ranges, contributor counts,
tiles_touched) are torch.int32 tensors holding the same bits; 64-bit keys are torch.int64.
"""
from __future__ import annotations

import ctypes as C
import dataclasses

import torch

from . import _abi
from ._abi import (GS_BWD_ADAPTIVE, GS_BWD_DIRECT, GS_BWD_SM, GS_BWD_WARP, GS_ERR_CAPACITY, GsError, check,
                   gs_camera, gs_options, gs_params, gs_proj)

__all__ = ["Proj", "BinResult", "StepContext", "gs_train_step_host", "make_camera", "make_options", "alloc_proj", "gs_preprocess",
           "gs_sort_workspace_bytes", "gs_bin_and_sort", "gs_bin_and_sort_async", "gs_render_fwd", "gs_render_bwd",
           "gs_preprocess_bwd",
           "gs_device_error", "GsError", "GS_BWD_DIRECT", "GS_BWD_WARP", "GS_BWD_ADAPTIVE", "GS_BWD_SM"]


_dummy = {}


def _ptr(t) -> int | None:
    """Device address of a tensor; an empty tensor gets the address of a small valid buffer
    (torch reports 0 for it, which the C ABI rejects as NULL)."""
    if t is None:
        return None
    if t.numel() == 0:
        key = str(t.device)
        if key not in _dummy:
            _dummy[key] = torch.zeros(64, dtype=torch.float32, device=t.device)
        return _dummy[key].data_ptr()
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def make_camera(cam) -> gs_camera:
    """gs_camera from any object with R (9), t (3), fx, fy, cx, cy, width, height, bg (3)."""
    c = gs_camera()
    c.R[:] = [float(v) for v in torch.as_tensor(cam.R, dtype=torch.float32).reshape(9).tolist()]
    c.t[:] = [float(v) for v in torch.as_tensor(cam.t, dtype=torch.float32).reshape(3).tolist()]
    c.fx, c.fy, c.cx, c.cy = float(cam.fx), float(cam.fy), float(cam.cx), float(cam.cy)
    c.width, c.height = int(cam.width), int(cam.height)
    c.bg[:] = [float(v) for v in torch.as_tensor(cam.bg, dtype=torch.float32).reshape(3).tolist()]
    return c


def make_options(sh_degree: int, bwd_mode: int | str = 0, adaptive_threshold: int = 0, staging: int = 0,
                 near_z: float = 0.0, lowpass: float = 0.0, jacobian_clamp: float = 0.0,
                 spin_limit: int = 0) -> gs_options:
    if isinstance(bwd_mode, str):
        bwd_mode = _abi.BWD_MODES[bwd_mode]
    return gs_options(bwd_mode=int(bwd_mode), adaptive_threshold=int(adaptive_threshold),
                      sh_degree=int(sh_degree), staging=int(staging), near_z=float(near_z),
                      lowpass=float(lowpass), jacobian_clamp=float(jacobian_clamp), spin_limit=int(spin_limit))


@dataclasses.dataclass
class Proj:
    rec: torch.Tensor            # [N, 12] float32: mean_x, mean_y, A, B, C, opacity, r, g, b, 0, 0, 0
    depth: torch.Tensor          # [N] float32
    radius: torch.Tensor         # [N] int32
    tiles_touched: torch.Tensor  # [N] int32 (uint32 bits)

    @property
    def n(self) -> int:
        return int(self.rec.shape[0])

    @property
    def mean2d(self):
        return self.rec[:, 0:2]

    @property
    def conic(self):
        return self.rec[:, 2:5]

    @property
    def opacity(self):
        return self.rec[:, 5]

    @property
    def rgb(self):
        return self.rec[:, 6:9]

    def struct(self) -> gs_proj:
        return gs_proj(rec=_ptr(self.rec), depth=_ptr(self.depth), radius=_ptr(self.radius),
                       tiles_touched=_ptr(self.tiles_touched), n=self.n)


def alloc_proj(n: int, device) -> Proj:
    return Proj(rec=torch.empty((n, 12), dtype=torch.float32, device=device),
                depth=torch.empty(n, dtype=torch.float32, device=device),
                radius=torch.empty(n, dtype=torch.int32, device=device),
                tiles_touched=torch.empty(n, dtype=torch.int32, device=device))


def proj_from_arrays(mean2d, conic, opacity, rgb, depth, radius, device) -> Proj:
    """A Proj built from separate (host or device) arrays, e.g. projected Gaussians made elsewhere."""
    n = int(torch.as_tensor(radius).shape[0])
    rec = torch.zeros((n, 12), dtype=torch.float32)
    rec[:, 0:2] = torch.as_tensor(mean2d, dtype=torch.float32)
    rec[:, 2:5] = torch.as_tensor(conic, dtype=torch.float32)
    rec[:, 5] = torch.as_tensor(opacity, dtype=torch.float32)
    rec[:, 6:9] = torch.as_tensor(rgb, dtype=torch.float32)
    return Proj(rec=rec.to(device), depth=torch.as_tensor(depth, dtype=torch.float32).to(device).contiguous(),
                radius=torch.as_tensor(radius, dtype=torch.int32).to(device).contiguous(),
                tiles_touched=torch.zeros(n, dtype=torch.int32, device=device))


def _params(mean3d, log_scale, quat, opacity_logit, sh) -> gs_params:
    for t in (mean3d, log_scale, quat, opacity_logit, sh):
        if t.dtype != torch.float32 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("parameters must be contiguous float32 CUDA tensors")
    return gs_params(mean3d=_ptr(mean3d), log_scale=_ptr(log_scale), quat=_ptr(quat),
                     opacity_logit=_ptr(opacity_logit), sh=_ptr(sh), n=int(mean3d.shape[0]))


def gs_preprocess(params: dict, cam, opt: gs_options, out: Proj | None = None, stream=None) -> Proj:
    """params: dict with mean3d [N,3], log_scale [N,3], quat [N,4], opacity_logit [N], sh [N,K,3]."""
    p = _params(params["mean3d"], params["log_scale"], params["quat"], params["opacity_logit"], params["sh"])
    if out is None:
        out = alloc_proj(p.n, params["mean3d"].device)
    c, ps = make_camera(cam) if not isinstance(cam, gs_camera) else cam, out.struct()
    check(_abi.load().gs_preprocess(C.byref(p), C.byref(c), C.byref(opt), C.byref(ps), _stream(stream)),
          "gs_preprocess")
    return out


def gs_sort_workspace_bytes(n: int, capacity: int, width: int, height: int) -> int:
    return int(_abi.load().gs_sort_workspace_bytes(int(n), int(capacity), int(width), int(height)))


@dataclasses.dataclass
class BinResult:
    keys: torch.Tensor | None   # [D] int64 (uint64 bits: tile << 32 | depth bits)
    vals: torch.Tensor          # [D] int32 Gaussian indices
    ranges: torch.Tensor        # [T, 2] int32: [start, end) per tile
    n_dup: int | torch.Tensor  # D (a device int64 tensor [1] from gs_bin_and_sort_async)


class SortBuffers:
    """Device buffers of gs_bin_and_sort, grown on demand and reused across calls."""

    def __init__(self, device):
        self.device = torch.device(device)
        self.capacity = 0
        self.workspace = None
        self.keys = None
        self.vals = None

    def ensure(self, n: int, capacity: int, width: int, height: int, want_keys: bool):
        need = gs_sort_workspace_bytes(n, capacity, width, height)
        if self.workspace is None or self.workspace.numel() < need:
            self.workspace = torch.empty(need, dtype=torch.uint8, device=self.device)
        if capacity > self.capacity or self.vals is None:
            self.vals = torch.empty(max(capacity, 1), dtype=torch.int32, device=self.device)
            self.keys = None
            self.capacity = capacity
        if want_keys and (self.keys is None or self.keys.numel() < self.vals.numel()):
            self.keys = torch.empty(self.vals.numel(), dtype=torch.int64, device=self.device)


def gs_bin_and_sort(proj: Proj, cam, opt: gs_options, capacity: int | None = None, buffers: SortBuffers | None = None,
                    want_keys: bool = True, ranges: torch.Tensor | None = None, stream=None) -> BinResult:
    """Tile duplication + stable radix sort + tile ranges. With capacity None the call retries
    once with the exact number of duplicates when the first capacity was too small."""
    c = make_camera(cam) if not isinstance(cam, gs_camera) else cam
    dev = proj.rec.device
    T = ((c.width + 15) // 16) * ((c.height + 15) // 16)
    if ranges is None:
        ranges = torch.empty((T, 2), dtype=torch.int32, device=dev)
    buffers = buffers or SortBuffers(dev)
    cap = capacity if capacity is not None else max(buffers.capacity, 1 << 16, 4 * proj.n)
    lib = _abi.load()
    ps = proj.struct()
    for attempt in range(2):
        buffers.ensure(proj.n, cap, c.width, c.height, want_keys)
        d = C.c_int64(0)
        st = lib.gs_bin_and_sort(C.byref(ps), C.byref(c), C.byref(opt), _ptr(buffers.workspace),
                                 buffers.workspace.numel(), _ptr(buffers.keys) if want_keys else None,
                                 _ptr(buffers.vals), cap, C.byref(d), _ptr(ranges), _stream(stream))
        if st == GS_ERR_CAPACITY and capacity is None and attempt == 0:
            cap = int(d.value)
            continue
        check(st, "gs_bin_and_sort")
        D = int(d.value)
        return BinResult(keys=buffers.keys[:D] if want_keys else None, vals=buffers.vals[:D], ranges=ranges, n_dup=D)
    raise AssertionError("unreachable")


def gs_bin_and_sort_async(proj: Proj, cam, opt: gs_options, capacity: int, buffers: SortBuffers | None = None,
                          want_keys: bool = False, ranges: torch.Tensor | None = None,
                          n_dup: torch.Tensor | None = None, static_workspace: bool = False,
                          stream=None) -> BinResult:
    """gs_bin_and_sort without host synchronisation (capturable in a CUDA graph). The result's
    vals / keys span the whole capacity and its n_dup is a device int64 tensor [1] holding D;
    overflowing the capacity leaves empty ranges and a device check error."""
    c = make_camera(cam) if not isinstance(cam, gs_camera) else cam
    dev = proj.rec.device
    T = ((c.width + 15) // 16) * ((c.height + 15) // 16)
    if ranges is None:
        ranges = torch.empty((T, 2), dtype=torch.int32, device=dev)
    if n_dup is None:
        n_dup = torch.zeros(1, dtype=torch.int64, device=dev)
    buffers = buffers or SortBuffers(dev)
    buffers.ensure(0 if static_workspace else proj.n, capacity, c.width, c.height, want_keys)
    ps = proj.struct()
    ws = None if static_workspace else buffers.workspace
    check(_abi.load().gs_bin_and_sort_async(C.byref(ps), C.byref(c), C.byref(opt), _ptr(ws) if ws is not None else None,
                                            ws.numel() if ws is not None else 0,
                                            _ptr(buffers.keys) if want_keys else None, _ptr(buffers.vals), capacity,
                                            _ptr(n_dup), _ptr(ranges), _stream(stream)), "gs_bin_and_sort_async")
    return BinResult(keys=buffers.keys if want_keys else None, vals=buffers.vals, ranges=ranges, n_dup=n_dup)


def gs_render_fwd(proj: Proj, vals: torch.Tensor, ranges: torch.Tensor, cam, opt: gs_options, out=None, stream=None):
    """Returns (image [3,H,W] float32, t_final [H,W] float32, n_contrib [H,W] int32)."""
    c = make_camera(cam) if not isinstance(cam, gs_camera) else cam
    dev = proj.rec.device
    if out is None:
        out = (torch.empty((3, c.height, c.width), dtype=torch.float32, device=dev),
               torch.empty((c.height, c.width), dtype=torch.float32, device=dev),
               torch.empty((c.height, c.width), dtype=torch.int32, device=dev))
    image, t_final, n_contrib = out
    ps = proj.struct()
    check(_abi.load().gs_render_fwd(C.byref(ps), _ptr(vals), _ptr(ranges), C.byref(c), C.byref(opt), _ptr(image),
                                    _ptr(t_final), _ptr(n_contrib), _stream(stream)), "gs_render_fwd")
    return image, t_final, n_contrib


def gs_render_bwd(proj: Proj, vals, ranges, cam, opt: gs_options, dl_dimage, t_final, n_contrib, grad2d=None,
                  stream=None) -> torch.Tensor:
    """Returns grad2d [N, 12] float32 (columns: dmean_x, dmean_y, dA, dB, dC, dopacity, dr, dg, db, 0, 0, 0)."""
    c = make_camera(cam) if not isinstance(cam, gs_camera) else cam
    if grad2d is None:
        grad2d = torch.empty((proj.n, 12), dtype=torch.float32, device=proj.rec.device)
    ps = proj.struct()
    check(_abi.load().gs_render_bwd(C.byref(ps), _ptr(vals), _ptr(ranges), C.byref(c), C.byref(opt),
                                    _ptr(dl_dimage.contiguous()), _ptr(t_final), _ptr(n_contrib), _ptr(grad2d),
                                    _stream(stream)), "gs_render_bwd")
    return grad2d


def gs_render_bwd_sqerr(proj: Proj, vals, ranges, cam, opt: gs_options, image, target, t_final, n_contrib,
                        grad2d=None, loss=None, stream=None) -> torch.Tensor:
    """gs_render_bwd with dL/dimage = image - target formed inside the kernel (the squared-error
    loss 0.5 |image - target|^2, written to `loss`, a device float tensor [1], when given).
    Returns grad2d [N, 12]."""
    c = make_camera(cam) if not isinstance(cam, gs_camera) else cam
    if grad2d is None:
        grad2d = torch.empty((proj.n, 12), dtype=torch.float32, device=proj.rec.device)
    ps = proj.struct()
    check(_abi.load().gs_render_bwd_sqerr(C.byref(ps), _ptr(vals), _ptr(ranges), C.byref(c), C.byref(opt),
                                          _ptr(image.contiguous()), _ptr(target.contiguous()), _ptr(t_final),
                                          _ptr(n_contrib), _ptr(grad2d), _ptr(loss) if loss is not None else None,
                                          _stream(stream)), "gs_render_bwd_sqerr")
    return grad2d


def alloc_param_grads(params: dict) -> dict:
    return {"mean3d": torch.zeros_like(params["mean3d"]), "log_scale": torch.zeros_like(params["log_scale"]),
            "quat": torch.zeros_like(params["quat"]), "opacity_logit": torch.zeros_like(params["opacity_logit"]),
            "sh": torch.zeros_like(params["sh"])}


def gs_preprocess_bwd(params: dict, cam, opt: gs_options, proj: Proj, grad2d, out: dict | None = None,
                      accumulate: bool = False, stream=None) -> dict:
    p = _params(params["mean3d"], params["log_scale"], params["quat"], params["opacity_logit"], params["sh"])
    if out is None:
        out = alloc_param_grads(params)
    c = make_camera(cam) if not isinstance(cam, gs_camera) else cam
    ps = proj.struct()
    check(_abi.load().gs_preprocess_bwd(C.byref(p), C.byref(c), C.byref(opt), C.byref(ps), _ptr(grad2d),
                                        _ptr(out["mean3d"]), _ptr(out["log_scale"]), _ptr(out["quat"]),
                                        _ptr(out["opacity_logit"]), _ptr(out["sh"]), int(bool(accumulate)),
                                        _stream(stream)), "gs_preprocess_bwd")
    return out


def gs_preprocess_bwd_stats(params: dict, cam, opt: gs_options, proj: Proj, grad2d, grad_norm_accum, view_count,
                            max_radius, grad_mag=None, ndc: bool = False, out: dict | None = None,
                            accumulate: bool = False, stream=None) -> dict:
    """gs_preprocess_bwd that also adds the view's densification statistics (and, with grad_mag,
    the 2-norm of the view's parameter gradients) in the same kernel."""
    p = _params(params["mean3d"], params["log_scale"], params["quat"], params["opacity_logit"], params["sh"])
    if out is None:
        out = alloc_param_grads(params)
    c = make_camera(cam) if not isinstance(cam, gs_camera) else cam
    ps = proj.struct()
    st = _abi.gs_densify_outputs(grad_norm_accum=_ptr(grad_norm_accum), view_count=_ptr(view_count),
                                 max_radius=_ptr(max_radius), grad_mag=_ptr(grad_mag) if grad_mag is not None else None,
                                 ndc=int(bool(ndc)))
    check(_abi.load().gs_preprocess_bwd_stats(C.byref(p), C.byref(c), C.byref(opt), C.byref(ps), _ptr(grad2d),
                                              _ptr(out["mean3d"]), _ptr(out["log_scale"]), _ptr(out["quat"]),
                                              _ptr(out["opacity_logit"]), _ptr(out["sh"]), int(bool(accumulate)),
                                              C.byref(st), _stream(stream)), "gs_preprocess_bwd_stats")
    return out


PARAM_NAMES = ("mean3d", "log_scale", "quat", "opacity_logit", "sh")


def _tensors(d: dict) -> _abi.gs_tensors:
    for k in PARAM_NAMES:
        t = d[k]
        if t.dtype != torch.float32 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("Adam tensors must be contiguous float32 CUDA tensors")
    return _abi.gs_tensors(mean3d=_ptr(d["mean3d"]), log_scale=_ptr(d["log_scale"]), quat=_ptr(d["quat"]),
                           opacity_logit=_ptr(d["opacity_logit"]), sh=_ptr(d["sh"]), n=int(d["mean3d"].shape[0]))


def make_adam_options(lr: dict, step: int, sh_degree: int, beta1: float = 0.0, beta2: float = 0.0,
                      eps: float = 0.0) -> _abi.gs_adam_options:
    """lr: learning rates keyed mean3d, log_scale, quat, opacity, sh_dc, sh_rest."""
    return _abi.gs_adam_options(lr_mean3d=lr["mean3d"], lr_log_scale=lr["log_scale"], lr_quat=lr["quat"],
                                lr_opacity=lr["opacity"], lr_sh_dc=lr["sh_dc"], lr_sh_rest=lr["sh_rest"],
                                beta1=beta1, beta2=beta2, eps=eps, step=int(step), sh_degree=int(sh_degree))


def gs_adam_step(params: dict, grads: dict, exp_avg: dict, exp_avg_sq: dict, radius, opt: _abi.gs_adam_options,
                 stream=None) -> None:
    """Sparse Adam step in place on params / exp_avg / exp_avg_sq for the Gaussians with radius > 0."""
    P, G, M, V = _tensors(params), _tensors(grads), _tensors(exp_avg), _tensors(exp_avg_sq)
    check(_abi.load().gs_adam_step(C.byref(P), C.byref(G), C.byref(M), C.byref(V), _ptr(radius), C.byref(opt),
                                   _stream(stream)), "gs_adam_step")


def gs_densify_stats(proj: Proj, grad2d, width: int, height: int, grad_norm_accum, view_count, max_radius,
                     ndc: bool = False, param_grads: dict | None = None, grad_mag=None, sh_degree: int = 3,
                     stream=None) -> None:
    """Adds one view's densification statistics in place (see include/gs.h); with param_grads, also
    writes each Gaussian's parameter-gradient 2-norm into grad_mag."""
    ps = proj.struct()
    pg = C.byref(_tensors(param_grads)) if param_grads is not None else None
    check(_abi.load().gs_densify_stats(C.byref(ps), _ptr(grad2d), int(width), int(height), int(bool(ndc)),
                                       _ptr(grad_norm_accum), _ptr(view_count), _ptr(max_radius), pg,
                                       _ptr(grad_mag) if grad_mag is not None else None, int(sh_degree),
                                       _stream(stream)), "gs_densify_stats")


def gs_loss_l1_dssim(image, target, lam: float = 0.2, workspace=None, out=None, stream=None):
    """(loss, dL/dimage) of the L1 + D-SSIM image loss; loss is a one-element device tensor."""
    _, h, w = image.shape
    need = int(_abi.load().gs_loss_workspace_bytes(int(w), int(h)))
    if workspace is None or workspace.numel() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device=image.device)
    loss, dl = out if out is not None else (torch.empty(1, device=image.device), torch.empty_like(image))
    check(_abi.load().gs_loss_l1_dssim(_ptr(image.contiguous()), _ptr(target.contiguous()), int(w), int(h),
                                       float(lam), _ptr(workspace), need, _ptr(loss), _ptr(dl), _stream(stream)),
          "gs_loss_l1_dssim")
    return loss, dl


def gs_preprocess2d(params: dict, cam, opt: gs_options, out: Proj | None = None, rec2d=None, stream=None):
    """Surfel preprocessing: (Proj for the binning, rec2d [N, 16])."""
    p = _params(params["mean3d"], params["log_scale"], params["quat"], params["opacity_logit"], params["sh"])
    dev = params["mean3d"].device
    if out is None:
        out = alloc_proj(p.n, dev)
    if rec2d is None:
        rec2d = torch.empty((p.n, 16), dtype=torch.float32, device=dev)
    c = make_camera(cam) if not isinstance(cam, gs_camera) else cam
    ps = out.struct()
    check(_abi.load().gs_preprocess2d(C.byref(p), C.byref(c), C.byref(opt), C.byref(ps), _ptr(rec2d), _stream(stream)),
          "gs_preprocess2d")
    return out, rec2d


def gs_render2d_fwd(rec2d, vals, ranges, cam, opt: gs_options, out=None, stream=None):
    c = make_camera(cam) if not isinstance(cam, gs_camera) else cam
    dev = rec2d.device
    if out is None:
        out = (torch.empty((3, c.height, c.width), dtype=torch.float32, device=dev),
               torch.empty((c.height, c.width), dtype=torch.float32, device=dev),
               torch.empty((c.height, c.width), dtype=torch.int32, device=dev))
    image, t_final, n_contrib = out
    check(_abi.load().gs_render2d_fwd(_ptr(rec2d), int(rec2d.shape[0]), _ptr(vals), _ptr(ranges), C.byref(c),
                                      C.byref(opt), _ptr(image), _ptr(t_final), _ptr(n_contrib), _stream(stream)),
          "gs_render2d_fwd")
    return image, t_final, n_contrib


def gs_render2d_bwd(rec2d, vals, ranges, cam, opt: gs_options, dl_dimage, t_final, n_contrib, grad2d=None, stream=None):
    c = make_camera(cam) if not isinstance(cam, gs_camera) else cam
    if grad2d is None:
        grad2d = torch.empty((rec2d.shape[0], 16), dtype=torch.float32, device=rec2d.device)
    check(_abi.load().gs_render2d_bwd(_ptr(rec2d), int(rec2d.shape[0]), _ptr(vals), _ptr(ranges), C.byref(c),
                                      C.byref(opt), _ptr(dl_dimage.contiguous()), _ptr(t_final), _ptr(n_contrib),
                                      _ptr(grad2d), _stream(stream)), "gs_render2d_bwd")
    return grad2d


def gs_preprocess2d_bwd(params: dict, cam, opt: gs_options, proj: Proj, grad2d, out: dict | None = None,
                        accumulate: bool = False, stream=None) -> dict:
    p = _params(params["mean3d"], params["log_scale"], params["quat"], params["opacity_logit"], params["sh"])
    if out is None:
        out = alloc_param_grads(params)
    c = make_camera(cam) if not isinstance(cam, gs_camera) else cam
    ps = proj.struct()
    check(_abi.load().gs_preprocess2d_bwd(C.byref(p), C.byref(c), C.byref(opt), C.byref(ps), _ptr(grad2d),
                                          _ptr(out["mean3d"]), _ptr(out["log_scale"]), _ptr(out["quat"]),
                                          _ptr(out["opacity_logit"]), _ptr(out["sh"]), int(bool(accumulate)),
                                          _stream(stream)), "gs_preprocess2d_bwd")
    return out


def gs_kernel_launches() -> int:
    """Number of kernels this library has launched in the process (a host-side counter; kernels
    replayed from a CUDA graph are counted once, at capture)."""
    return int(_abi.load().gs_kernel_launches())


def gs_device_error(stream=None) -> int:
    """Synchronises and returns (and clears) the device error status: 0, GS_ERR_TIMEOUT or GS_ERR_DEVICE_CHECK."""
    return int(_abi.load().gs_device_error(_stream(stream)))


class StepContext:
    """Device buffers of the end-to-end training step with host buffers (gs_step_context_create):
    n Gaussians of SH degree `sh_degree`, images of at most max_width x max_height, `capacity`
    duplicates. Freed by close() (or when garbage-collected)."""

    def __init__(self, n: int, sh_degree: int, max_width: int, max_height: int, capacity: int):
        lib = _abi.load()
        h = C.c_void_p()
        _abi.check(lib.gs_step_context_create(int(n), int(sh_degree), int(max_width), int(max_height), int(capacity),
                                              C.byref(h)), "gs_step_context_create")
        self._h = h
        self.n, self.sh_degree, self.capacity = int(n), int(sh_degree), int(capacity)

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _abi.check(_abi.load().gs_step_context_destroy(self._h), "gs_step_context_destroy")
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _host_ptr(t) -> int:
    if t.device.type != "cpu" or not t.is_contiguous() or t.dtype != torch.float32:
        raise ValueError("host buffers must be contiguous float32 CPU tensors")
    return t.data_ptr()


def gs_train_step_host(ctx: StepContext, host_params: dict, host_target, cam, opt: gs_options, host_grads: dict,
                       host_loss=None, host_n_dup=None, stream=None) -> None:
    """One training step of one view through the C ABI with host buffers (gs_train_step_host): the
    parameters and the target are copied in, the step runs on the device, the parameter gradients
    (and the loss and D when given: a 1-element float32 / int64 CPU tensor) are copied back into
    `host_grads`. Enqueued on `stream`; synchronise it before reading the outputs."""
    p = gs_params(mean3d=_host_ptr(host_params["mean3d"]), log_scale=_host_ptr(host_params["log_scale"]),
                  quat=_host_ptr(host_params["quat"]), opacity_logit=_host_ptr(host_params["opacity_logit"]),
                  sh=_host_ptr(host_params["sh"]), n=int(host_params["mean3d"].shape[0]))
    g = _abi.gs_tensors(mean3d=_host_ptr(host_grads["mean3d"]), log_scale=_host_ptr(host_grads["log_scale"]),
                        quat=_host_ptr(host_grads["quat"]), opacity_logit=_host_ptr(host_grads["opacity_logit"]),
                        sh=_host_ptr(host_grads["sh"]), n=int(host_grads["mean3d"].shape[0]))
    if host_n_dup is not None and (host_n_dup.device.type != "cpu" or host_n_dup.dtype != torch.int64):
        raise ValueError("host_n_dup must be an int64 CPU tensor")
    c = make_camera(cam)
    _abi.check(_abi.load().gs_train_step_host(ctx._h, C.byref(p), _host_ptr(host_target), C.byref(c), C.byref(opt),
                                              C.byref(g), None if host_loss is None else _host_ptr(host_loss),
                                              None if host_n_dup is None else host_n_dup.data_ptr(), _stream(stream)),
               "gs_train_step_host")
