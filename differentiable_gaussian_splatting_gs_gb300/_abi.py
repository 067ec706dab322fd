"""ctypes binding of the C ABI in include/gs.h (argument marshalling only).

Every compute step runs in the CUDA library libgs_gb300.so; this module only converts Python
and torch objects into the structs and pointers the ABI takes. Loading fails loudly when the
library has not been built: there is no fallback implementation.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libgs_gb300.so")

GS_OK = 0
GS_ERR_ARG = -1
GS_ERR_CAPACITY = -2
GS_ERR_CUDA = -3
GS_ERR_TIMEOUT = -4
GS_ERR_DEVICE_CHECK = -5

GS_BWD_DEFAULT, GS_BWD_DIRECT, GS_BWD_WARP, GS_BWD_ADAPTIVE, GS_BWD_SM = 0, 1, 2, 3, 4
GS_STAGE_DEFAULT, GS_STAGE_BULK, GS_STAGE_LOADS = 0, 1, 2

BWD_MODES = {"direct": GS_BWD_DIRECT, "warp": GS_BWD_WARP, "adaptive": GS_BWD_ADAPTIVE, "sm": GS_BWD_SM}

# every symbol include/gs.h declares
EXPORTS = ("gs_preprocess", "gs_sort_workspace_bytes", "gs_bin_and_sort", "gs_render_fwd", "gs_render_bwd",
           "gs_preprocess_bwd", "gs_status_string", "gs_last_error_message", "gs_device_error",
           "gs_selftest_timeout", "gs_kernel_launches", "gs_version", "gs_bin_and_sort_static", "gs_adam_step",
           "gs_densify_stats", "gs_loss_workspace_bytes", "gs_loss_l1_dssim", "gs_preprocess2d",
           "gs_render2d_fwd", "gs_render2d_bwd", "gs_preprocess2d_bwd", "gs_bin_and_sort_async",
           "gs_preprocess_bwd_stats", "gs_selftest_sort_timeout", "gs_render_bwd_sqerr",
           "gs_step_context_create", "gs_step_context_destroy", "gs_train_step_host")
GS_STATIC_SORT_WORKSPACE_BYTES = 32 << 20
GS_SELFTEST_SORT_WORKSPACE_BYTES = 128 << 10


class gs_camera(C.Structure):
    _fields_ = [("R", C.c_float * 9), ("t", C.c_float * 3), ("fx", C.c_float), ("fy", C.c_float),
                ("cx", C.c_float), ("cy", C.c_float), ("width", C.c_int32), ("height", C.c_int32),
                ("bg", C.c_float * 3)]


class gs_options(C.Structure):
    _fields_ = [("bwd_mode", C.c_int32), ("adaptive_threshold", C.c_int32), ("sh_degree", C.c_int32),
                ("staging", C.c_int32), ("near_z", C.c_float), ("lowpass", C.c_float),
                ("jacobian_clamp", C.c_float), ("spin_limit", C.c_uint32)]


class gs_params(C.Structure):
    _fields_ = [("mean3d", C.c_void_p), ("log_scale", C.c_void_p), ("quat", C.c_void_p),
                ("opacity_logit", C.c_void_p), ("sh", C.c_void_p), ("n", C.c_int64)]


class gs_proj(C.Structure):
    _fields_ = [("rec", C.c_void_p), ("depth", C.c_void_p), ("radius", C.c_void_p),
                ("tiles_touched", C.c_void_p), ("n", C.c_int64)]


class gs_densify_outputs(C.Structure):
    _fields_ = [("grad_norm_accum", C.c_void_p), ("view_count", C.c_void_p), ("max_radius", C.c_void_p),
                ("grad_mag", C.c_void_p), ("ndc", C.c_int32)]


class gs_tensors(C.Structure):
    _fields_ = [("mean3d", C.c_void_p), ("log_scale", C.c_void_p), ("quat", C.c_void_p),
                ("opacity_logit", C.c_void_p), ("sh", C.c_void_p), ("n", C.c_int64)]


class gs_adam_options(C.Structure):
    _fields_ = [("lr_mean3d", C.c_float), ("lr_log_scale", C.c_float), ("lr_quat", C.c_float),
                ("lr_opacity", C.c_float), ("lr_sh_dc", C.c_float), ("lr_sh_rest", C.c_float),
                ("beta1", C.c_float), ("beta2", C.c_float), ("eps", C.c_float), ("step", C.c_int32),
                ("sh_degree", C.c_int32)]


class GsError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: status {status}: {message}")
        self.status = status


_lock = threading.Lock()
_lib = None


def load():
    """Loads libgs_gb300.so (built by `build()`); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; call __graft_entry__.build() or "
                               "differentiable_gaussian_splatting_gs_gb300.build.build_library()")
        lib = C.CDLL(LIB_PATH)
        P, I64, I32 = C.c_void_p, C.c_int64, C.c_int32
        pcam, popt = C.POINTER(gs_camera), C.POINTER(gs_options)
        ppar, pproj = C.POINTER(gs_params), C.POINTER(gs_proj)
        lib.gs_preprocess.argtypes = [ppar, pcam, popt, pproj, P]
        lib.gs_sort_workspace_bytes.argtypes = [I64, I64, I32, I32]
        lib.gs_sort_workspace_bytes.restype = C.c_size_t
        lib.gs_bin_and_sort.argtypes = [pproj, pcam, popt, P, C.c_size_t, P, P, I64, C.POINTER(I64), P, P]
        lib.gs_render_fwd.argtypes = [pproj, P, P, pcam, popt, P, P, P, P]
        lib.gs_render_bwd.argtypes = [pproj, P, P, pcam, popt, P, P, P, P, P]
        lib.gs_render_bwd_sqerr.argtypes = [pproj, P, P, pcam, popt, P, P, P, P, P, P, P]
        lib.gs_render_bwd_sqerr.restype = C.c_int
        lib.gs_preprocess_bwd.argtypes = [ppar, pcam, popt, pproj, P, P, P, P, P, P, I32, P]
        lib.gs_preprocess_bwd_stats.argtypes = [ppar, pcam, popt, pproj, P, P, P, P, P, P, I32,
                                                C.POINTER(gs_densify_outputs), P]
        lib.gs_preprocess_bwd_stats.restype = C.c_int
        lib.gs_status_string.argtypes = [C.c_int]
        lib.gs_status_string.restype = C.c_char_p
        lib.gs_last_error_message.argtypes = []
        lib.gs_last_error_message.restype = C.c_char_p
        lib.gs_device_error.argtypes = [P]
        lib.gs_version.argtypes = []
        lib.gs_selftest_timeout.argtypes = [C.c_uint32, P]
        lib.gs_selftest_sort_timeout.argtypes = [P, C.c_size_t, C.c_uint32, P]
        lib.gs_selftest_sort_timeout.restype = C.c_int
        lib.gs_bin_and_sort_static.argtypes = [pproj, pcam, popt, P, P, I64, C.POINTER(I64), P, P]
        lib.gs_bin_and_sort_static.restype = C.c_int
        lib.gs_bin_and_sort_async.argtypes = [pproj, pcam, popt, P, C.c_size_t, P, P, I64, P, P, P]
        lib.gs_bin_and_sort_async.restype = C.c_int
        lib.gs_kernel_launches.argtypes = []
        lib.gs_kernel_launches.restype = C.c_int64
        pten = C.POINTER(gs_tensors)
        lib.gs_adam_step.argtypes = [pten, pten, pten, pten, P, C.POINTER(gs_adam_options), P]
        lib.gs_adam_step.restype = C.c_int
        lib.gs_densify_stats.argtypes = [pproj, P, I32, I32, I32, P, P, P, pten, P, I32, P]
        lib.gs_densify_stats.restype = C.c_int
        lib.gs_loss_workspace_bytes.argtypes = [I32, I32]
        lib.gs_loss_workspace_bytes.restype = C.c_size_t
        lib.gs_loss_l1_dssim.argtypes = [P, P, I32, I32, C.c_float, P, C.c_size_t, P, P, P]
        lib.gs_loss_l1_dssim.restype = C.c_int
        lib.gs_preprocess2d.argtypes = [ppar, pcam, popt, pproj, P, P]
        lib.gs_render2d_fwd.argtypes = [P, I64, P, P, pcam, popt, P, P, P, P]
        lib.gs_render2d_bwd.argtypes = [P, I64, P, P, pcam, popt, P, P, P, P, P]
        lib.gs_preprocess2d_bwd.argtypes = [ppar, pcam, popt, pproj, P, P, P, P, P, P, I32, P]
        for name in ("gs_preprocess2d", "gs_render2d_fwd", "gs_render2d_bwd", "gs_preprocess2d_bwd"):
            getattr(lib, name).restype = C.c_int
        lib.gs_step_context_create.argtypes = [I64, I32, I32, I32, I64, C.POINTER(C.c_void_p)]
        lib.gs_step_context_create.restype = C.c_int
        lib.gs_step_context_destroy.argtypes = [P]
        lib.gs_step_context_destroy.restype = C.c_int
        lib.gs_train_step_host.argtypes = [P, ppar, P, pcam, popt, C.POINTER(gs_tensors), P, P, P]
        lib.gs_train_step_host.restype = C.c_int
        for name in ("gs_preprocess", "gs_bin_and_sort", "gs_render_fwd", "gs_render_bwd",
                     "gs_preprocess_bwd", "gs_device_error", "gs_version", "gs_selftest_timeout"):
            getattr(lib, name).restype = C.c_int
        _lib = lib
        return lib


def check(status: int, where: str) -> int:
    if status != GS_OK:
        lib = load()
        msg = lib.gs_last_error_message().decode(errors="replace")
        raise GsError(status, where, msg or lib.gs_status_string(status).decode())
    return status
