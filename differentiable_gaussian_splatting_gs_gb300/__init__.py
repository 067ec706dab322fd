"""GB300 (sm_103a) library for the training step of a tile-based 3D Gaussian splatting rasterizer.

    include/gs.h      the C ABI (gs_preprocess, gs_bin_and_sort, gs_render_fwd, gs_render_bwd,
                      gs_preprocess_bwd)
    csrc/             the CUDA kernels and the C-ABI implementation
    build.py          nvcc build of libgs_gb300.so (in-tree, sm_103a)
    _abi.py           ctypes structs and prototypes
    api.py            torch-facing binding with the same names
    step.py           one training step of one or more views through the five calls
"""
from .api import (BinResult, GsError, Proj, SortBuffers, alloc_param_grads, alloc_proj, gs_bin_and_sort,
                  gs_device_error, gs_preprocess, gs_preprocess_bwd, gs_render_bwd, gs_render_fwd,
                  gs_sort_workspace_bytes, make_camera, make_options, proj_from_arrays)

__all__ = ["BinResult", "GsError", "Proj", "SortBuffers", "alloc_param_grads", "alloc_proj", "gs_bin_and_sort",
           "gs_device_error", "gs_preprocess", "gs_preprocess_bwd", "gs_render_bwd", "gs_render_fwd",
           "gs_sort_workspace_bytes", "make_camera", "make_options", "proj_from_arrays"]
