"""Float64 CPU oracle for the tile-based 3D Gaussian splatting training step.

TEST INFRASTRUCTURE. Only the test suite, the smoke check (`__graft_entry__.smoke`) and the
benchmark's CPU-baseline leg may import this package. It shares no code with the CUDA library
and the CUDA library never imports it.

    _lib.py        ctypes binding of gs_oracle.cpp (preprocess, binning + stable sort, render
                   forward/backward with marginal-decision flags, preprocess backward by dual numbers)
    brute.py       numpy brute-force per-pixel renderer for tiny scenes (no tiles list, no sort code)
    gs_oracle.cpp  the float64 implementation (3D Gaussians, and surfels of 2D Gaussian splatting)
    optim.py       numpy sparse Adam (the update phase after the backward)
"""
from ._lib import (MARGINAL, bin_and_sort, build, preprocess, preprocess2d, preprocess2d_bwd, preprocess_bwd,
                   quat_to_rotmat, render, render2d, sh_basis, view_step, view_step2d)

__all__ = ["MARGINAL", "bin_and_sort", "build", "preprocess", "preprocess2d", "preprocess2d_bwd", "preprocess_bwd",
           "quat_to_rotmat", "render", "render2d", "sh_basis", "view_step", "view_step2d"]
