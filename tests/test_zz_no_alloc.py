"""The sort entry point that allocates nothing (gs_bin_and_sort_static) against the regular one.

Some callers cannot hand the library a workspace: a plug-in that only receives its input and
output buffers from a host application which owns all device memory under a fixed budget (the
plug-in may not call cudaMalloc itself), or a real-time loop in which an allocation could stall or
fail in the middle of a frame. gs_bin_and_sort_static serves them from a 32 MiB device array
inside the library. This file is collected last on purpose: it
calls the static entry point twice in a row (the array keeps the previous call's contents) and
must give exactly what gs_bin_and_sort gives, whether it runs alone or after the other tests.
"""
import ctypes as C

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import gs_scenes  # noqa: E402
import oracle  # noqa: E402
from differentiable_gaussian_splatting_gs_gb300 import _abi, api  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _proj(s, cam):
    pre = oracle.preprocess(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, s.sh_degree, cam)
    return api.proj_from_arrays(pre["mean2d"], pre["conic"], pre["opacity"], pre["rgb"], pre["depth"],
                                pre["radius"], DEV)


def _static_call(proj, cam, opt, capacity):
    lib = _abi.load()
    c = api.make_camera(cam)
    T = ((c.width + 15) // 16) * ((c.height + 15) // 16)
    keys = torch.full((max(capacity, 1),), -1, dtype=torch.int64, device=DEV)
    vals = torch.full((max(capacity, 1),), -1, dtype=torch.int32, device=DEV)
    ranges = torch.full((T, 2), -1, dtype=torch.int32, device=DEV)
    d = C.c_int64(0)
    ps = proj.struct()
    st = lib.gs_bin_and_sort_static(C.byref(ps), C.byref(c), C.byref(opt), keys.data_ptr(), vals.data_ptr(),
                                    capacity, C.byref(d), ranges.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return st, int(d.value), keys, vals, ranges


@pytest.mark.parametrize("cfg,n,res", [(0, None, 1.0), (1, 20_000, 1.0)])
def test_static_workspace_sort_matches_regular_entry_point_twice(cfg, n, res):
    s = gs_scenes.make_scene(cfg, n=n, res_scale=res)
    cam = s.cameras[0]
    opt = api.make_options(s.sh_degree)
    proj = _proj(s, cam)
    ref = api.gs_bin_and_sort(proj, cam, opt)
    cap = ref.n_dup + 1000
    for _ in range(2):
        st, D, keys, vals, ranges = _static_call(proj, cam, opt, cap)
        assert st == _abi.GS_OK, _abi.load().gs_last_error_message()
        assert D == ref.n_dup
        assert torch.equal(vals[:D], ref.vals) and torch.equal(keys[:D], ref.keys)
        assert torch.equal(ranges, ref.ranges)
        assert api.gs_device_error() == _abi.GS_OK


def test_static_workspace_rejects_requests_beyond_its_size():
    # two million culled Gaussians (all inputs valid, zeroed) need more than 32 MiB of workspace:
    # the call must refuse before touching the device
    n = 2_000_000
    cam = gs_scenes.make_scene(0).cameras[0]
    proj = api.Proj(rec=torch.zeros((n, 12), dtype=torch.float32, device=DEV),
                    depth=torch.zeros(n, dtype=torch.float32, device=DEV),
                    radius=torch.zeros(n, dtype=torch.int32, device=DEV),
                    tiles_touched=torch.zeros(n, dtype=torch.int32, device=DEV))
    cap = 1000
    assert api.gs_sort_workspace_bytes(n, cap, cam.width, cam.height) > _abi.GS_STATIC_SORT_WORKSPACE_BYTES
    st, D, _, _, _ = _static_call(proj, cam, api.make_options(0), cap)
    assert st == _abi.GS_ERR_ARG
    assert b"static workspace" in _abi.load().gs_last_error_message()
