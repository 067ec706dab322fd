"""Host-side checks of the C-ABI library that need no GPU: it builds, loads, exports every entry
point include/gs.h declares, sizes the sort workspace, and rejects bad arguments before touching
the device."""
import ctypes as C
import os
import re

import pytest

import __graft_entry__
from differentiable_gaussian_splatting_gs_gb300 import _abi, api

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return _abi.load()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "gs.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gs_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_five_phases():
    names = declared_symbols()
    for n in ("gs_preprocess", "gs_bin_and_sort", "gs_render_fwd", "gs_render_bwd", "gs_preprocess_bwd"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert set(names) == set(_abi.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    assert lib.gs_version() >> 16 == 1
    for st in (_abi.GS_OK, _abi.GS_ERR_ARG, _abi.GS_ERR_CAPACITY, _abi.GS_ERR_CUDA, _abi.GS_ERR_TIMEOUT,
               _abi.GS_ERR_DEVICE_CHECK):
        assert lib.gs_status_string(st).decode().startswith("GS_")


def test_workspace_size_matches_the_documented_layout(lib):
    a = lib.gs_sort_workspace_bytes(1000, 10_000, 128, 128)
    n, T = 1_000_000, 82 * 53
    b = lib.gs_sort_workspace_bytes(n, 10_000_000, 1297, 840)
    assert 0 < a < b
    # counting tile pass in two levels: depth sort and packed rectangles (24 bytes per Gaussian), the
    # coarse lists (4 bytes per duplicate of capacity), the chunk x super-tile table (super-tiles of
    # 4x4 tiles, here 21 x 14; rows are chunks of at most 256 Gaussians or about 8192 coarse entries)
    # and the fine counts (16 words per 256-entry segment)
    ts = ((82 + 3) // 4) * ((53 + 3) // 4)
    rows = (n + 255) // 256 + 10_000_000 // 8192 + 1
    assert b >= 24 * n + 4 * 10_000_000 + 4 * ts * rows
    small = lib.gs_sort_workspace_bytes(n, 1, 1297, 840)
    assert 4 * 10_000_000 < b - small <= 4.25 * 10_000_000 + 4 * ts * (10_000_000 // 8192) * (1 + 1 / 512) + 65536
    # more than 49,152 tiles: radix tile passes, 12 more bytes per duplicate of capacity
    big1 = lib.gs_sort_workspace_bytes(n, 1_000_000, 4112, 4112)
    big2 = lib.gs_sort_workspace_bytes(n, 2_000_000, 4112, 4112)
    assert big2 - big1 >= 12 * 1_000_000
    assert lib.gs_sort_workspace_bytes(-1, 0, 1, 1) == 0
    assert lib.gs_sort_workspace_bytes(10, 10, 0, 16) == 0


def _cam(w=64, h=64, f=64.0):
    c = _abi.gs_camera()
    c.R[:] = [1, 0, 0, 0, 1, 0, 0, 0, 1]
    c.fx = c.fy = f
    c.cx, c.cy, c.width, c.height = w / 2, h / 2, w, h
    return c


def test_bad_arguments_are_rejected_on_the_host(lib):
    cam, opt = _cam(), api.make_options(0)
    p = _abi.gs_params(n=10)  # null pointers with n > 0
    proj = _abi.gs_proj(n=10)
    assert lib.gs_preprocess(C.byref(p), C.byref(cam), C.byref(opt), C.byref(proj), None) == _abi.GS_ERR_ARG
    assert b"NULL" in lib.gs_last_error_message()
    assert lib.gs_preprocess(C.byref(p), None, C.byref(opt), C.byref(proj), None) == _abi.GS_ERR_ARG
    bad = api.make_options(7)
    assert lib.gs_preprocess(C.byref(p), C.byref(cam), C.byref(bad), C.byref(proj), None) == _abi.GS_ERR_ARG
    assert b"sh_degree" in lib.gs_last_error_message()
    neg = _abi.gs_params(n=-1)
    assert lib.gs_preprocess(C.byref(neg), C.byref(cam), C.byref(opt), C.byref(proj), None) == _abi.GS_ERR_ARG
    big = _cam(w=100000)
    assert lib.gs_preprocess(C.byref(p), C.byref(big), C.byref(opt), C.byref(proj), None) == _abi.GS_ERR_ARG
    mode = api.make_options(0, bwd_mode=9)
    assert lib.gs_render_bwd(C.byref(proj), None, None, C.byref(cam), C.byref(mode), None, None, None, None,
                             None) == _abi.GS_ERR_ARG
    d = C.c_int64(0)
    assert lib.gs_bin_and_sort(C.byref(proj), C.byref(cam), C.byref(opt), None, 0, None, None, -5, C.byref(d),
                               None, None) == _abi.GS_ERR_ARG
    misaligned = _abi.gs_proj(rec=8, depth=16, radius=16, tiles_touched=16, n=10)
    assert lib.gs_render_fwd(C.byref(misaligned), 16, 16, C.byref(cam), C.byref(opt), 16, 16, 16,
                             None) == _abi.GS_ERR_ARG
    assert b"16-byte" in lib.gs_last_error_message()


def test_new_entry_points_reject_bad_arguments_on_the_host(lib):
    cam, opt = _cam(), api.make_options(0)
    # aligned placeholder addresses: every call below fails on the host before any device work
    proj = _abi.gs_proj(rec=256, depth=256, radius=256, tiles_touched=256, n=10)
    # the sort without host synchronisation: capacity, ranges, image size
    assert lib.gs_bin_and_sort_async(C.byref(proj), C.byref(cam), C.byref(opt), None, 0, None, None, -1, None, None,
                                     None) == _abi.GS_ERR_ARG
    assert lib.gs_bin_and_sort_async(C.byref(proj), C.byref(cam), C.byref(opt), None, 0, None, None, 100, None, None,
                                     None) == _abi.GS_ERR_ARG
    assert b"tile_ranges" in lib.gs_last_error_message()
    huge = _cam(w=4096, h=4096)  # 65,536 tiles: beyond the counting pass
    assert lib.gs_bin_and_sort_async(C.byref(proj), C.byref(huge), C.byref(opt), None, 0, None, 256, 100, None, 256,
                                     None) == _abi.GS_ERR_ARG
    assert b"49152" in lib.gs_last_error_message()
    # the preprocess backward with statistics: the statistics block is required
    p = _abi.gs_params(n=0)
    empty = _abi.gs_proj(n=0)
    assert lib.gs_preprocess_bwd_stats(C.byref(p), C.byref(cam), C.byref(opt), C.byref(empty), None, None, None, None,
                                       None, None, 0, None, None) == _abi.GS_ERR_ARG
    assert b"stats" in lib.gs_last_error_message()
    # the surfel backward has no shared-memory mode
    sm = api.make_options(0, bwd_mode="sm")
    assert lib.gs_render2d_bwd(None, 0, None, None, C.byref(cam), C.byref(sm), None, None, None, None,
                               None) == _abi.GS_ERR_ARG
    assert b"GS_BWD_SM" in lib.gs_last_error_message()


def test_host_step_entry_points_reject_bad_arguments_on_the_host(lib):
    """The end-to-end pair checks its arguments before any CUDA call."""
    h = C.c_void_p()
    assert lib.gs_step_context_create(10, 3, 64, 64, 100, None) == _abi.GS_ERR_ARG
    assert lib.gs_step_context_create(-1, 3, 64, 64, 100, C.byref(h)) == _abi.GS_ERR_ARG
    assert lib.gs_step_context_create(10, 4, 64, 64, 100, C.byref(h)) == _abi.GS_ERR_ARG
    assert b"sh_degree" in lib.gs_last_error_message()
    assert lib.gs_step_context_create(10, 3, 0, 64, 100, C.byref(h)) == _abi.GS_ERR_ARG
    assert lib.gs_step_context_create(10, 3, 4096, 4096, 100, C.byref(h)) == _abi.GS_ERR_ARG
    assert b"49152" in lib.gs_last_error_message()
    assert lib.gs_step_context_create(10, 3, 64, 64, -5, C.byref(h)) == _abi.GS_ERR_ARG
    assert h.value is None  # not set on failure
    assert lib.gs_step_context_destroy(None) == _abi.GS_OK
    cam, opt = _cam(), api.make_options(3)
    p, g = _abi.gs_params(n=10), _abi.gs_tensors(n=10)
    assert lib.gs_train_step_host(None, C.byref(p), 256, C.byref(cam), C.byref(opt), C.byref(g), None, None,
                                  None) == _abi.GS_ERR_ARG
    assert b"NULL" in lib.gs_last_error_message()


def test_product_path_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_abi, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_abi, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _abi.load()
