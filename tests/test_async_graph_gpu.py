"""The sort that does not synchronise (gs_bin_and_sort_async) and the training step captured into a
CUDA graph, against the synchronising entry points.

Bars: the sorted lists, tile ranges and duplicate counts are bit-exact; gradients from a graph
replay equal an eager step's up to the order of the float atomics
(1e-3 of each tensor's largest magnitude: the log-scale gradient cancels, and over three views the
run-to-run spread of the atomics' summation order has reached 1e-4 of its largest magnitude); a
capacity overflow leaves every tile range empty and reports a device check error.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import gs_scenes  # noqa: E402
import oracle  # noqa: E402
from differentiable_gaussian_splatting_gs_gb300 import _abi, api, step  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
NAMES = ("mean3d", "log_scale", "quat", "opacity_logit", "sh")


def _params(s):
    return {k: torch.from_numpy(np.ascontiguousarray(getattr(s, k))).to(DEV) for k in NAMES}


def _proj(s, cam):
    pre = oracle.preprocess(s.mean3d, s.log_scale, s.quat, s.opacity_logit, s.sh, s.sh_degree, cam)
    return api.proj_from_arrays(pre["mean2d"], pre["conic"], pre["opacity"], pre["rgb"], pre["depth"],
                                pre["radius"], DEV)


@pytest.mark.parametrize("cfg,n,res", [(0, None, 1.0), (1, 20_000, 1.0), (2, 100_000, 0.5), (4, 3_000, 0.25)])
@pytest.mark.parametrize("static", [False, True])
def test_async_sort_matches_synchronising_sort(cfg, n, res, static):
    s = gs_scenes.make_scene(cfg, n=n, res_scale=res)
    cam = s.cameras[0]
    opt = api.make_options(s.sh_degree)
    proj = _proj(s, cam)
    ref = api.gs_bin_and_sort(proj, cam, opt)
    D = ref.n_dup
    cap = D + 777  # ragged spare capacity
    b = api.gs_bin_and_sort_async(proj, cam, opt, cap, want_keys=True, static_workspace=static)
    torch.cuda.synchronize()
    assert int(b.n_dup.item()) == D
    assert torch.equal(b.vals[:D], ref.vals) and torch.equal(b.keys[:D], ref.keys)
    assert torch.equal(b.ranges, ref.ranges)
    assert api.gs_device_error() == _abi.GS_OK


def test_async_sort_exact_capacity_and_overflow():
    s = gs_scenes.make_scene(1, n=20_000)
    cam = s.cameras[0]
    opt = api.make_options(s.sh_degree)
    proj = _proj(s, cam)
    ref = api.gs_bin_and_sort(proj, cam, opt)
    D = ref.n_dup
    b = api.gs_bin_and_sort_async(proj, cam, opt, D)  # exactly enough
    torch.cuda.synchronize()
    assert torch.equal(b.vals[:D], ref.vals) and torch.equal(b.ranges, ref.ranges)
    assert api.gs_device_error() == _abi.GS_OK
    # one entry short: nothing is written past the capacity, all ranges are empty, D is reported
    buf = api.SortBuffers(DEV)
    buf.ensure(proj.n, D - 1, cam.width, cam.height, False)
    buf.vals = torch.full((D,), -7, dtype=torch.int32, device=DEV)  # one guard entry past the capacity
    b = api.gs_bin_and_sort_async(proj, cam, opt, D - 1, buffers=buf)
    torch.cuda.synchronize()
    assert int(b.n_dup.item()) == D
    assert int(b.ranges.abs().max()) == 0
    assert int(buf.vals[D - 1]) == -7
    assert api.gs_device_error() == _abi.GS_ERR_DEVICE_CHECK
    assert api.gs_device_error() == _abi.GS_OK  # reading clears it


def test_async_sort_empty_and_all_culled():
    s = gs_scenes.make_scene(0, n=300)
    cam = s.cameras[0]
    opt = api.make_options(0)
    s.mean3d[:, 2] = -1.0
    proj = api.gs_preprocess(_params(s), cam, opt)
    b = api.gs_bin_and_sort_async(proj, cam, opt, 1024)
    torch.cuda.synchronize()
    assert int(b.n_dup.item()) == 0 and int(b.ranges.abs().max()) == 0
    empty = {k: v[:0] for k, v in _params(s).items()}
    proj = api.gs_preprocess(empty, cam, opt)
    b = api.gs_bin_and_sort_async(proj, cam, opt, 0)
    torch.cuda.synchronize()
    assert int(b.n_dup.item()) == 0 and int(b.ranges.abs().max()) == 0
    assert api.gs_device_error() == _abi.GS_OK


def test_async_sort_rejects_images_beyond_the_counting_pass():
    s = gs_scenes.make_scene(0, n=100)
    cam = s.cameras[0]
    opt = api.make_options(0)
    proj = api.gs_preprocess(_params(s), cam, opt)
    big = api.make_camera(cam)
    big.width, big.height = 4096, 4096  # 65,536 tiles
    with pytest.raises(api.GsError, match="49152"):
        api.gs_bin_and_sort_async(proj, big, opt, 1024)


@pytest.mark.parametrize("cfg,n,res,views,two", [(1, 20_000, 1.0, None, False), (3, 20_000, 0.25, 3, False),
                                                  (3, 20_000, 0.25, 4, True)])
def test_graphed_step_matches_eager_step(cfg, n, res, views, two):
    """two: the views on two streams with two buffer sets (train_step_async_overlapped), the
    preprocess backwards chained in view order."""
    s = gs_scenes.make_scene(cfg, n=n, res_scale=res, views=views)
    params = _params(s)
    opt = api.make_options(s.sh_degree)
    targets = [torch.from_numpy(t).to(DEV) for t in s.targets[:len(s.cameras)]]
    bufs = step.StepBuffers(s.n, DEV)
    grads_ref = api.alloc_param_grads(params)
    out = step.train_step(params, s.cameras, targets, opt, grads_ref, bufs)
    cap = bufs.sort.capacity
    grads = api.alloc_param_grads(params)
    bufs2 = step.StepBuffers(s.n, DEV) if two else None
    g = step.GraphedStep(params, s.cameras, targets, opt, grads, bufs, cap, buffers2=bufs2)
    for k in NAMES:
        grads[k].fill_(123.0)  # the replay must overwrite them
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert g.n_dup.cpu().tolist() == out["n_dup"]
    assert g.launches > 0
    for k in NAMES:
        a, r = grads[k].cpu().numpy(), grads_ref[k].cpu().numpy()
        assert np.abs(a - r).max() <= 1e-3 * max(np.abs(r).max(), 1e-30), k
    assert api.gs_device_error() == _abi.GS_OK


def test_graphed_step_times_its_raster_kernels():
    """External timing events captured in the graph record at every replay: the forward and
    backward raster times are positive and fit inside the replay's own time."""
    try:
        torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        pytest.skip("this torch has no external events")
    s = gs_scenes.make_scene(1, n=20_000)
    params = _params(s)
    opt = api.make_options(s.sh_degree)
    targets = [torch.from_numpy(s.targets[0]).to(DEV)]
    bufs = step.StepBuffers(s.n, DEV)
    grads = api.alloc_param_grads(params)
    step.train_step(params, s.cameras, targets, opt, grads, bufs)

    def xev():
        return torch.cuda.Event(enable_timing=True, external=True)
    ev = [((xev(), xev()), (xev(), xev()))]
    g = step.GraphedStep(params, s.cameras, targets, opt, grads, bufs, bufs.sort.capacity, events=ev)
    for _ in range(2):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        total = e0.elapsed_time(e1)
        fwd, bwd = ev[0][0][0].elapsed_time(ev[0][0][1]), ev[0][1][0].elapsed_time(ev[0][1][1])
        assert 0 < fwd < total and 0 < bwd < total and fwd + bwd < total
    assert api.gs_device_error() == _abi.GS_OK


def test_graphed_surfel_step_matches_eager_surfel_step():
    s = gs_scenes.make_scene(1, n=20_000)
    params = _params(s)
    opt = api.make_options(s.sh_degree)
    targets = [torch.from_numpy(s.targets[0]).to(DEV)]
    bufs = step.StepBuffers(s.n, DEV)
    cap = api.gs_bin_and_sort(api.gs_preprocess2d(params, s.cameras[0], opt, out=bufs.proj)[0], s.cameras[0], opt,
                              buffers=bufs.sort).n_dup + 1000
    n_dup = torch.zeros(1, dtype=torch.int64, device=DEV)
    grads_ref = api.alloc_param_grads(params)
    step.train_step_surfels_async(params, s.cameras, targets, opt, grads_ref, bufs, cap, n_dup)
    torch.cuda.synchronize()
    grads = api.alloc_param_grads(params)
    g = step.GraphedStep(params, s.cameras, targets, opt, grads, bufs, cap, surfels=True)
    for k in NAMES:
        grads[k].fill_(123.0)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert g.n_dup.cpu().tolist() == n_dup.cpu().tolist()
    for k in NAMES:
        a, r = grads[k].cpu().numpy(), grads_ref[k].cpu().numpy()
        assert np.abs(a - r).max() <= 1e-3 * max(np.abs(r).max(), 1e-30), k
    assert api.gs_device_error() == _abi.GS_OK


def test_back_to_back_views_without_synchronisation():
    """Three views' preprocess and sort enqueued back to back on one stream with no synchronisation
    in between, each into its own buffers (the kernels of consecutive calls may overlap through
    programmatic dependent launch), against the synchronising sort of each view run alone."""
    s = gs_scenes.make_scene(3, n=20_000, res_scale=0.25, views=3)
    params = _params(s)
    opt = api.make_options(s.sh_degree)
    refs = []
    for cam in s.cameras:
        refs.append(api.gs_bin_and_sort(api.gs_preprocess(params, cam, opt), cam, opt))
    projs, bufs, ranges, ndup = [], [], [], []
    for cam, r in zip(s.cameras, refs):
        projs.append(api.alloc_proj(s.n, DEV))
        b = api.SortBuffers(DEV)
        b.ensure(s.n, r.n_dup + 100, cam.width, cam.height, False)
        bufs.append(b)
        ranges.append(torch.empty((((cam.width + 15) // 16) * ((cam.height + 15) // 16), 2), dtype=torch.int32,
                                  device=DEV))
        ndup.append(torch.zeros(1, dtype=torch.int64, device=DEV))
    torch.cuda.synchronize()
    outs = []
    for v, cam in enumerate(s.cameras):
        proj = api.gs_preprocess(params, cam, opt, out=projs[v])
        outs.append(api.gs_bin_and_sort_async(proj, cam, opt, refs[v].n_dup + 100, buffers=bufs[v],
                                              ranges=ranges[v], n_dup=ndup[v]))
    torch.cuda.synchronize()
    for r, o in zip(refs, outs):
        D = r.n_dup
        assert int(o.n_dup.item()) == D
        assert torch.equal(o.vals[:D], r.vals) and torch.equal(o.ranges, r.ranges)
    assert api.gs_device_error() == _abi.GS_OK
