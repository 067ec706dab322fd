"""The end-to-end entry point gs_train_step_host (host buffers in and out, the whole step of one view
on the device) against the same step through the device-pointer calls (step.train_step_async),
which the parity tests check against the oracle: D bit for bit; the gradients up to the order of
the float atomics (1e-3 of each tensor's largest magnitude, the bar of the graph-replay tests) and
the loss to float32 rounding (their summation orders vary from run to run). Also two contexts on
two streams in turn (the pipelined use), the capacity overflow, and argument checks that need a
context."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from differentiable_gaussian_splatting_gs_gb300 import _abi, api, step  # noqa: E402

from _cases import PARAM_NAMES, scene  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _device_step(s, view, opt, capacity):
    params = {k: torch.from_numpy(np.ascontiguousarray(getattr(s, k))).to(DEV) for k in PARAM_NAMES}
    grads = api.alloc_param_grads(params)
    bufs = step.StepBuffers(s.n, DEV)
    n_dup = torch.zeros(1, dtype=torch.int64, device=DEV)
    losses = torch.zeros(1, device=DEV)
    target = torch.from_numpy(s.targets[view]).to(DEV)
    step.train_step_async(params, [s.cameras[view]], [target], opt, grads, bufs, capacity, n_dup, losses=losses)
    torch.cuda.synchronize()
    return {k: v.cpu() for k, v in grads.items()}, float(losses[0]), int(n_dup[0])


def _host_inputs(s, view):
    hp = {k: torch.from_numpy(np.ascontiguousarray(getattr(s, k))).pin_memory() for k in PARAM_NAMES}
    ht = torch.from_numpy(np.ascontiguousarray(s.targets[view])).pin_memory()
    return hp, ht


def _close(got, want):
    return float((got - want).abs().max()) <= 1e-3 * max(float(want.abs().max()), 1e-30)


def _host_outputs(hp):
    hg = {k: torch.full_like(v, float("nan")).pin_memory() for k, v in hp.items()}
    return hg, torch.zeros(1).pin_memory(), torch.zeros(1, dtype=torch.int64).pin_memory()


@pytest.mark.parametrize("name", ["object", "outdoor", "contention"])
def test_host_step_equals_the_device_step(name):
    s, view = scene(name)
    cam = s.cameras[view]
    opt = api.make_options(s.sh_degree)
    capacity = 4 << 20
    want, want_loss, want_d = _device_step(s, view, opt, capacity)
    hp, ht = _host_inputs(s, view)
    hg, hl, hd = _host_outputs(hp)
    ctx = api.StepContext(s.n, s.sh_degree, cam.width, cam.height, capacity)
    api.gs_train_step_host(ctx, hp, ht, cam, opt, hg, hl, hd)
    torch.cuda.synchronize()
    assert api.gs_device_error() == _abi.GS_OK
    assert int(hd[0]) == want_d > 0
    for k in PARAM_NAMES:
        assert _close(hg[k], want[k]), k
    assert abs(float(hl[0]) - want_loss) <= 1e-5 * abs(want_loss)
    ctx.close()


def test_two_contexts_on_two_streams_in_turn():
    """The pipelined use: steps alternate between two contexts and two streams, each with its own
    host buffers, so that one step's copies can overlap the other's compute; every step's outputs
    equal the device step's."""
    s, view = scene("outdoor")
    cam = s.cameras[view]
    opt = api.make_options(s.sh_degree)
    capacity = 4 << 20
    want, _, want_d = _device_step(s, view, opt, capacity)
    streams = [torch.cuda.Stream(DEV), torch.cuda.Stream(DEV)]
    ctxs = [api.StepContext(s.n, s.sh_degree, cam.width, cam.height, capacity) for _ in range(2)]
    ins = [_host_inputs(s, view) for _ in range(2)]
    outs = [[_host_outputs(ins[b][0]) for b in range(2)] for _ in range(2)]
    for k in range(4):
        b = k % 2
        hp, ht = ins[b]
        hg, hl, hd = outs[k // 2][b]
        api.gs_train_step_host(ctxs[b], hp, ht, cam, opt, hg, hl, hd, stream=streams[b])
    torch.cuda.synchronize()
    assert api.gs_device_error() == _abi.GS_OK
    for r in range(2):
        for b in range(2):
            hg, _, hd = outs[r][b]
            assert int(hd[0]) == want_d
            for name in PARAM_NAMES:
                assert _close(hg[name], want[name]), name
    for c in ctxs:
        c.close()


def test_host_step_capacity_overflow_and_argument_checks():
    s, view = scene("object")
    cam = s.cameras[view]
    opt = api.make_options(s.sh_degree)
    hp, ht = _host_inputs(s, view)
    hg, hl, hd = _host_outputs(hp)
    ctx = api.StepContext(s.n, s.sh_degree, cam.width, cam.height, 1000)
    api.gs_train_step_host(ctx, hp, ht, cam, opt, hg, hl, hd)
    torch.cuda.synchronize()
    # the duplicates past the capacity are dropped, the check bit set, and D reported
    assert api.gs_device_error() == _abi.GS_ERR_DEVICE_CHECK
    assert int(hd[0]) > 1000
    with pytest.raises(_abi.GsError) as ei:  # another SH degree than the context's
        api.gs_train_step_host(ctx, hp, ht, cam, api.make_options(0), hg, hl, hd)
    assert ei.value.status == _abi.GS_ERR_ARG
    small = api.StepContext(s.n, s.sh_degree, cam.width // 2, cam.height, 1000)
    with pytest.raises(_abi.GsError) as ei:  # an image larger than the context's
        api.gs_train_step_host(small, hp, ht, cam, opt, hg, hl, hd)
    assert ei.value.status == _abi.GS_ERR_ARG
    ctx.close()
    small.close()
    assert api.gs_device_error() == _abi.GS_OK
