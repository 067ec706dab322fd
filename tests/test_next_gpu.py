"""GPU parity of the NEXT-stage kernels against the float64 oracle: sparse Adam (gs_adam_step).

Tolerance of the Adam step, from its float32 arithmetic: m and v are one fused multiply-add of
float32 inputs (relative error below 1e-6 of the terms); the parameter step lr m^ / (sqrt(v^) + eps)
is a chain of a few correctly rounded operations (relative error below 1e-5 of the step); the new
parameter is then rounded to float32 (half an ulp of it).
"""
import numpy as np
import pytest
import torch

import gs_scenes
from oracle import optim

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from differentiable_gaussian_splatting_gs_gb300 import _abi, api  # noqa: E402

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")
F32_B1, F32_B2, F32_EPS = (float(np.float32(x)) for x in (0.9, 0.999, 1e-15))


def _dev(d):
    return {k: torch.from_numpy(np.ascontiguousarray(a)).to(DEV) for k, a in d.items()}


def _check_adam(st, p64, m64, v64, P, M, V, step_params):
    for name in optim.NAMES:
        g = st["grads"][name].astype(np.float64)
        p0 = step_params[name].astype(np.float64)
        m_old = st["exp_avg_prev"][name].astype(np.float64)
        v_old = st["exp_avg_sq_prev"][name].astype(np.float64)
        pg, mg, vg = (T[name].cpu().numpy().astype(np.float64) for T in (P, M, V))
        tol_m = 1e-6 * (F32_B1 * np.abs(m_old) + (1 - F32_B1) * np.abs(g)) + 1e-30
        tol_v = 1e-6 * (F32_B2 * v_old + (1 - F32_B2) * g * g) + 1e-30
        tol_p = 2.0 ** -24 * np.abs(p64[name]) + 1e-5 * np.abs(p64[name] - p0) + 1e-30
        assert np.all(np.abs(mg - m64[name]) <= tol_m), name
        assert np.all(np.abs(vg - v64[name]) <= tol_v), name
        assert np.all(np.abs(pg - p64[name]) <= tol_p), (name, np.max(np.abs(pg - p64[name]) - tol_p))


@pytest.mark.parametrize("n,deg", [(20_001, 3), (4097, 1), (3, 0), (1, 2)])
def test_sparse_adam_matches_oracle_two_steps_in_a_row(n, deg):
    st = gs_scenes.make_adam_state(n, deg, seed=n % 97)
    lr = gs_scenes.ADAM_LR
    P, G, M, V = _dev(st["params"]), _dev(st["grads"]), _dev(st["exp_avg"]), _dev(st["exp_avg_sq"])
    radius = torch.from_numpy(np.where(st["visible"], 3, 0).astype(np.int32)).to(DEV)
    p, m, v = st["params"], st["exp_avg"], st["exp_avg_sq"]
    for t in (6, 7):
        step_params = {k: P[k].cpu().numpy() for k in P}
        st["exp_avg_prev"] = {k: M[k].cpu().numpy() for k in M}
        st["exp_avg_sq_prev"] = {k: V[k].cpu().numpy() for k in V}
        # the oracle steps from the GPU's float32 state, so each step is compared on its own
        # the kernel receives beta1, beta2 and eps as float32 values: the oracle uses the same values
        p, m, v = optim.adam_step_sparse(step_params, st["grads"], st["exp_avg_prev"], st["exp_avg_sq_prev"],
                                         st["visible"], lr, t, beta1=F32_B1, beta2=F32_B2, eps=F32_EPS)
        api.gs_adam_step(P, G, M, V, radius, api.make_adam_options(lr, t, deg))
        torch.cuda.synchronize()
        _check_adam(st, p, m, v, P, M, V, step_params)
        hid = ~st["visible"]
        for name in optim.NAMES:  # hidden Gaussians: bit-identical
            assert np.array_equal(P[name].cpu().numpy()[hid], step_params[name][hid])
    assert api.gs_device_error() == 0


def test_sparse_adam_all_hidden_and_empty():
    st = gs_scenes.make_adam_state(1000, 3, seed=1, visible_frac=0.0)
    P, G, M, V = _dev(st["params"]), _dev(st["grads"]), _dev(st["exp_avg"]), _dev(st["exp_avg_sq"])
    radius = torch.zeros(1000, dtype=torch.int32, device=DEV)
    before = {k: P[k].clone() for k in P}
    api.gs_adam_step(P, G, M, V, radius, api.make_adam_options(gs_scenes.ADAM_LR, 3, 3))
    torch.cuda.synchronize()
    assert all(torch.equal(P[k], before[k]) for k in P)
    e = {k: torch.empty((0,) + tuple(P[k].shape[1:]), device=DEV) for k in P}
    api.gs_adam_step(e, e, e, e, torch.empty(0, dtype=torch.int32, device=DEV),
                     api.make_adam_options(gs_scenes.ADAM_LR, 1, 3))


def test_sparse_adam_rejects_bad_arguments():
    st = gs_scenes.make_adam_state(16, 0, seed=2)
    P, G, M, V = _dev(st["params"]), _dev(st["grads"]), _dev(st["exp_avg"]), _dev(st["exp_avg_sq"])
    radius = torch.ones(16, dtype=torch.int32, device=DEV)
    with pytest.raises(_abi.GsError):
        api.gs_adam_step(P, G, M, V, radius, api.make_adam_options(gs_scenes.ADAM_LR, 0, 0))
    with pytest.raises(_abi.GsError):
        api.gs_adam_step(P, G, M, V, radius, api.make_adam_options(gs_scenes.ADAM_LR, 1, 0, beta1=1.5))


@pytest.mark.parametrize("n,deg,ndc", [(20_003, 3, False), (777, 0, True), (5, 1, False)])
def test_densify_stats_match_oracle(n, deg, ndc):
    st = gs_scenes.make_adam_state(n, deg, seed=n % 89)
    rng = np.random.default_rng(n)
    radius = np.where(st["visible"], rng.integers(1, 60, n), 0).astype(np.int32)
    g2 = np.zeros((n, 12), dtype=np.float32)
    g2[:, :9] = (rng.normal(0, 1, (n, 9)) * 10.0 ** rng.uniform(-7, -2, (n, 9))).astype(np.float32)
    acc0 = rng.uniform(0, 1e-3, n).astype(np.float32)
    cnt0 = rng.integers(0, 5, n).astype(np.int32)
    mr0 = rng.integers(0, 40, n).astype(np.int32)
    proj = api.alloc_proj(n, DEV)
    proj.radius.copy_(torch.from_numpy(radius))
    acc, cnt, mr = (torch.from_numpy(a.copy()).to(DEV) for a in (acc0, cnt0, mr0))
    mag = torch.full((n,), -1.0, device=DEV)
    G = _dev(st["grads"])
    api.gs_densify_stats(proj, torch.from_numpy(g2).to(DEV), 1297, 840, acc, cnt, mr, ndc=ndc, param_grads=G,
                         grad_mag=mag, sh_degree=deg)
    torch.cuda.synchronize()
    ra, rc, rm, rmag = optim.densify_stats(radius, g2, 1297, 840, ndc, acc0, cnt0, mr0, st["grads"])
    # float32: the norm of two products within 4 ulps, then one rounded addition
    tol = 4 * 2.0 ** -24 * (ra - acc0.astype(np.float64)) + 2.0 ** -24 * np.abs(ra) + 1e-38
    assert np.all(np.abs(acc.cpu().numpy() - ra) <= tol)
    assert np.array_equal(cnt.cpu().numpy(), rc) and np.array_equal(mr.cpu().numpy(), rm)
    # a sum of 11 + 3K squares in float32: relative error below 1e-5
    assert np.allclose(mag.cpu().numpy(), rmag, rtol=1e-5, atol=1e-38)


from oracle import loss as oloss  # noqa: E402


def _render_like(rng, h, w):
    yy, xx = np.mgrid[0:h, 0:w]
    base = 0.5 + 0.3 * np.sin(xx / 11.0)[None] * np.cos(yy / 7.0)[None] * np.array([1.0, 0.7, 0.4])[:, None, None]
    return np.clip(base + 0.02 * rng.normal(size=(3, h, w)), 0, 1).astype(np.float32)


@pytest.mark.parametrize("h,w,lam", [(37, 70, 0.2), (16, 32, 1.0), (5, 3, 0.2), (840, 1297, 0.2)])
def test_l1_dssim_loss_matches_oracle(h, w, lam):
    rng = np.random.default_rng(h * w)
    x = _render_like(rng, h, w)
    y = rng.uniform(0, 1, (3, h, w)).astype(np.float32)
    y[:, : h // 3] = np.clip(x[:, : h // 3] + 0.01 * rng.normal(size=(3, h // 3, w)), 0, 1)  # a close part too
    loss, dl = api.gs_loss_l1_dssim(torch.from_numpy(x).to(DEV), torch.from_numpy(y).to(DEV), lam)
    torch.cuda.synchronize()
    rl, rg = oloss.loss_l1_dssim(x, y, lam)
    assert abs(loss.item() - rl) <= 1e-5 * abs(rl)
    g = dl.cpu().numpy()
    assert np.abs(g - rg).max() <= 1e-4 * np.abs(rg).max()


def test_l1_dssim_of_an_image_with_itself():
    rng = np.random.default_rng(3)
    x = torch.from_numpy(_render_like(rng, 48, 64)).to(DEV)
    loss, dl = api.gs_loss_l1_dssim(x, x.clone(), 0.2)
    torch.cuda.synchronize()
    assert abs(loss.item()) < 1e-6 and dl.abs().max().item() < 1e-4 / x.numel()


def _step_grad2d(s, view, params, opt):
    from differentiable_gaussian_splatting_gs_gb300 import step
    cam = s.cameras[view]
    bufs = step.StepBuffers(s.n, DEV)
    proj = api.gs_preprocess(params, cam, opt, out=bufs.proj)
    b = api.gs_bin_and_sort(proj, cam, opt, buffers=bufs.sort)
    img, tf, nc = api.gs_render_fwd(proj, b.vals, b.ranges, cam, opt)
    dl = img - torch.from_numpy(s.targets[view]).to(DEV)
    return cam, proj, api.gs_render_bwd(proj, b.vals, b.ranges, cam, opt, dl, tf, nc), bufs


@pytest.mark.parametrize("cfg,n,ndc", [(0, None, False), (1, 20_000, True), (1, 20_000, False)])
def test_fused_statistics_equal_the_separate_call(cfg, n, ndc):
    """gs_preprocess_bwd_stats = gs_preprocess_bwd followed by gs_densify_stats, bit for bit."""
    s = gs_scenes.make_scene(cfg, n=n)
    params = {k: torch.from_numpy(np.ascontiguousarray(getattr(s, k))).to(DEV) for k in optim.NAMES}
    opt = api.make_options(s.sh_degree)
    cam, proj, g2, bufs = _step_grad2d(s, 0, params, opt)
    rng = np.random.default_rng(7)
    acc0 = torch.from_numpy(rng.uniform(0, 1e-3, s.n).astype(np.float32)).to(DEV)
    cnt0 = torch.from_numpy(rng.integers(0, 5, s.n).astype(np.int32)).to(DEV)
    mr0 = torch.from_numpy(rng.integers(0, 40, s.n).astype(np.int32)).to(DEV)
    a = [t.clone() for t in (acc0, cnt0, mr0)] + [torch.full((s.n,), -1.0, device=DEV)]
    b = [t.clone() for t in (acc0, cnt0, mr0)] + [torch.full((s.n,), -1.0, device=DEV)]
    ga = api.gs_preprocess_bwd(params, cam, opt, proj, g2)
    api.gs_densify_stats(proj, g2, cam.width, cam.height, a[0], a[1], a[2], ndc=ndc, param_grads=ga, grad_mag=a[3],
                         sh_degree=s.sh_degree)
    gb = api.gs_preprocess_bwd_stats(params, cam, opt, proj, g2, b[0], b[1], b[2], grad_mag=b[3], ndc=ndc)
    torch.cuda.synchronize()
    for k in optim.NAMES:
        assert torch.equal(ga[k], gb[k]), k
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert int((a[1] != cnt0).sum()) == int((proj.radius > 0).sum())
    assert api.gs_device_error() == 0


def test_fused_statistics_over_two_views():
    """Accumulating views: the counters add up as two separate calls would, and grad_mag is the
    norm of the second view's own gradients."""
    s = gs_scenes.make_scene(3, n=20_000, res_scale=0.25, views=2)
    params = {k: torch.from_numpy(np.ascontiguousarray(getattr(s, k))).to(DEV) for k in optim.NAMES}
    opt = api.make_options(s.sh_degree)
    z = lambda dt: torch.zeros(s.n, dtype=dt, device=DEV)  # noqa: E731
    acc_f, cnt_f, mr_f, mag_f = z(torch.float32), z(torch.int32), z(torch.int32), z(torch.float32)
    acc_s, cnt_s, mr_s, mag_s = z(torch.float32), z(torch.int32), z(torch.int32), z(torch.float32)
    grads = None
    for v in range(2):
        cam, proj, g2, bufs = _step_grad2d(s, v, params, opt)
        grads = api.gs_preprocess_bwd_stats(params, cam, opt, proj, g2, acc_f, cnt_f, mr_f, grad_mag=mag_f,
                                            out=grads, accumulate=v > 0)
        own = api.gs_preprocess_bwd(params, cam, opt, proj, g2)  # this view alone
        api.gs_densify_stats(proj, g2, cam.width, cam.height, acc_s, cnt_s, mr_s, param_grads=own, grad_mag=mag_s,
                             sh_degree=s.sh_degree)
    torch.cuda.synchronize()
    assert torch.equal(acc_f, acc_s) and torch.equal(cnt_f, cnt_s) and torch.equal(mr_f, mr_s)
    assert torch.equal(mag_f, mag_s)
    assert int(cnt_f.max()) <= 2 and api.gs_device_error() == 0
