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
