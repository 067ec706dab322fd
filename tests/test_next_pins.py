"""Pins of the oracle's NEXT-stage functions (run on the CPU).

Sparse Adam (oracle/optim.py) is checked against torch.optim.Adam, an independent implementation
of the same update, on the visible rows; against the closed form of Adam's first step; and for the
rows it must leave alone.
"""
import numpy as np
import pytest
import torch

import gs_scenes
from oracle import optim


def _torch_adam(state, lr, steps, beta1=0.9, beta2=0.999, eps=1e-15):
    """torch.optim.Adam in float64 over the visible rows, one parameter group per learning rate."""
    vis = state["visible"]
    ts = {}
    groups = []
    for name in optim.NAMES:
        p = torch.tensor(state["params"][name][vis], dtype=torch.float64)
        if name == "sh":
            dc = p[:, :1].clone().requires_grad_(True)
            rest = p[:, 1:].clone().requires_grad_(True)
            ts["sh_dc"], ts["sh_rest"] = dc, rest
            groups += [{"params": [dc], "lr": lr["sh_dc"]}, {"params": [rest], "lr": lr["sh_rest"]}]
        else:
            t = p.clone().requires_grad_(True)
            ts[name] = t
            groups.append({"params": [t], "lr": lr["opacity" if name == "opacity_logit" else name]})
    opt = torch.optim.Adam(groups, betas=(beta1, beta2), eps=eps)
    # seed the moments: torch keeps exp_avg / exp_avg_sq per parameter and a step count
    for name, t in ts.items():
        src = "sh" if name.startswith("sh") else name
        m = torch.tensor(state["exp_avg"][src][vis], dtype=torch.float64)
        v = torch.tensor(state["exp_avg_sq"][src][vis], dtype=torch.float64)
        if name == "sh_dc":
            m, v = m[:, :1], v[:, :1]
        elif name == "sh_rest":
            m, v = m[:, 1:], v[:, 1:]
        opt.state[t] = {"step": torch.tensor(float(steps[0] - 1)), "exp_avg": m.clone(), "exp_avg_sq": v.clone()}
    for _ in steps:
        for name, t in ts.items():
            src = "sh" if name.startswith("sh") else name
            g = torch.tensor(state["grads"][src][vis], dtype=torch.float64)
            g = g[:, :1] if name == "sh_dc" else (g[:, 1:] if name == "sh_rest" else g)
            t.grad = g.clone()
        opt.step()
    out = {n: ts[n].detach().numpy() for n in ts if not n.startswith("sh")}
    out["sh"] = np.concatenate([ts["sh_dc"].detach().numpy(), ts["sh_rest"].detach().numpy()], axis=1)
    return out


@pytest.mark.parametrize("deg,first_step,nsteps", [(3, 1, 1), (3, 4, 3), (0, 1, 2)])
def test_sparse_adam_matches_torch_adam_on_visible_rows(deg, first_step, nsteps):
    st = gs_scenes.make_adam_state(300, deg, seed=deg + first_step)
    lr = gs_scenes.ADAM_LR
    p, m, v = st["params"], st["exp_avg"], st["exp_avg_sq"]
    for t in range(first_step, first_step + nsteps):
        p, m, v = optim.adam_step_sparse(p, st["grads"], m, v, st["visible"], lr, t)
    ref = _torch_adam(st, lr, list(range(first_step, first_step + nsteps)))
    vis = st["visible"]
    for name in optim.NAMES:
        np.testing.assert_allclose(p[name][vis], ref[name], rtol=1e-12, atol=1e-15, err_msg=name)


def test_sparse_adam_first_step_moves_each_visible_element_by_its_learning_rate():
    # t = 1 from zero moments: m^ = g, v^ = g^2, so the step is lr * g / (|g| + eps) = lr * sign(g)
    st = gs_scenes.make_adam_state(200, 3, seed=7)
    zeros = {k: np.zeros_like(a) for k, a in st["params"].items()}
    lr = gs_scenes.ADAM_LR
    p, m, v = optim.adam_step_sparse(st["params"], st["grads"], zeros, zeros, st["visible"], lr, 1, eps=1e-300)
    vis = st["visible"]
    for name in optim.NAMES:
        g = st["grads"][name][vis].astype(np.float64)
        step = st["params"][name][vis].astype(np.float64) - p[name][vis]
        lr_arr = optim._lr_array(name, st["params"][name].shape, lr)
        # the step is read back as a difference of O(1) numbers: float64 rounding of about 1e-16
        np.testing.assert_allclose(step, lr_arr * np.sign(g), rtol=1e-12, atol=1e-15, err_msg=name)
        np.testing.assert_allclose(m[name][vis], 0.1 * g, rtol=1e-12, err_msg=name)
        np.testing.assert_allclose(v[name][vis], 0.001 * g * g, rtol=1e-12, err_msg=name)


def test_sparse_adam_leaves_hidden_gaussians_alone():
    st = gs_scenes.make_adam_state(500, 2, seed=3)
    # give hidden rows non-zero gradients: they must still be ignored
    grads = {k: np.where(st["visible"].reshape((-1,) + (1,) * (a.ndim - 1)), a, 1.0).astype(np.float32)
             for k, a in st["grads"].items()}
    p, m, v = optim.adam_step_sparse(st["params"], grads, st["exp_avg"], st["exp_avg_sq"], st["visible"],
                                     gs_scenes.ADAM_LR, 5)
    hid = ~st["visible"]
    for name in optim.NAMES:
        assert np.array_equal(p[name][hid], st["params"][name][hid].astype(np.float64))
        assert np.array_equal(m[name][hid], st["exp_avg"][name][hid].astype(np.float64))
        assert np.array_equal(v[name][hid], st["exp_avg_sq"][name][hid].astype(np.float64))


def test_densify_stats_closed_forms():
    # 3-4-5 gradients, an NDC scale, hidden rows left alone, the max radius
    radius = np.array([2, 0, 5, 7])
    g2 = np.zeros((4, 12))
    g2[:, 0], g2[:, 1] = [3.0, 1.0, 0.5, 0.0], [4.0, 1.0, 1.2, -2.0]
    acc0, cnt0, mr0 = np.array([1.0, 1.0, 0.0, 0.0]), np.array([1, 3, 0, 2]), np.array([4, 9, 1, 9])
    acc, cnt, mr, mag = optim.densify_stats(radius, g2, 640, 480, False, acc0, cnt0, mr0)
    assert np.allclose(acc, [6.0, 1.0, 1.3, 2.0]) and mag is None
    assert list(cnt) == [2, 3, 1, 3] and list(mr) == [4, 9, 5, 9]
    acc, _, _, _ = optim.densify_stats(radius, g2, 640, 480, True, np.zeros(4), cnt0, mr0)
    assert np.isclose(acc[0], np.hypot(3.0 * 320, 4.0 * 240))


def test_densify_gradient_magnitude_is_the_norm_of_the_concatenated_gradients():
    st = gs_scenes.make_adam_state(50, 3, seed=11)
    radius = np.where(st["visible"], 4, 0)
    g2 = np.zeros((50, 12))
    *_, mag = optim.densify_stats(radius, g2, 8, 8, False, np.zeros(50), np.zeros(50), np.zeros(50), st["grads"])
    flat = np.concatenate([st["grads"][k].reshape(50, -1).astype(np.float64) for k in optim.NAMES], axis=1)
    ref = np.linalg.norm(flat, axis=1)  # library routine
    assert np.allclose(mag[st["visible"]], ref[st["visible"]], rtol=1e-13) and np.all(mag[~st["visible"]] == 0)


from oracle import loss as oloss  # noqa: E402


def test_windowed_sum_equals_brute_force_2d_window():
    rng = np.random.default_rng(5)
    a = rng.normal(size=(2, 9, 14))
    w = oloss.window()
    ref = np.zeros_like(a)
    for c in range(2):
        for i in range(9):
            for j in range(14):
                for di in range(-5, 6):
                    for dj in range(-5, 6):
                        if 0 <= i + di < 9 and 0 <= j + dj < 14:
                            ref[c, i, j] += w[di + 5] * w[dj + 5] * a[c, i + di, j + dj]
    assert np.allclose(oloss.windowed(a), ref, rtol=1e-13, atol=1e-15)
    assert np.isclose(w.sum(), 1.0) and np.allclose(w, w[::-1])


def test_ssim_closed_forms_and_identity():
    rng = np.random.default_rng(6)
    x = rng.uniform(0, 1, (3, 20, 24))
    l, g = oloss.loss_l1_dssim(x, x)
    assert abs(l) < 1e-14 and np.abs(g).max() < 1e-14  # SSIM(x, x) = 1 is its maximum
    a, b = np.full((1, 30, 30), 0.3), np.full((1, 30, 30), 0.7)
    S = oloss.ssim_terms(a, b)[-1]
    # away from the zero padding: no variance, S = (2ab + C1) / (a^2 + b^2 + C1)
    assert np.isclose(S[0, 15, 15], (2 * 0.3 * 0.7 + oloss.C1) / (0.09 + 0.49 + oloss.C1), rtol=1e-12)


@pytest.mark.parametrize("lam", [0.2, 1.0])
def test_loss_gradient_matches_central_differences(lam):
    rng = np.random.default_rng(7)
    x = rng.uniform(0.1, 0.9, (3, 7, 9))
    y = np.clip(x + rng.choice([-1, 1], x.shape) * rng.uniform(0.05, 0.2, x.shape), 0, 1)
    _, g = oloss.loss_l1_dssim(x, y, lam)
    h = 1e-6
    fd = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        fd[idx] = (oloss.loss_l1_dssim(xp, y, lam)[0] - oloss.loss_l1_dssim(xm, y, lam)[0]) / (2 * h)
    assert np.allclose(g, fd, rtol=1e-6, atol=1e-9 * np.abs(g).max())
