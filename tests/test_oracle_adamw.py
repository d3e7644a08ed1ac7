"""Pins the oracle's AdamW arithmetic.

Adam per coordinate (ZeRO reading notes, papers.chlience.com, 3):
m <- b1 m + (1-b1) g, v <- b2 v + (1-b2) g^2, theta <- theta - lr m_hat/(sqrt(v_hat)+eps),
with decoupled weight decay.  Pinned against torch.optim.AdamW (an independent
fp32 implementation, a few ulps apart because its operation order differs),
against the closed form of the first step, and against special cases."""
import numpy as np
import pytest
import torch

from helpers import f32, hyper32, ulp_dist


def _oracle_steps(orc, theta0, grads16, dt, h, steps):
    master = theta0.copy()
    m = np.zeros_like(master)
    v = np.zeros_like(master)
    param = np.zeros(master.size, np.uint16)
    out = []
    for t in range(1, steps + 1):
        sc = orc.make_scalars(h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], t)
        orc.apply(grads16[t - 1], dt, master, m, v, param, dt, 1.0, sc)
        out.append((master.copy(), m.copy(), v.copy(), param.copy()))
    return out


@pytest.mark.parametrize("dt", [1, 2])
def test_matches_torch_adamw(orc, dt):
    rng = np.random.default_rng(11 + dt)
    n, steps = 50000, 3
    h = hyper32()
    theta0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g32 = [(rng.standard_normal(n) * 10.0 ** rng.uniform(-5, -1, n)).astype(np.float32) for _ in range(steps)]
    grads16 = [orc.round_to_16(g, dt) for g in g32]
    ours = _oracle_steps(orc, theta0, grads16, dt, h, steps)

    p = torch.nn.Parameter(torch.from_numpy(theta0.copy()))
    opt = torch.optim.AdamW([p], lr=h["lr"], betas=(h["beta1"], h["beta2"]), eps=h["eps"],
                            weight_decay=h["weight_decay"], foreach=False)
    u = 2.0 ** -24
    th_prev, m_prev, v_prev = theta0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t in range(steps):
        # one step from the same state on both sides (torch's state is re-synced to the oracle's)
        with torch.no_grad():
            p.copy_(torch.from_numpy(th_prev))
        if t > 0:
            st = opt.state[p]
            st["exp_avg"].copy_(torch.from_numpy(m_prev))
            st["exp_avg_sq"].copy_(torch.from_numpy(v_prev))
        g = orc.widen_16(grads16[t], dt)
        p.grad = torch.from_numpy(g.copy())
        opt.step()
        st = opt.state[p]
        m_ref, v_ref = st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()
        th, m, v, _ = ours[t]
        # v is a sum of non-negative terms: a few ulps apart
        assert ulp_dist(v, v_ref).max() <= 4
        # m and theta are differences that can cancel: compare against the size of their terms
        m_terms = h["beta1"] * np.abs(m_prev.astype(np.float64)) + (1 - h["beta1"]) * np.abs(g)
        assert (np.abs(m - m_ref) <= 4 * u * m_terms).all()
        th_terms = np.abs(th_prev.astype(np.float64)) + h["lr"]
        assert (np.abs(th - p.detach().numpy()) <= 8 * u * th_terms).all()
        th_prev, m_prev, v_prev = th, m, v


def test_first_step_closed_form(orc):
    # at t = 1 the bias corrections cancel: m_hat = g, v_hat = g^2, so
    # theta_1 = theta_0 (1 - lr wd) - lr g / (|g| + eps): a step of ~lr per element.
    rng = np.random.default_rng(5)
    n = 20000
    h = hyper32()
    theta0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g16 = orc.round_to_16((rng.standard_normal(n) * 1e-3).astype(np.float32), 1)
    th1 = _oracle_steps(orc, theta0, [g16], 1, h, 1)[0][0]
    g = orc.widen_16(g16, 1).astype(np.float64)
    closed = theta0.astype(np.float64) * (1 - h["lr"] * h["weight_decay"]) - h["lr"] * g / (np.abs(g) + h["eps"])
    assert np.abs(th1 - closed).max() <= 4 * np.spacing(np.abs(closed).astype(np.float32)).max()
    big = np.abs(g) > 1e-5
    step = th1[big].astype(np.float64) - theta0[big] * (1 - h["lr"] * h["weight_decay"])
    assert np.allclose(np.abs(step), h["lr"], rtol=2e-3)
    assert np.all(np.sign(step) == -np.sign(g[big]))


def test_zero_gradient_only_decays(orc):
    n = 1000
    h = hyper32()
    theta0 = np.linspace(-1, 1, n).astype(np.float32)
    zero = np.zeros(n, np.uint16)
    th, m, v, param = _oracle_steps(orc, theta0, [zero, zero], 2, h, 2)[-1]
    assert not m.any() and not v.any()
    wdf = np.float32(1.0 - np.float64(h["lr"]) * np.float64(h["weight_decay"]))
    assert np.array_equal(th, (theta0 * wdf) * wdf)
    assert np.array_equal(param, orc.round_to_16(th, 2))


def test_scalars_closed_form(orc):
    h = hyper32()
    for t in (1, 2, 3, 100, 10000):
        s = orc.make_scalars(h["lr"], h["beta1"], h["beta2"], h["eps"], h["weight_decay"], t)
        assert s.ss == pytest.approx(h["lr"] / (1 - h["beta1"] ** t), rel=1e-7)
        assert s.rb2 == pytest.approx((1 - h["beta2"] ** t) ** -0.5, rel=1e-7)
        # 1 - beta1 is taken of the fp32 beta1 (0.8999999761...), then rounded once
        assert s.omb1 == f32(1.0 - h["beta1"]) and s.b2 == f32(0.999)
