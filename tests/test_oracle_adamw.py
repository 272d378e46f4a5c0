"""Pins of the oracle's AdamW step for the adapters (paged optimizers:
inquiringlines.com note, mechanism paragraph; ashishsrivastav.com, section
"Paged Optimizers: Managing Fragmentation"). The update rule itself is a
reading (AdamW with decoupled weight decay); it is pinned by closed forms and
by torch.optim.AdamW in float64."""
import numpy as np
import torch

HP = dict(lr=2e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)


def test_first_step_from_zero_state(oracle):
    rng = np.random.default_rng(1)
    p0 = rng.standard_normal(1000)
    g = rng.standard_normal(1000)
    p, m, v = p0.copy(), np.zeros(1000), np.zeros(1000)
    oracle.adamw_step(p, g, m, v, step=1, **HP)
    # bias-corrected m and v are g and g^2 after one step
    lr, wd, eps = HP["lr"], HP["weight_decay"], HP["eps"]
    expect = p0 * (1 - lr * wd) - lr * g / (np.abs(g) + eps)
    assert np.allclose(p, expect, rtol=0, atol=1e-15)
    assert np.allclose(m, 0.1 * g) and np.allclose(v, 0.001 * g * g)


def test_constant_gradient_walks_linearly(oracle):
    # with a constant gradient the corrected moments stay g and g^2, so
    # without decay every step moves lr * g / (|g| + eps)
    hp = dict(HP, weight_decay=0.0)
    g = np.array([0.5, -2.0, 3e-3, -7.0])
    p, m, v = np.zeros(4), np.zeros(4), np.zeros(4)
    for t in range(1, 26):
        oracle.adamw_step(p, g, m, v, step=t, **hp)
    assert np.allclose(p, -25 * hp["lr"] * g / (np.abs(g) + hp["eps"]), rtol=1e-12, atol=0)


def test_decay_alone(oracle):
    p0 = np.array([1.0, -3.0, 0.25])
    p, m, v = p0.copy(), np.zeros(3), np.zeros(3)
    for t in range(1, 11):
        oracle.adamw_step(p, np.zeros(3), m, v, step=t, **HP)
    assert np.allclose(p, p0 * (1 - HP["lr"] * HP["weight_decay"]) ** 10, rtol=1e-14, atol=0)


def test_matches_torch_adamw(oracle):
    rng = np.random.default_rng(2)
    p0 = rng.standard_normal(257)
    grads = [rng.standard_normal(257) * (1 + t) for t in range(6)]
    tp = torch.tensor(p0, dtype=torch.float64, requires_grad=True)
    opt = torch.optim.AdamW([tp], lr=HP["lr"], betas=(HP["beta1"], HP["beta2"]), eps=HP["eps"],
                            weight_decay=HP["weight_decay"])
    p, m, v = p0.copy(), np.zeros(257), np.zeros(257)
    for t, gr in enumerate(grads, 1):
        tp.grad = torch.tensor(gr, dtype=torch.float64)
        opt.step()
        oracle.adamw_step(p, gr, m, v, step=t, **HP)
    assert np.allclose(p, tp.detach().numpy(), rtol=1e-13, atol=1e-15)
    st = opt.state[tp]
    assert np.allclose(m, st["exp_avg"].numpy(), rtol=1e-13) and np.allclose(v, st["exp_avg_sq"].numpy(), rtol=1e-13)
