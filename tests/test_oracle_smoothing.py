"""Pins of the label-smoothing oracle (q = (1 - eps) onehot + eps / V)."""
import math
from decimal import Decimal, getcontext

import numpy as np
import pytest
import torch

import gen
from oracle import ce_oracle as O


@pytest.mark.parametrize("V", [1, 2, 1000, 128256])
@pytest.mark.parametrize("eps", [0.0, 0.1, 0.9])
def test_uniform_rows(V, eps):
    z = np.full((2, V), -0.5)
    labels = np.array([0, V - 1])
    r = O.ce_smoothed(z, labels, eps, "sum", grad_output=1.5)
    np.testing.assert_allclose(r["loss_rows"], math.log(V), rtol=1e-13, atol=1e-300)
    want = np.full((2, V), 1.5 * (1 - eps) / V)
    want[np.arange(2), labels] = 1.5 * (1 - eps) * (1.0 / V - 1.0)
    np.testing.assert_allclose(r["grad"], want, rtol=1e-12, atol=1e-300)


@pytest.mark.parametrize("V", [2, 1000])
@pytest.mark.parametrize("m", [0.0, 17.0, 50.0])
@pytest.mark.parametrize("eps", [0.05, 0.3])
def test_margin_row(V, m, eps):
    z = np.full((1, V), 0.25)
    z[0, 3 % V] += m
    t = np.array([3 % V])
    r = O.ce_smoothed(z, t, eps, "sum")
    q = (V - 1) * math.exp(-m)
    want = math.log1p(q) + eps * m * (1 - 1.0 / V)
    assert abs(r["loss_rows"][0] - want) <= 1e-13 * want + 1e-300
    g = r["grad"][0]
    assert abs(g[t[0]] - (-q / (1 + q) + eps * (1 - 1.0 / V))) <= 1e-13
    others = np.delete(g, t[0])
    np.testing.assert_allclose(others, math.exp(-m) / (1 + q) - eps / V, rtol=1e-12, atol=1e-18)


def test_eps_zero_is_the_plain_oracle():
    p = gen.custom(40, 300, "f32", seed=2, n_margin=5, n_ignore=3)
    z = O.widen(p.full(), "f32")
    a = O.ce_smoothed(z, p.labels, 0.0, "mean")
    b = O.ce(z, p.labels, "mean")
    assert np.array_equal(a["loss_rows"], b["loss_rows"]) and np.array_equal(a["grad"], b["grad"])


@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
@pytest.mark.parametrize("eps", [0.1, 0.6])
def test_against_torch_float64(reduction, eps):
    p = gen.custom(48, 700, "f32", seed=13, std=3.0, n_margin=5, margin=(3.0, 10.0), n_ignore=4)
    z = O.widen(p.full(), "f32")
    zt = torch.tensor(z, requires_grad=True)
    loss = torch.nn.functional.cross_entropy(zt, torch.tensor(p.labels), ignore_index=O.IGNORE_INDEX,
                                             reduction=reduction, label_smoothing=eps)
    go = np.linspace(0.5, 1.5, 48) if reduction == "none" else 1.0
    loss.backward(torch.tensor(go) if reduction == "none" else torch.tensor(1.0, dtype=torch.float64))
    r = O.ce_smoothed(z, p.labels, eps, reduction, grad_output=go)
    if reduction == "none":
        np.testing.assert_allclose(r["loss_rows"], loss.detach().numpy(), rtol=1e-12, atol=1e-13)
    else:
        assert abs(r["loss_out"] - loss.item()) <= 1e-12 * abs(loss.item())
    np.testing.assert_allclose(r["grad"], zt.grad.numpy(), rtol=1e-9, atol=1e-15)


def test_brute_force_decimal():
    getcontext().prec = 400
    rng = np.random.default_rng(4)
    z = rng.normal(0, 2, (6, 5))
    labels = rng.integers(0, 5, 6)
    z[0, labels[0]] += 40.0
    z[1, labels[1]] += 300.0
    eps = 0.2
    r = O.ce_smoothed(z, labels, eps, "sum")
    for i in range(6):
        zs = [Decimal(float(v)) for v in z[i]]
        tot = sum((v.exp() for v in zs), Decimal(0))
        logp = [v - tot.ln() for v in zs]
        q = [Decimal(eps) / 5 + (Decimal(1 - eps) if j == labels[i] else 0) for j in range(5)]
        loss = -sum(qj * lp for qj, lp in zip(q, logp))
        grad = [lp.exp() - qj for lp, qj in zip(logp, q)]
        assert abs(r["loss_rows"][i] - float(loss)) <= 1e-13 * float(loss)
        np.testing.assert_allclose(r["grad"][i], [float(g) for g in grad], rtol=1e-12, atol=1e-17)
