"""Pins of the oracle's load-balance metrics, loss and gradient.

Reading (the pages name the load-balance loss and the per-expert counts it is
built from, not its formula): f_e = c_e/(T*K), P_e = mean_t softmax(l_t)_e,
L = E * sum_e f_e P_e, gradient with f held fixed."""
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "load_balance_example.txt")


def test_uniform_routing_gives_exactly_one():
    T, E, K = 64, 8, 2
    idx = (np.arange(T * K).reshape(T, K) % E).astype(np.int32)   # every expert 16 times
    r = O.load_balance(np.zeros((T, E)), idx, E)
    assert r["loss"] == 1.0
    assert np.all(r["f"] == 1.0 / E) and np.all(r["P"] == 1.0 / E)
    assert r["max_over_uniform"] == 1.0 and r["n_empty"] == 0


def test_collapsed_routing_closed_form():
    """K = 1, every token to expert 0 with logit gap g: f = e_0,
    P_0 = 1 / (1 + (E-1) e^-g), L = E * P_0."""
    T, E, g = 10, 16, 7.0
    l = np.zeros((T, E))
    l[:, 0] = g
    idx = np.zeros((T, 1), dtype=np.int32)
    r = O.load_balance(l, idx, E)
    p0 = 1.0 / (1.0 + (E - 1) * np.exp(-g))
    assert abs(r["loss"] - E * p0) < 1e-13
    assert r["max_over_uniform"] == E and r["n_empty"] == E - 1


def test_metrics_hand_example():
    """tests/golden/load_balance_example.txt: E=4, K=2, three tokens routed by hand."""
    rows = [ln.split() for ln in open(GOLDEN) if ln.strip() and not ln.startswith("#")]
    kv = {r[0]: [float(v) for v in r[1:]] for r in rows}
    idx = np.array(kv["idx"], dtype=np.int32).reshape(3, 2)
    r = O.load_balance(np.zeros((3, 4)), idx, 4)
    assert np.allclose(r["f"], kv["f"], rtol=0, atol=1e-15)
    assert r["max_over_uniform"] == kv["max_over_uniform"][0]
    assert r["n_empty"] == int(kv["n_empty"][0])
    assert abs(r["loss"] - kv["loss"][0]) < 1e-15


@pytest.mark.parametrize("T,E,K", [(5, 4, 2), (17, 8, 3), (9, 32, 8)])
def test_gradient_matches_torch_autograd(T, E, K):
    g = np.random.default_rng(T * E + K)
    l = g.normal(size=(T, E))
    idx = np.argsort(-l, axis=1, kind="stable")[:, :K].astype(np.int32)
    r = O.load_balance(l, idx, E)
    lt = torch.tensor(l, dtype=torch.float64, requires_grad=True)
    f = torch.tensor(r["f"], dtype=torch.float64)
    loss = E * (f * torch.softmax(lt, dim=1).mean(0)).sum()
    assert abs(loss.item() - r["loss"]) < 1e-12
    loss.backward()
    got = O.load_balance_backward(l, r["f"], scale=1.0)
    assert np.allclose(got, lt.grad.numpy(), rtol=1e-10, atol=1e-13)
    assert np.allclose(O.load_balance_backward(l, r["f"], scale=-2.5), -2.5 * got, rtol=1e-14)


def test_gradient_finite_differences_and_row_sums():
    g = np.random.default_rng(3)
    T, E, K = 6, 5, 2
    l = g.normal(size=(T, E))
    idx = np.argsort(-l, axis=1, kind="stable")[:, :K]
    f = O.load_balance(l, idx, E)["f"]
    loss = lambda x: E * float(np.dot(f, O.softmax(x).mean(0)))  # noqa: E731
    d = O.load_balance_backward(l, f)
    h = 1e-6
    for t, i in [(0, 0), (2, 3), (5, 4)]:
        lp, lm = l.copy(), l.copy()
        lp[t, i] += h
        lm[t, i] -= h
        assert abs((loss(lp) - loss(lm)) / (2 * h) - d[t, i]) < 1e-8
    assert np.allclose(d.sum(axis=1), 0.0, atol=1e-15)   # softmax gradients sum to zero per token
