"""Pins of the oracle's train step (value and gradients): torch autograd of
an independently written dense-masked layer, central finite differences,
and exact zeros for experts that receive no token."""

import numpy as np
import pytest

import oracle
from oracle_pins import autograd_discrepancy, fd_discrepancy, tiny_problem


@pytest.mark.parametrize("E,k,hs", [(4, 2, 0), (4, 2, 6), (6, 3, 0), (4, 1, 5)])
def test_gradients_match_torch_autograd(E, k, hs):
    x, p, G = tiny_problem(T=13, d=8, h=12, E=E, k=k, hs=hs, seed=11 + E + k + hs)
    assert autograd_discrepancy(oracle, x, p, k, G) < 1e-11


@pytest.mark.parametrize("hs", [0, 6])
def test_gradients_match_finite_differences(hs):
    x, p, G = tiny_problem(T=7, d=8, h=12, E=4, k=2, hs=hs, seed=21 + hs)
    assert fd_discrepancy(oracle, x, p, 2, G, n_probe=5) < 1e-7


def test_empty_expert_gets_exactly_zero_gradient():
    x, p, G = tiny_problem(T=12, d=8, h=12, E=4, k=1, seed=5)
    # impose a routing that never uses expert 3
    logits = oracle.router_logits(x, p["w_router"])
    idx = np.argmax(logits[:, :3], axis=1)[:, None]
    L, fwd, grads = oracle.train_step(x, p, 1, G, idx=idx)
    assert fwd["counts"][3] == 0
    assert np.all(grads["dw_gate"][3] == 0)
    assert np.all(grads["dw_up"][3] == 0)
    assert np.all(grads["dw_down"][3] == 0)
    assert np.all(grads["dw_router"][:, 3] == 0)


def test_router_gradient_sums_to_zero_per_token():
    # softmax over the selected logits is invariant to a common shift
    x, p, G = tiny_problem(T=10, d=8, h=12, E=5, k=3, seed=9)
    _, _, grads = oracle.train_step(x, p, 3, G)
    np.testing.assert_allclose(grads["dlogits"].sum(1), 0.0, atol=1e-13)
