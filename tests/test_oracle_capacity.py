"""Pins of the oracle's capacity routing (each expert keeps its first C pairs
in increasing pair id; dropped pairs leave the mixture, not the softmax)."""

import numpy as np
import pytest

import oracle
from oracle_pins import (autograd_discrepancy, capacity_permutation_discrepancy,
                         dense_discrepancy, tiny_problem)


@pytest.mark.parametrize("capacity", [1, 3, 7, 40])
def test_capacity_sort_matches_running_counters(capacity):
    rng = np.random.default_rng(capacity)
    idx = np.stack([rng.permutation(6)[:3] for _ in range(40)])
    assert capacity_permutation_discrepancy(oracle, idx, 6, capacity) == 0


def test_capacity_at_or_above_the_largest_count_is_dropless():
    rng = np.random.default_rng(1)
    idx = np.stack([rng.permutation(5)[:2] for _ in range(30)])
    counts = np.bincount(idx.reshape(-1), minlength=5)
    for cap in (int(counts.max()), int(counts.max()) + 9):
        for a, b in zip(oracle.counting_sort(idx, 5, cap), oracle.counting_sort(idx, 5)):
            assert np.array_equal(a, b)
    x, p, G = tiny_problem(T=13, d=8, h=12, E=4, k=2, hs=5, seed=3)
    L0, f0, g0 = oracle.train_step(x, p, 2, G)
    L1, f1, g1 = oracle.train_step(x, p, 2, G, capacity=26)
    assert L0 == L1 and np.array_equal(f0["y"], f1["y"])
    for k in g0:
        assert np.array_equal(g0[k], g1[k]), k


@pytest.mark.parametrize("capacity", [1, 2, 4])
def test_capacity_forward_matches_dense_masked(capacity):
    x, p, _ = tiny_problem(T=13, d=8, h=12, E=4, k=2, hs=5, seed=3)
    assert dense_discrepancy(oracle, x, p, 2, capacity=capacity) < 1e-12


@pytest.mark.parametrize("capacity", [1, 4])
def test_capacity_train_step_matches_torch_autograd(capacity):
    x, p, G = tiny_problem(T=13, d=8, h=12, E=4, k=2, hs=5, seed=3)
    assert autograd_discrepancy(oracle, x, p, 2, G, capacity=capacity) < 1e-9


def test_fully_dropped_token_keeps_only_the_shared_expert():
    # capacity 1 on 2 experts, every token on both: only token 0 is kept
    x, p, G = tiny_problem(T=5, d=8, h=12, E=2, k=2, hs=5, seed=4)
    fwd = oracle.forward(x, p, 2, capacity=1)
    assert np.array_equal(fwd["counts"], [1, 1])
    shared = oracle.swiglu_expert(x, p["ws_gate"], p["ws_up"], p["ws_down"])[3]
    assert np.array_equal(fwd["y"][1:], shared[1:])
    assert np.all(fwd["inv_perm"][2:] == -1)
    _, _, grads = oracle.train_step(x, p, 2, G, capacity=1)
    # a dropped pair's gate gradient is zero, but the softmax still couples
    # it to the kept slot of its token: the logit gradient of token 0 is not
    assert np.all(grads["dgate"][1:] == 0.0)
    assert np.any(grads["dlogits"][0] != 0.0)
    assert np.all(grads["dlogits"][1:] == 0.0)


def test_router_bias_offsets_the_logits_and_trains_no_bias():
    from oracle_pins import autograd_discrepancy
    x, p, G = tiny_problem(T=13, d=8, h=12, E=4, k=2, hs=5, seed=3)
    # no bias and a zero bias give the same step
    L0, f0, g0 = oracle.train_step(x, p, 2, G)
    pz = dict(p, router_bias=np.zeros(4))
    L1, f1, g1 = oracle.train_step(x, pz, 2, G)
    assert L0 == L1 and all(np.array_equal(g0[k], g1[k]) for k in g0)
    # a bias far above every logit puts its expert in every token's first slot
    pb = dict(p, router_bias=np.array([0.0, 0.0, 50.0, 0.0]))
    fwd = oracle.forward(x, pb, 2)
    assert np.all(fwd["idx"][:, 0] == 2)
    # value and gradients agree with torch autograd with the offset held constant
    pr = dict(p, router_bias=np.array([0.3, -0.2, 0.1, -0.4]))
    assert autograd_discrepancy(oracle, x, pr, 2, G) < 1e-9
    assert autograd_discrepancy(oracle, x, pr, 2, G, capacity=4) < 1e-9
