"""Pins of the oracle's forward pass: the dense-masked brute force, special
cases that reduce to textbook layers, the parameter count and a hand-worked
closed-form case."""

import json
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle_pins import dense_discrepancy, tiny_problem

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_case.json")


@pytest.mark.parametrize("E,k,hs", [(4, 2, 0), (4, 2, 6), (8, 3, 0), (5, 1, 0), (3, 3, 4)])
def test_sorted_dispatch_equals_dense_masked(E, k, hs):
    x, p, _ = tiny_problem(T=23, d=8, h=12, E=E, k=k, hs=hs, seed=E + k + hs)
    assert dense_discrepancy(oracle, x, p, k) < 1e-12


def test_one_expert_is_a_dense_swiglu_mlp():
    x, p, _ = tiny_problem(T=11, d=8, h=12, E=1, k=1, seed=3)
    y = oracle.forward(x, p, 1)["y"]
    tx = torch.tensor(x)
    ref = (torch.nn.functional.silu(tx @ torch.tensor(p["w_gate"][0]))
           * (tx @ torch.tensor(p["w_up"][0]))) @ torch.tensor(p["w_down"][0])
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-13, atol=1e-13)


def test_k_equals_E_is_full_softmax_mixture():
    x, p, _ = tiny_problem(T=9, d=8, h=12, E=4, k=4, seed=4)
    y = oracle.forward(x, p, 4)["y"]
    w = scipy.special.softmax(x @ p["w_router"], axis=1)
    tx = torch.tensor(x)
    ref = np.zeros_like(x)
    for e in range(4):
        o = ((torch.nn.functional.silu(tx @ torch.tensor(p["w_gate"][e]))
              * (tx @ torch.tensor(p["w_up"][e]))) @ torch.tensor(p["w_down"][e])).numpy()
        ref += w[:, e:e + 1] * o
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_silu_closed_forms():
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(oracle.silu(np.array([np.log(3.0)])), [0.75 * np.log(3.0)], rtol=1e-15)
    np.testing.assert_allclose(oracle.silu(np.array([-np.log(3.0)])), [-0.25 * np.log(3.0)], rtol=1e-15)
    assert abs(oracle.silu(np.array([40.0]))[0] - 40.0) < 1e-12


def test_param_count_matches_pages():
    # gpu_nn benchmark page, moe rows: params = 12587008 (E=8, d=512, h=1024)
    assert oracle.param_count(512, 1024, 8) == 12_587_008


def test_hand_worked_case():
    g = json.load(open(GOLDEN))
    k = g["top_k"]
    x = np.array(g["x"])
    p = {key: np.array(g[key]) for key in ("w_router", "w_gate", "w_up", "w_down")}
    p.update(ws_gate=None, ws_up=None, ws_down=None)
    G = np.array(g["upstream"])
    L, fwd, grads = oracle.train_step(x, p, k, G)
    ex = g["expected"]
    assert fwd["idx"].tolist() == ex["idx"]
    assert fwd["counts"].tolist() == ex["counts"]
    assert fwd["offsets"].tolist() == ex["offsets"]
    assert fwd["perm"].tolist() == ex["perm"]
    assert fwd["inv_perm"].tolist() == ex["inv_perm"]
    np.testing.assert_allclose(fwd["gates"], ex["gates"]["value"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(fwd["y"], ex["y"]["value"], rtol=1e-14, atol=1e-15)
    assert abs(L - ex["loss"]["value"]) < 1e-13
    np.testing.assert_allclose(grads["dw_down"], ex["dw_down"]["value"], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(grads["dw_router"], ex["dw_router"]["value"], rtol=1e-13, atol=1e-15)


def test_fed_routing_reproduces_own_routing():
    x, p, _ = tiny_problem(T=15, d=8, h=12, E=4, k=2, seed=7)
    a = oracle.forward(x, p, 2)
    b = oracle.forward(x, p, 2, idx=a["idx"])
    np.testing.assert_allclose(a["y"], b["y"], rtol=0, atol=1e-14)
