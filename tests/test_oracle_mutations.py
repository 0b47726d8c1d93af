"""Mutation checks of the oracle's pins: a copy of the oracle with one
plausible mistake planted in its source (on the CPU) must fail at least one
pin.  This shows the pins can see dropped terms, wrong signs, wrong indices
and swapped operands."""

import importlib.util
import os

import numpy as np
import pytest

import oracle
from oracle_pins import (autograd_discrepancy, capacity_permutation_discrepancy,
                         dense_discrepancy, permutation_discrepancy, routing_discrepancy,
                         tiny_problem)

SRC = os.path.join(os.path.dirname(os.path.dirname(__file__)), "oracle", "moe_oracle.py")


def mutant(old, new):
    text = open(SRC).read()
    assert text.count(old) == 1, old
    spec = importlib.util.spec_from_loader("oracle_mutant", loader=None)
    mod = importlib.util.module_from_spec(spec)
    exec(compile(text.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


MUTATIONS = [
    # ties resolved towards the higher expert index
    ("tie", 'order = np.argsort(-logits, axis=1, kind="stable")',
     'order = (E - 1) - np.argsort(-logits[:, ::-1], axis=1, kind="stable")'),
    # softmax over all logits instead of the selected ones
    ("gates_all", "gates = z / z.sum(axis=1, keepdims=True)\n    return idx, gates",
     "gates = z / np.exp(logits - sel[:, :1]).sum(axis=1, keepdims=True)\n    return idx, gates"),
    # unstable order inside an expert
    ("unstable", "members = np.nonzero((flat == e) & keep)[0]  # increasing pair id",
     "members = np.nonzero((flat == e) & keep)[0][::-1]"),
    # combine takes the other slot's expert output
    ("slot", "rows = inv_perm[np.arange(T) * top_k + j]",
     "rows = inv_perm[np.arange(T) * top_k + (top_k - 1 - j)]"),
    # silu with the wrong sign inside the sigmoid
    ("silu_sign", "return a / (1.0 + np.exp(-a))", "return a / (1.0 + np.exp(a))"),
    # dropped softmax-Jacobian term in the router gradient
    ("router_term", "dsel = gates * (dgate - np.sum(gates * dgate, axis=1, keepdims=True))",
     "dsel = gates * dgate"),
    # silu derivative without its second factor
    ("dsilu", "dA_g = dH * A_u * s * (1.0 + A_g * (1.0 - s))", "dA_g = dH * A_u * s"),
    # up/gate swapped in the input gradient
    ("dx_swap", "dX = dA_g @ w_gate.T + dA_u @ w_up.T", "dX = dA_g @ w_up.T + dA_u @ w_gate.T"),
    # gate applied twice to the expert output gradient
    ("gate_twice", "dO = g * G[toks]", "dO = g * g * G[toks]"),
    # router input-gradient term dropped
    ("router_dx", "dx += dlogits @ _f64(params[\"w_router\"]).T", "pass"),
    # capacity keeps an expert's last pairs instead of its first
    ("capacity_last", "keep[members if not capacity else members[:capacity]] = True",
     "keep[members if not capacity else members[-capacity:]] = True"),
    # capacity renormalises the gates over the kept slots
    ("capacity_renorm", "        y[kept] += gates[kept, j:j + 1] * O[rows[kept]]",
     "        kg = gates * capacity_keep(idx, E, capacity)\n"
     "        kg = kg / np.maximum(kg.sum(axis=1, keepdims=True), 1e-300)\n"
     "        y[kept] += kg[kept, j:j + 1] * O[rows[kept]]"),
]


def any_pin_fails(mod):
    rng = np.random.default_rng(0)
    logits = rng.integers(-2, 3, size=(30, 5)).astype(np.float64)
    if routing_discrepancy(mod, logits, 2) > 1e-12:
        return True
    idx = np.stack([rng.permutation(6)[:3] for _ in range(40)])
    if permutation_discrepancy(mod, idx, 6) != 0:
        return True
    if capacity_permutation_discrepancy(mod, idx, 6, 15) != 0:
        return True
    x, p, G = tiny_problem(T=13, d=8, h=12, E=4, k=2, hs=5, seed=3)
    if dense_discrepancy(mod, x, p, 2) > 1e-12:
        return True
    if dense_discrepancy(mod, x, p, 2, capacity=4) > 1e-12:
        return True
    if autograd_discrepancy(mod, x, p, 2, G, capacity=4) > 1e-9:
        return True
    return autograd_discrepancy(mod, x, p, 2, G) > 1e-9


def test_unmutated_oracle_passes_the_same_pins():
    assert not any_pin_fails(oracle)


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new):
    assert any_pin_fails(mutant(old, new)), name
