"""Pins of the oracle's routing (top-k + softmax over the selected logits)
and of its counting-sort permutation."""

import numpy as np
import pytest

import oracle
from oracle_pins import brute_force_topk, permutation_discrepancy, routing_discrepancy

from dropless_mixture_experts_gb300.synthetic import CONFIGS, make_inputs


@pytest.mark.parametrize("E,k", [(4, 1), (4, 2), (5, 3), (6, 6), (8, 2)])
def test_topk_matches_brute_force_with_ties(E, k):
    rng = np.random.default_rng(E * 10 + k)
    # small integer logits force many exact ties; include signed zeros
    logits = rng.integers(-2, 3, size=(40, E)).astype(np.float64)
    logits[0, :] = 0.0
    logits[1, :] = -0.0
    logits[2, ::2] = -0.0
    assert routing_discrepancy(oracle, logits, k) < 1e-15


def test_topk_continuous_logits():
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((64, 8)).astype(np.float32).astype(np.float64)
    assert routing_discrepancy(oracle, logits, 2) < 1e-15


def test_tie_goes_to_lower_index_and_slots_descend():
    idx, gates = oracle.route_from_logits(np.array([[1.0, 3.0, 3.0, 2.0, 3.0]]), 3)
    assert idx.tolist() == [[1, 2, 4]]
    np.testing.assert_allclose(gates, [[1 / 3] * 3], rtol=0, atol=1e-15)
    idx, _ = oracle.route_from_logits(np.array([[0.0, -0.0, 0.0]]), 2)
    assert idx.tolist() == [[0, 1]]


def test_gate_invariants():
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((500, 64))
    idx, gates = oracle.route_from_logits(logits, 8)
    np.testing.assert_allclose(gates.sum(1), 1.0, rtol=0, atol=1e-14)
    assert np.all(np.diff(gates, axis=1) <= 0)
    assert all(len(set(r)) == 8 for r in idx.tolist())
    # k = 1: the gate is exactly 1
    _, g1 = oracle.route_from_logits(logits, 1)
    assert np.all(g1 == 1.0)


def test_brute_force_helper_itself():
    # the helper's notion of order on a case checked by hand
    assert brute_force_topk(np.array([2.0, 5.0, 5.0, -1.0]), 2).tolist() == [1, 2]


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (9, 4, 2), (300, 8, 2), (257, 64, 8), (50, 5, 5)])
def test_counting_sort_matches_library_sort(T, E, k):
    rng = np.random.default_rng(T + E + k)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    assert permutation_discrepancy(oracle, idx, E) == 0
    counts, offsets, perm, inv = oracle.counting_sort(idx, E)
    assert counts.sum() == T * k
    assert np.array_equal(np.sort(perm), np.arange(T * k))          # bijection
    assert np.array_equal(perm[inv], np.arange(T * k))


def test_counting_sort_empty_and_single_expert():
    idx = np.zeros((10, 1), dtype=np.int64)  # every token on expert 0 of 4
    counts, offsets, perm, inv = oracle.counting_sort(idx, 4)
    assert counts.tolist() == [10, 0, 0, 0]
    assert offsets.tolist() == [0, 10, 10, 10, 10]
    assert perm.tolist() == list(range(10))


def test_uniform_routing_load_sanity():
    """Sanity only (not parity): with i.i.d. router weights the busiest
    expert's share of pairs is near 1/E, as in the pages' layer runs
    (max_expert_frac about 0.13 at E=8, k=2)."""
    cfg = CONFIGS["e8k2_bf16_32k"]
    inp = make_inputs(cfg, with_upstream=False)
    logits = oracle.router_logits(inp["x"], inp["w_router"])
    idx, _ = oracle.route_from_logits(logits, cfg.top_k)
    counts = np.bincount(idx.reshape(-1), minlength=cfg.experts)
    frac = counts.max() / idx.size
    assert 0.125 <= frac < 0.2
    assert np.count_nonzero(counts == 0) == 0
