"""Independent checks that pin the float64 oracle to something other than
itself.  Each returns a discrepancy (0 / small = the oracle agrees).  They are
used by the pin tests and, against deliberately broken copies of the oracle,
by the mutation tests (a pin that cannot see a planted mistake is useless).
"""

from __future__ import annotations

import itertools

import numpy as np
import scipy.special
import torch


def brute_force_topk(logits_row, k):
    """The unique ordered k-tuple of distinct experts whose logits are
    non-increasing, whose equal logits appear in increasing index order, and
    such that every chosen expert beats every unchosen one under the rule
    'larger logit wins, equal logits go to the lower index'.  Found by
    enumerating every ordered k-tuple."""
    E = len(logits_row)

    def beats(a, b):
        return logits_row[a] > logits_row[b] or (logits_row[a] == logits_row[b] and a < b)

    found = []
    for tup in itertools.permutations(range(E), k):
        if not all(beats(tup[i], tup[i + 1]) for i in range(k - 1)):
            continue
        rest = [e for e in range(E) if e not in tup]
        if all(beats(a, b) for a in tup for b in rest):
            found.append(tup)
    assert len(found) == 1, found
    return np.array(found[0])


def routing_discrepancy(oracle, logits, k):
    """Max over tokens of (index mismatch vs brute force) + gate error vs
    scipy's softmax of the selected logits + gate error vs the renormalised
    full softmax."""
    idx, gates = oracle.route_from_logits(logits, k)
    bad = 0.0
    full = scipy.special.softmax(np.asarray(logits, np.float64), axis=1)
    for t in range(logits.shape[0]):
        bf = brute_force_topk(logits[t], k)
        if not np.array_equal(idx[t], bf):
            bad = max(bad, 1.0)
            continue
        ref = scipy.special.softmax(np.asarray(logits[t], np.float64)[bf])
        bad = max(bad, float(np.max(np.abs(gates[t] - ref))))
        renorm = full[t, bf] / full[t, bf].sum()
        bad = max(bad, float(np.max(np.abs(gates[t] - renorm))))
    return bad


def permutation_discrepancy(oracle, idx, E):
    """0 when counts/offsets/perm/inv_perm equal what numpy's library
    routines give: bincount, cumsum, a lexicographic sort by (expert, pair)
    and the inverse of that permutation."""
    counts, offsets, perm, inv = oracle.counting_sort(idx, E)
    flat = np.asarray(idx).reshape(-1)
    ref_counts = np.bincount(flat, minlength=E)
    ref_offsets = np.concatenate([[0], np.cumsum(ref_counts)])
    ref_perm = np.lexsort((np.arange(flat.size), flat))
    ref_inv = np.empty_like(ref_perm)
    ref_inv[ref_perm] = np.arange(flat.size)
    bad = 0
    bad += int(not np.array_equal(counts, ref_counts))
    bad += int(not np.array_equal(offsets, ref_offsets))
    bad += int(not np.array_equal(perm, ref_perm))
    bad += int(not np.array_equal(inv, ref_inv))
    return bad


def capacity_permutation_discrepancy(oracle, idx, E, capacity):
    """0 when the oracle's capacity-routed counting sort equals an
    independent construction: pairs visited in increasing id with one running
    counter per expert decide what is kept; bincount, cumsum and a
    lexicographic sort by (expert, pair) of the kept pairs give counts,
    offsets and perm (-1 past the kept rows); inv_perm is -1 on dropped
    pairs."""
    counts, offsets, perm, inv = oracle.counting_sort(idx, E, capacity)
    flat = np.asarray(idx).reshape(-1)
    seen = [0] * E
    kept = []
    for p_, e in enumerate(flat):
        if seen[e] < capacity:
            kept.append(p_)
        seen[e] += 1
    kept = np.array(kept, dtype=np.int64)
    ref_counts = np.bincount(flat[kept], minlength=E)
    ref_offsets = np.concatenate([[0], np.cumsum(ref_counts)])
    ref_perm = np.full(flat.size, -1)
    ref_perm[:kept.size] = kept[np.lexsort((kept, flat[kept]))]
    ref_inv = np.full(flat.size, -1)
    ref_inv[ref_perm[:kept.size]] = np.arange(kept.size)
    bad = 0
    bad += int(not np.array_equal(counts, ref_counts))
    bad += int(not np.array_equal(offsets, ref_offsets))
    bad += int(not np.array_equal(perm, ref_perm))
    bad += int(not np.array_equal(inv, ref_inv))
    return bad


def torch_keep_mask(sel_idx, E, capacity):
    """Capacity keep mask [T, k] from torch library ops: a pair's rank in its
    expert is the running count (cumsum over pairs in id order) of the
    one-hot expert matrix, minus one; kept when the rank is below the
    capacity (None: every pair)."""
    T, k = sel_idx.shape
    if not capacity:
        return torch.ones((T, k), dtype=torch.float64)
    onehot = torch.nn.functional.one_hot(sel_idx.reshape(-1), E).to(torch.float64)
    rank = (torch.cumsum(onehot, dim=0) * onehot).sum(dim=1) - 1.0
    return (rank < capacity).to(torch.float64).reshape(T, k)


def torch_dense_layer(x, params, k, idx=None, capacity=None):
    """The dense-masked layer written with torch library ops in float64 and
    differentiated by torch autograd (with a capacity, the gates of dropped
    pairs are masked out of the mixture, not out of the softmax).  Returns
    (y, {name: tensor}) with the tensors requiring grad."""
    t = {kk: (None if v is None else torch.tensor(np.asarray(v, np.float64), requires_grad=True))
         for kk, v in params.items() if kk != "router_bias"}
    tx = torch.tensor(np.asarray(x, np.float64), requires_grad=True)
    logits = tx @ t["w_router"]
    if params.get("router_bias") is not None:  # a constant offset: no gradient
        logits = logits + torch.tensor(np.asarray(params["router_bias"], np.float64))
    if idx is None:
        sel, sel_idx = torch.topk(logits, k, dim=1)
    else:
        sel_idx = torch.tensor(np.asarray(idx, np.int64))
        sel = torch.gather(logits, 1, sel_idx)
    gates = torch.softmax(sel, dim=1)
    E = t["w_gate"].shape[0]
    keep = torch_keep_mask(sel_idx, E, capacity)
    mask = torch.zeros(logits.shape, dtype=torch.float64).scatter(1, sel_idx, gates * keep)
    y = torch.zeros_like(tx)
    for e in range(E):
        a = torch.nn.functional.silu(tx @ t["w_gate"][e]) * (tx @ t["w_up"][e])
        y = y + mask[:, e:e + 1] * (a @ t["w_down"][e])
    if t.get("ws_down") is not None:
        a = torch.nn.functional.silu(tx @ t["ws_gate"]) * (tx @ t["ws_up"])
        y = y + a @ t["ws_down"]
    leaves = {"x": tx}
    leaves.update({kk: v for kk, v in t.items() if v is not None})
    return y, leaves, sel_idx.numpy()


GRAD_NAMES = {"x": "dx", "w_router": "dw_router", "w_gate": "dw_gate", "w_up": "dw_up",
              "w_down": "dw_down", "ws_gate": "dws_gate", "ws_up": "dws_up", "ws_down": "dws_down"}


def autograd_discrepancy(oracle, x, params, k, G, capacity=None):
    """Max relative difference between the oracle's value and gradients and
    torch autograd through the dense-masked torch formulation."""
    y, leaves, idx = torch_dense_layer(x, params, k, capacity=capacity)
    L = (y * torch.tensor(np.asarray(G, np.float64))).sum()
    L.backward()
    Lo, fwd, grads = oracle.train_step(x, params, k, G, capacity=capacity)
    worst = abs(Lo - L.item()) / max(1.0, abs(L.item()))
    worst = max(worst, float(np.max(np.abs(fwd["y"] - y.detach().numpy()))))
    for name, leaf in leaves.items():
        ref = leaf.grad.numpy()
        got = grads[GRAD_NAMES[name]]
        scale = max(1e-30, float(np.max(np.abs(ref))))
        worst = max(worst, float(np.max(np.abs(got - ref))) / scale)
    return worst


def fd_discrepancy(oracle, x, params, k, G, n_probe=6, eps=1e-6, seed=0):
    """Central finite differences of L = sum(y*G) on a few random entries of
    every input/parameter, holding the routing fixed only where the
    perturbation does not change it (entries whose perturbation flips the
    top-k are skipped).  Returns the max relative error."""
    rng = np.random.default_rng(seed)
    base_idx = oracle.route_from_logits(oracle.router_logits(x, params["w_router"]), k)[0]
    _, _, grads = oracle.train_step(x, params, k, G)
    worst = 0.0
    tensors = {"x": x}
    tensors.update({kk: v for kk, v in params.items() if v is not None})
    for name, arr in tensors.items():
        arr = np.asarray(arr, np.float64)
        g = grads[GRAD_NAMES[name]]
        for _ in range(n_probe):
            pos = tuple(int(rng.integers(0, s)) for s in arr.shape)
            vals = []
            ok = True
            for sgn in (+1, -1):
                a2 = arr.copy()
                a2[pos] += sgn * eps
                xx = a2 if name == "x" else np.asarray(x, np.float64)
                pp = dict(params)
                if name != "x":
                    pp[name] = a2
                idx2 = oracle.route_from_logits(oracle.router_logits(xx, pp["w_router"]), k)[0]
                if not np.array_equal(idx2, base_idx):
                    ok = False
                    break
                vals.append(oracle.loss(oracle.forward(xx, pp, k)["y"], G))
            if not ok:
                continue
            fd = (vals[0] - vals[1]) / (2 * eps)
            scale = max(1e-3, float(np.max(np.abs(g))))
            worst = max(worst, abs(fd - g[pos]) / scale)
    return worst


def dense_discrepancy(oracle, x, params, k, capacity=None):
    """Sorted-dispatch forward vs the brute-force dense-masked forward."""
    y_sorted = oracle.forward(x, params, k, capacity=capacity)["y"]
    y_dense = oracle.dense_masked_forward(x, params, k, capacity=capacity)
    return float(np.max(np.abs(y_sorted - y_dense)))


def tiny_problem(T=7, d=8, h=12, E=4, k=2, hs=0, seed=0, margin=1e-3):
    """A small float64 problem whose top-k gaps all exceed ``margin`` (so a
    finite-difference step cannot flip the routing)."""
    rng = np.random.default_rng(seed)
    for _ in range(1000):
        x = rng.standard_normal((T, d))
        p = {
            "w_router": rng.standard_normal((d, E)) / np.sqrt(d),
            "w_gate": rng.standard_normal((E, d, h)) / np.sqrt(d),
            "w_up": rng.standard_normal((E, d, h)) / np.sqrt(d),
            "w_down": rng.standard_normal((E, h, d)) / np.sqrt(h),
            "ws_gate": None, "ws_up": None, "ws_down": None,
        }
        if hs:
            p["ws_gate"] = rng.standard_normal((d, hs)) / np.sqrt(d)
            p["ws_up"] = rng.standard_normal((d, hs)) / np.sqrt(d)
            p["ws_down"] = rng.standard_normal((hs, d)) / np.sqrt(hs)
        logits = x @ p["w_router"]
        srt = -np.sort(-logits, axis=1)
        if k < E and np.min(srt[:, k - 1] - srt[:, k]) < margin:
            continue
        G = rng.standard_normal((T, d))
        return x, p, G
    raise RuntimeError("no well-separated problem found")
