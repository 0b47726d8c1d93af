"""Float64 CPU oracle of the dropless, sorted-dispatch mixture-of-experts layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module.  The CUDA library never calls it and shares no code with it; the only
thing both sides consume is the seeded input generator, which holds none of
the method's arithmetic.

What it computes (plain definitions, in float64, no blocking or fusion):

* router logits ``x @ W_r``, a bias-free ``d_model x experts`` router (the
  layer's parameter count on the gpu_nn benchmark page, ``results[suite=moe]
  .params`` = 12,587,008 = 8 * 3 * 512 * 1024 + 512 * 8, leaves no bias);
* top-k selection per token, ties to the lower expert index, slots in
  descending logit order, gates = softmax over the k selected logits;
* the counting-sort permutation of the token-expert pairs by expert (the
  ``sort_permute`` piece of the kernel_gmm_gpu benchmark page's pieces suite,
  dispatch ``sorted``), stable by pair id;
* per-expert bias-free SwiGLU FFNs ``(silu(X W_gate) * (X W_up)) W_down`` on
  each expert's rows (the ``experts_grouped_swiglu`` piece);
* the gate-weighted combine back to token order (``unpermute_combine`` piece)
  plus an optional always-on shared SwiGLU expert (the ``shared`` field of the
  gpu_moe_h100 benchmark page's ``v10_decoder`` rows);
* the train step's value and gradients with respect to the input and every
  parameter (the gpu_moe_h100 page's description: value_and_grad w.r.t. params
  and input), for the scalar L = sum(y * G) with G the upstream gradient;
* optionally capacity routing (the ``routing: capacity`` rows of the
  kernel_gmm_gpu page, which give neither the capacity nor the drop rule):
  each expert keeps its first ``capacity`` pairs in increasing pair id and
  drops the rest; a dropped pair contributes nothing to y, while the gates
  stay the softmax over all k selected logits.

Pins (``tests/test_oracle_*.py``) tie every function to something other than
itself: brute-force subset enumeration, library sorts and softmax, the
brute-force dense-masked formulation (the pages' ``dense`` routing), torch
autograd and central finite differences, closed forms and a hand-worked
golden case.
"""

from __future__ import annotations

import numpy as np

__all__ = [
    "param_count",
    "router_logits",
    "route_from_logits",
    "capacity_keep",
    "counting_sort",
    "silu",
    "swiglu_expert",
    "forward",
    "dense_masked_forward",
    "loss",
    "backward",
    "train_step",
]


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def param_count(d_model: int, d_hidden: int, experts: int, shared_hidden: int = 0) -> int:
    """Parameters of the layer: E experts x 3 bias-free SwiGLU matrices, a
    bias-free router and the optional shared expert.

    gpu_nn benchmark page, ``results[suite=moe].params`` (12,587,008 for
    E=8, d_model=512, d_hidden=1024, no shared expert)."""
    return experts * 3 * d_model * d_hidden + d_model * experts + 3 * d_model * shared_hidden


def router_logits(x, w_router, router_bias=None):
    """logits[t, e] = sum_i x[t, i] * W_r[i, e]  (the ``route`` piece), plus
    an optional fixed per-expert offset (the skewed-routing runs; the layer
    trains no bias)."""
    logits = _f64(x) @ _f64(w_router)
    return logits if router_bias is None else logits + _f64(router_bias)[None, :]


def route_from_logits(logits, top_k: int):
    """Top-k selection and softmax over the selected logits.

    For each token the experts are ranked by (-logit, expert index): the
    largest logit first, equal logits resolved towards the lower expert index
    (+0.0 and -0.0 compare equal).  Slot j holds the (j+1)-th ranked expert.
    gates[t, :] = softmax(logits[t, idx[t, :]]), evaluated with the largest
    selected logit subtracted.

    Returns (idx int64 [T, k], gates float64 [T, k]).
    """
    logits = _f64(logits)
    T, E = logits.shape
    if not 1 <= top_k <= E:
        raise ValueError("need 1 <= top_k <= experts")
    # A stable sort on -logit keeps equal logits in expert-index order.
    order = np.argsort(-logits, axis=1, kind="stable")
    idx = order[:, :top_k].astype(np.int64)
    sel = np.take_along_axis(logits, idx, axis=1)
    z = np.exp(sel - sel[:, :1])
    gates = z / z.sum(axis=1, keepdims=True)
    return idx, gates


def capacity_keep(idx, experts: int, capacity=None):
    """Which pairs capacity routing keeps: for each expert, its first
    ``capacity`` pairs in increasing pair id p = t*k + j (capacity None or 0:
    every pair, the dropless layer).  Returns a bool array shaped like idx."""
    flat = np.asarray(idx, dtype=np.int64).reshape(-1)
    keep = np.zeros(flat.size, dtype=bool)
    for e in range(experts):
        members = np.nonzero(flat == e)[0]  # increasing pair id
        keep[members if not capacity else members[:capacity]] = True
    return keep.reshape(np.shape(idx))


def counting_sort(idx, experts: int, capacity=None):
    """Counting sort of the T*k token-expert pairs by expert.

    Pair p = t*k + j carries expert idx[t, j].  counts[e] = number of pairs on
    expert e; offsets = exclusive prefix sum (length E+1); perm[r] = the pair
    at expert-sorted position r, pairs of one expert kept in increasing pair
    id (a token picks distinct experts, so this is also increasing token id);
    inv_perm[perm[r]] = r.

    With a capacity, only the pairs ``capacity_keep`` keeps are sorted:
    counts and offsets count kept pairs, perm[r] = -1 for r >= offsets[E]
    and inv_perm[p] = -1 for a dropped pair.
    """
    flat = np.asarray(idx, dtype=np.int64).reshape(-1)
    P = flat.size
    keep = capacity_keep(idx, experts, capacity).reshape(-1)
    counts = np.zeros(experts, dtype=np.int64)
    for e in range(experts):
        counts[e] = int(np.count_nonzero((flat == e) & keep))
    offsets = np.zeros(experts + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    perm = np.full(P, -1, dtype=np.int64)
    inv_perm = np.full(P, -1, dtype=np.int64)
    for e in range(experts):
        members = np.nonzero((flat == e) & keep)[0]  # increasing pair id
        pos = offsets[e] + np.arange(members.size)
        perm[pos] = members
        inv_perm[members] = pos
    return counts, offsets, perm, inv_perm


def silu(a):
    """silu(a) = a * sigmoid(a)."""
    a = _f64(a)
    return a / (1.0 + np.exp(-a))


def _sigmoid(a):
    return 1.0 / (1.0 + np.exp(-_f64(a)))


def swiglu_expert(X, w_gate, w_up, w_down):
    """One bias-free SwiGLU FFN on the rows of X.

    A_g = X W_gate, A_u = X W_up, H = silu(A_g) * A_u, O = H W_down.
    Returns (A_g, A_u, H, O)."""
    X = _f64(X)
    A_g = X @ _f64(w_gate)
    A_u = X @ _f64(w_up)
    H = silu(A_g) * A_u
    O = H @ _f64(w_down)
    return A_g, A_u, H, O


def forward(x, params, top_k: int, idx=None, logits=None, capacity=None):
    """Layer forward pass.

    params: dict with w_router [d,E], w_gate [E,d,h], w_up [E,d,h],
    w_down [E,h,d] and, optionally, ws_gate [d,hs], ws_up [d,hs],
    ws_down [hs,d] (the shared expert; absent or None = no shared expert).

    ``idx`` may be given to impose the routing (for parity runs that feed the
    routing decided on the device); the gates are then the softmax of the
    given or computed logits at those indices.  ``logits`` may be given to
    route from fed logits.  ``capacity`` (pairs per expert) switches on
    capacity routing (``capacity_keep``).

    y[t] = sum over kept slots j of gates[t, j] * O[inv_perm[t*k + j]]
    (slot order)  + shared(x[t]).
    Returns a dict holding every intermediate.
    """
    x = _f64(x)
    T, d = x.shape
    w_gate = _f64(params["w_gate"])
    E = w_gate.shape[0]
    if logits is None:
        logits = router_logits(x, params["w_router"], params.get("router_bias"))
    logits = _f64(logits)
    if idx is None:
        idx, gates = route_from_logits(logits, top_k)
    else:
        idx = np.asarray(idx, dtype=np.int64)
        sel = np.take_along_axis(logits, idx, axis=1)
        z = np.exp(sel - sel.max(axis=1, keepdims=True))
        gates = z / z.sum(axis=1, keepdims=True)
    counts, offsets, perm, inv_perm = counting_sort(idx, E, capacity)

    P = T * top_k
    h = w_gate.shape[2]
    A_g = np.zeros((P, h))
    A_u = np.zeros((P, h))
    H = np.zeros((P, h))
    O = np.zeros((P, d))
    tok_of_row = perm // top_k
    for e in range(E):
        rows = slice(offsets[e], offsets[e + 1])
        if offsets[e + 1] == offsets[e]:
            continue
        Xe = x[tok_of_row[rows]]
        A_g[rows], A_u[rows], H[rows], O[rows] = swiglu_expert(
            Xe, w_gate[e], params["w_up"][e], params["w_down"][e])

    y = np.zeros((T, d))
    for j in range(top_k):
        rows = inv_perm[np.arange(T) * top_k + j]
        kept = rows >= 0
        y[kept] += gates[kept, j:j + 1] * O[rows[kept]]

    shared = None
    if params.get("ws_down") is not None:
        shared = swiglu_expert(x, params["ws_gate"], params["ws_up"], params["ws_down"])
        y = y + shared[3]

    return dict(y=y, logits=logits, idx=idx, gates=gates, counts=counts,
                offsets=offsets, perm=perm, inv_perm=inv_perm, A_g=A_g,
                A_u=A_u, H=H, O=O, shared=shared)


def dense_masked_forward(x, params, top_k: int, idx=None, capacity=None):
    """Brute-force formulation: every expert on every token, weighted by a
    dense [T, E] gate matrix that is zero off the selected experts (the
    ``dense`` routing of the kernel_gmm_gpu benchmark page) and, with a
    capacity, at the dropped pairs.  No permutation is involved, so it checks
    the sorted dispatch end to end."""
    x = _f64(x)
    T, _ = x.shape
    E = _f64(params["w_gate"]).shape[0]
    logits = router_logits(x, params["w_router"], params.get("router_bias"))
    if idx is None:
        idx, gates = route_from_logits(logits, top_k)
    else:
        idx = np.asarray(idx, dtype=np.int64)
        sel = np.take_along_axis(logits, idx, axis=1)
        z = np.exp(sel - sel.max(axis=1, keepdims=True))
        gates = z / z.sum(axis=1, keepdims=True)
    G = np.zeros((T, E))
    np.put_along_axis(G, idx, gates * capacity_keep(idx, E, capacity), axis=1)
    y = np.zeros_like(x)
    for e in range(E):
        O = swiglu_expert(x, params["w_gate"][e], params["w_up"][e], params["w_down"][e])[3]
        y += G[:, e:e + 1] * O
    if params.get("ws_down") is not None:
        y += swiglu_expert(x, params["ws_gate"], params["ws_up"], params["ws_down"])[3]
    return y


def loss(y, upstream):
    """Scalar objective of the train step: L = sum(y * G)."""
    return float(np.sum(_f64(y) * _f64(upstream)))


def _swiglu_backward(X, A_g, A_u, H, dO, w_gate, w_up, w_down):
    """Gradients of O = (silu(X Wg) * (X Wu)) Wd given dO (per row).

    dH = dO Wd^T; dA_u = dH * silu(A_g);
    dA_g = dH * A_u * s * (1 + A_g (1 - s)) with s = sigmoid(A_g);
    dWd = H^T dO; dWg = X^T dA_g; dWu = X^T dA_u; dX = dA_g Wg^T + dA_u Wu^T."""
    w_gate, w_up, w_down = _f64(w_gate), _f64(w_up), _f64(w_down)
    dH = dO @ w_down.T
    s = _sigmoid(A_g)
    dA_u = dH * (A_g * s)
    dA_g = dH * A_u * s * (1.0 + A_g * (1.0 - s))
    dWd = H.T @ dO
    dWg = X.T @ dA_g
    dWu = X.T @ dA_u
    dX = dA_g @ w_gate.T + dA_u @ w_up.T
    return dX, dWg, dWu, dWd, dA_g, dA_u


def backward(x, params, top_k: int, upstream, fwd):
    """Analytic gradients of L = sum(y * G) with respect to x and every
    parameter, given the forward dict ``fwd`` (value_and_grad of the
    gpu_moe_h100 benchmark page's train step).

    Per pair (t, j) on expert e at sorted row r, with dy = G:
      dO_r = gates[t, j] * dy_t                (expert output gradient)
      dgate[t, j] = <dy_t, O_r>                (0 for a pair capacity dropped)
      expert weight / input gradients through the SwiGLU chain rule;
    router: the gates are a softmax of the selected logits, so
      dlogit[t, idx[t, j]] = g_j * (dgate_j - sum_i g_i dgate_i),
    zero on the experts that were not selected (selection is piecewise
    constant); dW_r = x^T dlogit; dx += dlogit W_r^T.
    """
    x = _f64(x)
    G = _f64(upstream)
    T, d = x.shape
    w_gate = _f64(params["w_gate"])
    E, _, h = w_gate.shape
    idx, gates = fwd["idx"], fwd["gates"]
    offsets, perm, inv_perm = fwd["offsets"], fwd["perm"], fwd["inv_perm"]
    P = T * top_k
    tok_of_row = perm // top_k
    pair_gate = gates.reshape(-1)

    dx = np.zeros((T, d))
    dW_gate = np.zeros_like(w_gate)
    dW_up = np.zeros_like(w_gate)
    dW_down = np.zeros((E, h, d))
    dgate_pair = np.zeros(P)
    for e in range(E):
        rows = np.arange(offsets[e], offsets[e + 1])
        if rows.size == 0:
            continue
        toks = tok_of_row[rows]
        g = pair_gate[perm[rows]][:, None]
        dO = g * G[toks]
        dgate_pair[perm[rows]] = np.sum(G[toks] * fwd["O"][rows], axis=1)
        dX, dWg, dWu, dWd, _, _ = _swiglu_backward(
            x[toks], fwd["A_g"][rows], fwd["A_u"][rows], fwd["H"][rows], dO,
            w_gate[e], params["w_up"][e], params["w_down"][e])
        dW_gate[e] = dWg
        dW_up[e] = dWu
        dW_down[e] = dWd
        # a token selects distinct experts, so `toks` has no repeats here
        dx[toks] += dX

    dgate = dgate_pair.reshape(T, top_k)
    dsel = gates * (dgate - np.sum(gates * dgate, axis=1, keepdims=True))
    dlogits = np.zeros((T, E))
    np.put_along_axis(dlogits, idx, dsel, axis=1)
    dW_router = x.T @ dlogits
    dx += dlogits @ _f64(params["w_router"]).T

    out = dict(dx=dx, dw_router=dW_router, dw_gate=dW_gate, dw_up=dW_up,
               dw_down=dW_down, dlogits=dlogits, dgate=dgate)
    if fwd["shared"] is not None:
        A_g, A_u, H, _ = fwd["shared"]
        dXs, dWg, dWu, dWd, _, _ = _swiglu_backward(
            x, A_g, A_u, H, G, params["ws_gate"], params["ws_up"], params["ws_down"])
        dx += dXs
        out.update(dws_gate=dWg, dws_up=dWu, dws_down=dWd)
    return out


def train_step(x, params, top_k: int, upstream, idx=None, logits=None, capacity=None):
    """value_and_grad: returns (L, fwd dict, grads dict)."""
    fwd = forward(x, params, top_k, idx=idx, logits=logits, capacity=capacity)
    grads = backward(x, params, top_k, upstream, fwd)
    return loss(fwd["y"], upstream), fwd, grads
