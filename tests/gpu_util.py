"""Helpers of the GPU parity tests: move the seeded inputs to the device,
run the layer through the C ABI, and compare against the float64 oracle."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from dropless_mixture_experts_gb300.layer import MoELayer
from dropless_mixture_experts_gb300.synthetic import make_inputs, params_of

# Tolerances on max|a - ref| / max|ref| per output tensor: float32 storage
# with strict float32 arithmetic, and bfloat16 storage with float32
# accumulation.
TOL = {"f32": 1e-4, "bf16": 2e-2}


def elem_err(a, ref):
    """The elementwise companion of rel_err: max over elements of
    |a - ref| / (|ref| + 1e-3 max|ref|) (reported beside the normwise metric,
    not held to the tolerance: near-zero elements of a bf16 result carry the
    rounding of the large terms that cancelled in them)."""
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    if not ref.size:
        return 0.0
    floor = 1e-3 * float(np.max(np.abs(ref)))
    if floor == 0.0:
        return float(np.max(np.abs(a)))
    return float(np.max(np.abs(a - ref) / (np.abs(ref) + floor)))


def rel_err(a, ref):
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = float(np.max(np.abs(ref))) if ref.size else 0.0
    if scale == 0.0:
        return float(np.max(np.abs(a))) if a.size else 0.0
    return float(np.max(np.abs(a - ref))) / scale


def to_dev(inp, dtype):
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    out = {}
    for k, v in inp.items():
        # the router bias is float32 for either storage type
        kd = torch.float32 if k == "router_bias" else td
        out[k] = None if v is None else torch.from_numpy(np.ascontiguousarray(v)).to("cuda").to(kd)
    return out


def host(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def run_layer(cfg, seed_offset=0, train=True, inputs=None):
    """Runs the layer on the device; returns (inputs, layer, results dict)."""
    inp = inputs if inputs is not None else make_inputs(cfg, seed_offset=seed_offset)
    dev = to_dev(inp, cfg.dtype)
    layer = MoELayer(cfg.tokens, cfg.d_model, cfg.d_hidden, cfg.experts, cfg.top_k,
                     cfg.shared_hidden, cfg.dtype, train=train, capacity=cfg.capacity)
    p = {k: dev[k] for k in params_of(inp)}
    res = {}
    if train:
        loss, dx, grads = layer.train_step(dev["x"], p, dev["upstream"])
        torch.cuda.synchronize()
        res["loss"] = float(loss.item())
        res["dx"] = host(dx)
        for k, v in grads.items():
            if v is not None:
                res[k] = host(v)
    else:
        layer.forward(dev["x"], p)
        torch.cuda.synchronize()
    status, detail = layer.device_status()
    res["status"] = status
    for k in ("y", "logits", "gates"):
        res[k] = host(getattr(layer, k))
    for k in ("idx", "counts", "offsets", "perm", "inv_perm"):
        res[k] = getattr(layer, k).cpu().numpy().astype(np.int64)
    return inp, layer, dev, res


def check_routing_bit_exact(res, cfg):
    """Oracle's selection and counting sort on the device's own logits."""
    idx, gates = oracle.route_from_logits(res["logits"], cfg.top_k)
    assert np.array_equal(idx, res["idx"]), "top-k indices differ"
    g_err = np.max(np.abs(gates - res["gates"]) / np.abs(gates))
    assert g_err < 1e-6, g_err
    counts, offsets, perm, inv = oracle.counting_sort(res["idx"], cfg.experts, cfg.capacity)
    assert np.array_equal(counts, res["counts"])
    assert np.array_equal(offsets, res["offsets"])
    assert np.array_equal(perm, res["perm"])
    assert np.array_equal(inv, res["inv_perm"])


def oracle_on_device_routing(inp, res, cfg, train=True):
    p = params_of(inp)
    if train:
        L, fwd, grads = oracle.train_step(inp["x"], p, cfg.top_k, inp["upstream"],
                                          idx=res["idx"], logits=res["logits"],
                                          capacity=cfg.capacity)
        return L, fwd, grads
    fwd = oracle.forward(inp["x"], p, cfg.top_k, idx=res["idx"], logits=res["logits"],
                         capacity=cfg.capacity)
    return None, fwd, None


GRADS = ("dw_router", "dw_gate", "dw_up", "dw_down", "dws_gate", "dws_up", "dws_down")
ROUTED = ("dw_gate", "dw_up", "dw_down")


def per_expert_err(a, ref, counts):
    """max over experts with at least one (kept) row of rel_err(a[e], ref[e]),
    each expert against its own scale: an expert with a handful of rows has
    a gradient far smaller than a hot expert's, and a whole-tensor scale
    would hide its errors."""
    worst = 0.0
    for e in np.nonzero(np.asarray(counts) > 0)[0]:
        worst = max(worst, rel_err(a[e], ref[e]))
    return worst


def compare_layer(inp, res, cfg, train=True, report=None):
    """Returns {name: rel_err} for every output of the forward / train step,
    with the routed weight gradients also checked expert by expert
    ("<name>/expert").  `report` (a dict), when given, receives the
    elementwise metric of every output beside the normwise one."""
    L, fwd, grads = oracle_on_device_routing(inp, res, cfg, train)
    errs = {"y": rel_err(res["y"], fwd["y"])}
    elem = {"y": elem_err(res["y"], fwd["y"])}
    logits_ref = oracle.router_logits(inp["x"], inp["w_router"], inp.get("router_bias"))
    errs["logits"] = rel_err(res["logits"], logits_ref)
    if train:
        errs["loss"] = abs(res["loss"] - L) / max(1e-30, float(np.sum(np.abs(fwd["y"] * inp["upstream"]))))
        errs["dx"] = rel_err(res["dx"], grads["dx"])
        elem["dx"] = elem_err(res["dx"], grads["dx"])
        for k in GRADS:
            if k in grads:
                errs[k] = rel_err(res[k], grads[k])
                elem[k] = elem_err(res[k], grads[k])
        for k in ROUTED:
            errs[k + "/expert"] = per_expert_err(res[k], grads[k], res["counts"])
    if report is not None:
        report["normwise"] = dict(errs)
        report["elementwise"] = elem
    return errs


def log_report(name, report):
    """Appends one parity record to the JSON-lines file named by the
    MOE_PARITY_LOG environment variable (nothing when it is unset)."""
    import json
    import os
    path = os.environ.get("MOE_PARITY_LOG")
    if not path:
        return
    with open(path, "a") as f:
        f.write(json.dumps({"case": name, **report}) + "\n")
