"""Parity at the full sizes of the benchmark workloads (the E8/k2 layer at
4k, 32k and 128k tokens in float32 and bfloat16, the fine-grained E64/k4
layer and the E64/k8 decoder block with a shared expert at 16k and 128k
tokens), in the launch configuration the bench times, against the float64
oracle run on the same device routing.  The oracle is run in full (a few
seconds to ~15 s of host BLAS per configuration)."""

import numpy as np
import pytest

from dropless_mixture_experts_gb300.synthetic import CONFIGS
from gpu_util import TOL, check_routing_bit_exact, compare_layer, log_report, run_layer

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

NAMES = list(CONFIGS)


@pytest.mark.parametrize("name", NAMES)
def test_full_size_train_step(name):
    cfg = CONFIGS[name]
    inp, layer, dev, res = run_layer(cfg, train=True)
    assert res["status"] == 0
    check_routing_bit_exact(res, cfg)
    report = {}
    errs = compare_layer(inp, res, cfg, train=True, report=report)
    log_report(name + "/train", report)
    bad = {k: v for k, v in errs.items() if not v <= TOL[cfg.dtype]}
    assert not bad, (name, errs)
    # routing sanity against the pages' layer runs: no empty expert, the
    # busiest expert near 1/E of the pairs
    counts = res["counts"]
    assert counts.sum() == cfg.tokens * cfg.top_k
    assert np.count_nonzero(counts == 0) == 0
    assert counts.max() / counts.sum() < 2.0 / cfg.experts


@pytest.mark.parametrize("name", ["e8k2_bf16_32k", "decoder_bf16_16k"])
def test_full_size_skewed_train_step(name):
    # skewed routing (the router bias ramp of the bench's --skew 0.9) at a
    # bench size: hot experts whose K ranges the weight-gradient schedule
    # cuts into chunks (partials summed by the last chunk to finish), empty
    # experts whose gradients must be exact zeros
    import dataclasses
    cfg = dataclasses.replace(CONFIGS[name], skew=0.9)
    inp, layer, dev, res = run_layer(cfg, train=True)
    assert res["status"] == 0
    check_routing_bit_exact(res, cfg)
    report = {}
    errs = compare_layer(inp, res, cfg, train=True, report=report)
    log_report(name + "/train_skew", report)
    bad = {k: v for k, v in errs.items() if not v <= TOL[cfg.dtype]}
    assert not bad, (name, errs)
    counts = res["counts"]
    assert counts.max() / counts.sum() > 2.0 / cfg.experts  # the routing is skewed
    for k in ("dw_gate", "dw_up", "dw_down"):
        for e in np.nonzero(counts == 0)[0]:
            assert not np.any(res[k][e]), (k, e)


@pytest.mark.parametrize("name", NAMES)
def test_full_size_forward_only(name):
    # the forward-only mode (nothing saved for a backward) the forward
    # throughput is measured in, against the oracle's forward on the same
    # device routing
    cfg = CONFIGS[name]
    inp, layer, dev, res = run_layer(cfg, train=False)
    assert res["status"] == 0
    check_routing_bit_exact(res, cfg)
    report = {}
    errs = compare_layer(inp, res, cfg, train=False, report=report)
    log_report(name + "/forward", report)
    bad = {k: v for k, v in errs.items() if not v <= TOL[cfg.dtype]}
    assert not bad, (name, errs)
