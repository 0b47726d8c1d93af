"""Parity of the CUDA path with the float64 oracle, through the C ABI.

Routing and the permutation are bit-exact on the device's own logits; every
floating-point output is within the stated tolerance of the oracle run on the
same routing.  Sizes span several 128-row tiles with ragged tails."""

import numpy as np
import pytest
import torch

import oracle
from dropless_mixture_experts_gb300.synthetic import MoEConfig, make_inputs, params_of
from gpu_util import (TOL, check_routing_bit_exact, compare_layer, log_report, rel_err, run_layer,
                      to_dev)

pytestmark = pytest.mark.gpu

SMALL = [
    MoEConfig(1000, 128, 192, 4, 2, 0, "f32", "f32_e4k2"),
    MoEConfig(1000, 128, 192, 4, 2, 0, "bf16", "bf16_e4k2"),
    MoEConfig(777, 128, 128, 8, 3, 128, "bf16", "bf16_e8k3_shared"),
    MoEConfig(300, 64, 64, 5, 5, 64, "f32", "f32_k_eq_E_shared"),
    MoEConfig(1, 128, 64, 4, 1, 0, "f32", "f32_one_token"),
    MoEConfig(4097, 128, 64, 16, 4, 0, "bf16", "bf16_e16k4"),
    MoEConfig(2050, 256, 128, 64, 8, 256, "bf16", "bf16_decoder_small"),
    # the largest top-k (a single-stage row stream) and rows that end inside
    # a 512-byte stream piece
    MoEConfig(300, 192, 64, 32, 32, 64, "bf16", "bf16_k32_shared"),
    MoEConfig(200, 64, 64, 32, 32, 0, "f32", "f32_k32"),
    MoEConfig(333, 640, 128, 8, 2, 0, "bf16", "bf16_d640"),
    # d = 512, h = 1024: the down, input-gradient and weight-gradient GEMMs
    # run as CTA pairs over experts padded to 256 rows (the last 128-row
    # tile of an expert may be empty); with a shared expert of 1024 over an
    # odd number of 128-row token tiles (the last pair's odd CTA past the
    # tokens)
    MoEConfig(1500, 512, 1024, 4, 2, 0, "bf16", "bf16_pairs"),
    MoEConfig(1100, 512, 1024, 4, 2, 1024, "bf16", "bf16_pairs_shared"),
    # the same pair paths with capacity routing (kept counts padded to 256)
    # and with skewed routing (empty and hot experts)
    MoEConfig(1500, 512, 1024, 4, 2, 0, "bf16", "bf16_pairs_capacity", capacity=500),
    MoEConfig(1500, 512, 1024, 8, 2, 0, "bf16", "bf16_pairs_skew", skew=0.9),
    # capacity routing: about half the pairs dropped; with a shared expert;
    # float32; one pair per expert
    MoEConfig(2000, 128, 128, 8, 2, 0, "bf16", "bf16_capacity_half", capacity=250),
    MoEConfig(1500, 128, 64, 16, 4, 128, "bf16", "bf16_capacity_shared", capacity=300),
    MoEConfig(700, 64, 64, 4, 2, 0, "f32", "f32_capacity", capacity=200),
    MoEConfig(300, 128, 64, 8, 2, 0, "bf16", "bf16_capacity_1", capacity=1),
    # skewed routing (router bias ramp): a few hot experts, many empty ones
    # at E=64; and skew with a capacity
    MoEConfig(2000, 128, 128, 8, 2, 0, "bf16", "bf16_skew", skew=0.9),
    MoEConfig(2050, 256, 128, 64, 8, 256, "bf16", "bf16_decoder_skew", skew=0.9),
    MoEConfig(1000, 128, 64, 8, 2, 0, "f32", "f32_skew", skew=0.9),
    MoEConfig(2000, 128, 128, 8, 2, 0, "bf16", "bf16_skew_capacity", capacity=250, skew=0.9),
    # degenerate routing: one expert (the layer is a dense SwiGLU MLP with
    # gate 1), and two experts both taken by every token
    MoEConfig(513, 128, 64, 1, 1, 0, "bf16", "bf16_one_expert"),
    MoEConfig(513, 128, 64, 1, 1, 64, "f32", "f32_one_expert_shared"),
    MoEConfig(700, 256, 128, 2, 2, 0, "bf16", "bf16_e2k2"),
    # float32 weight gradients cut into K chunks (experts of 1024-2048 rows
    # over few output tiles: up to eight chunks, summed in chunk order), with
    # a shared expert, and with skewed routing (empty experts: empty chunks)
    MoEConfig(4096, 128, 128, 4, 2, 128, "f32", "f32_dw_chunks_shared"),
    MoEConfig(4096, 128, 64, 8, 2, 0, "f32", "f32_dw_chunks_skew", skew=0.9),
    MoEConfig(4096, 128, 128, 4, 2, 0, "f32", "f32_dw_chunks_capacity", capacity=700),
    # more experts than the tensor-core router takes (E > 64): the logits
    # GEMM, the selection and the router backward on their general paths;
    # the most experts the counting sort takes (256)
    MoEConfig(1000, 128, 64, 128, 4, 64, "bf16", "bf16_e128k4_shared"),
    MoEConfig(1500, 128, 64, 256, 2, 0, "f32", "f32_e256k2"),
    MoEConfig(1000, 128, 64, 256, 2, 0, "bf16", "bf16_e256k2"),
    # a model width and a shared width that are multiples of 64 but not of
    # 128 (64-wide tiles and K blocks of the operand rows)
    MoEConfig(900, 192, 128, 8, 2, 192, "bf16", "bf16_d192_shared192"),
    MoEConfig(900, 192, 128, 8, 2, 192, "f32", "f32_d192_shared192"),
    # the narrowest widths (64) on the tensor-core path, every expert taken
    # by every token; the largest k with the most experts
    MoEConfig(500, 64, 64, 4, 4, 64, "bf16", "bf16_d64_k_eq_E_shared"),
    MoEConfig(300, 128, 64, 256, 32, 0, "bf16", "bf16_e256k32"),
    # one token on the tensor-core path with a shared expert; float32
    # capacity routing beside a shared expert
    MoEConfig(1, 128, 64, 4, 1, 64, "bf16", "bf16_one_token_shared"),
    MoEConfig(1500, 128, 64, 16, 4, 128, "f32", "f32_capacity_shared", capacity=300),
]


@pytest.mark.parametrize("cfg", SMALL, ids=[c.name for c in SMALL])
def test_train_step_matches_oracle(cfg):
    inp, layer, dev, res = run_layer(cfg)
    assert res["status"] == 0
    check_routing_bit_exact(res, cfg)
    report = {}
    errs = compare_layer(inp, res, cfg, train=True, report=report)
    log_report(cfg.name, report)
    bad = {k: v for k, v in errs.items() if not v <= TOL[cfg.dtype]}
    assert not bad, (errs, cfg)


# The numerics grid the kernel_gmm_gpu page planned for its check mode
# (1000 tokens, d128, h256; E 8 / 64; top-1 / top-4; skew 0 / 0.9; fp32 /
# bf16; its results are absent from the page): every combination, train step
# against the oracle.
SWEEP = [MoEConfig(1000, 128, 256, E, k, 0, dt, f"sweep_E{E}_k{k}_s{sk}_{dt}", skew=sk)
         for E in (8, 64) for k in (1, 4) for sk in (0.0, 0.9) for dt in ("f32", "bf16")]


@pytest.mark.parametrize("cfg", SWEEP, ids=[c.name for c in SWEEP])
def test_planned_numerics_sweep(cfg):
    inp, layer, dev, res = run_layer(cfg)
    assert res["status"] == 0
    check_routing_bit_exact(res, cfg)
    report = {}
    errs = compare_layer(inp, res, cfg, train=True, report=report)
    log_report(cfg.name, report)
    bad = {k: v for k, v in errs.items() if not v <= TOL[cfg.dtype]}
    assert not bad, (errs, cfg)


@pytest.mark.parametrize("cfg", SMALL[:3], ids=[c.name for c in SMALL[:3]])
def test_forward_only_matches_train_forward(cfg):
    inp, _, _, r_train = run_layer(cfg, train=True)
    _, _, _, r_fwd = run_layer(cfg, train=False, inputs=inp)
    assert np.array_equal(r_train["idx"], r_fwd["idx"])
    # the combine sums each token's shares in slot order: bit-identical
    assert np.array_equal(r_train["y"], r_fwd["y"])


@pytest.mark.parametrize("cfg", SMALL[1:3], ids=[c.name for c in SMALL[1:3]])
def test_train_step_is_deterministic(cfg):
    inp, _, _, a = run_layer(cfg, train=True)
    _, _, _, b = run_layer(cfg, train=True, inputs=inp)
    for k in ("y", "dx", "loss", "gates", "idx", "perm"):
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("name,shared_sms", [("decoder_bf16_16k", 0), ("decoder_bf16_16k", 48),
                                             ("e8k2_bf16_32k", 0), ("e8k2_f32_4k", 0)])
def test_repeated_train_steps_bit_identical(name, shared_sms):
    # every kernel of the path is deterministic, so repeated train steps on
    # the same inputs give the same bits; a race between a kernel's own
    # stages (a buffer overwritten while still being read) shows up here as
    # a difference between repeats, at sizes with hundreds of tiles per SM
    from dropless_mixture_experts_gb300.synthetic import CONFIGS
    from dropless_mixture_experts_gb300.layer import MoELayer
    cfg = CONFIGS[name]
    inp = make_inputs(cfg)
    dev = to_dev(inp, cfg.dtype)
    p = {k: dev[k] for k in params_of(inp)}
    layer = MoELayer(cfg.tokens, cfg.d_model, cfg.d_hidden, cfg.experts, cfg.top_k,
                     cfg.shared_hidden, cfg.dtype, train=True, shared_sms=shared_sms)
    first = None
    for _ in range(4):
        loss, dx, grads = layer.train_step(dev["x"], p, dev["upstream"])
        torch.cuda.synchronize()
        cur = {"loss": loss.clone(), "dx": dx.clone(), "y": layer.y.clone()}
        cur.update({k: v.clone() for k, v in grads.items() if v is not None})
        if first is None:
            first = cur
            continue
        for k, v in cur.items():
            assert torch.equal(v, first[k]), k
    assert layer.device_status()[0] == 0


@pytest.mark.parametrize("E,k", [(8, 2), (32, 4), (64, 8)])
def test_tensor_core_router_ties(E, k):
    # duplicated router columns give bit-equal logits (each output column of
    # the router GEMM is accumulated alone), so the tensor-core router's
    # selection meets exact ties: the lower expert index must win, and the
    # selection must equal the oracle's on the device's own logits
    cfg = MoEConfig(1500, 256, 128, E, k, 0, "bf16", f"router_ties_E{E}_k{k}")
    inp = make_inputs(cfg)
    w = inp["w_router"].copy()
    for e in range(0, E - 1, 3):
        w[:, e + 1] = w[:, e]
    inp["w_router"] = w
    _, _, _, res = run_layer(cfg, inputs=inp)
    assert res["status"] == 0
    lg = res["logits"]
    assert any(np.array_equal(lg[:, e], lg[:, e + 1]) for e in range(0, E - 1, 3))
    check_routing_bit_exact(res, cfg)


def _fed(cfg, logits):
    inp = make_inputs(cfg)
    dev = to_dev(inp, cfg.dtype)
    from dropless_mixture_experts_gb300.layer import MoELayer
    layer = MoELayer(cfg.tokens, cfg.d_model, cfg.d_hidden, cfg.experts, cfg.top_k,
                     cfg.shared_hidden, cfg.dtype, train=True)
    p = {k: dev[k] for k in params_of(inp)}
    lg = torch.from_numpy(np.ascontiguousarray(logits, np.float32)).cuda()
    loss, dx, grads = layer.train_step(dev["x"], p, dev["upstream"], logits_in=lg)
    torch.cuda.synchronize()
    return inp, layer


@pytest.mark.parametrize("case", ["ties", "one_expert", "empty_experts", "signed_zero"])
def test_fed_logits_routing_and_layer(case):
    cfg = MoEConfig(1500, 128, 64, 8, 2, 0, "f32", case)
    rng = np.random.default_rng(5)
    if case == "ties":
        logits = rng.integers(-2, 3, size=(cfg.tokens, cfg.experts)).astype(np.float32)
    elif case == "one_expert":
        logits = rng.standard_normal((cfg.tokens, cfg.experts)).astype(np.float32)
        logits[:, 3] = 50.0   # every token's first choice is expert 3
    elif case == "empty_experts":
        logits = rng.standard_normal((cfg.tokens, cfg.experts)).astype(np.float32)
        logits[:, 4:] = -50.0  # experts 4..7 never chosen
    else:
        logits = np.zeros((cfg.tokens, cfg.experts), np.float32)
        logits[::2, ::3] = -0.0
    inp, layer = _fed(cfg, logits)
    idx = layer.idx.cpu().numpy()
    ref_idx, ref_g = oracle.route_from_logits(logits.astype(np.float64), cfg.top_k)
    assert np.array_equal(idx, ref_idx)
    np.testing.assert_allclose(layer.gates.cpu().numpy(), ref_g, rtol=1e-6)
    counts, offsets, perm, inv = oracle.counting_sort(ref_idx, cfg.experts)
    assert np.array_equal(layer.counts.cpu().numpy(), counts)
    assert np.array_equal(layer.perm.cpu().numpy(), perm)
    assert np.array_equal(layer.inv_perm.cpu().numpy(), inv)
    L, fwd, grads = oracle.train_step(inp["x"], params_of(inp), cfg.top_k, inp["upstream"],
                                      idx=ref_idx, logits=logits)
    assert rel_err(layer.y.float().cpu().numpy(), fwd["y"]) < TOL["f32"]
    assert rel_err(layer.dx.float().cpu().numpy(), grads["dx"]) < TOL["f32"]
    for k in ("dw_gate", "dw_up", "dw_down", "dw_router"):
        assert rel_err(layer.grads[k].cpu().numpy(), grads[k]) < TOL["f32"], k
    if case == "empty_experts":
        assert np.all(layer.grads["dw_down"][4:].cpu().numpy() == 0)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_zero_tokens(dtype):
    from dropless_mixture_experts_gb300.layer import MoELayer
    layer = MoELayer(0, 128, 64, 4, 2, 64, dtype, train=True)
    inp = make_inputs(MoEConfig(1, 128, 64, 4, 2, 64, dtype))
    dev = to_dev(inp, dtype)
    p = {k: dev[k] for k in params_of(inp)}
    x = dev["x"][:0]
    loss, dx, grads = layer.train_step(x, p, dev["upstream"][:0])
    torch.cuda.synchronize()
    assert float(loss.item()) == 0.0
    for k, v in grads.items():
        if v is not None:
            assert torch.count_nonzero(v).item() == 0, k


def test_out_of_range_expert_index_is_reported_not_faulted():
    from dropless_mixture_experts_gb300 import abi
    from dropless_mixture_experts_gb300.layer import MoELayer
    layer = MoELayer(64, 128, 64, 4, 2, 0, "f32", train=False)
    layer.idx.copy_(torch.zeros(64, 2, dtype=torch.int32))
    layer.idx[5, 1] = 9   # not an expert
    layer.permute()
    status, detail = layer.device_status()
    assert status == abi.MOE_ERR_DEVICE_CHECK
    assert layer.device_status()[0] == 0   # cleared by the read


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rejected_expert_index_is_skipped_through_the_train_step(dtype):
    # a pair whose expert index is out of range gets no sorted row: the
    # permutation reports it and every later kernel skips the pair, so the
    # other tokens' outputs and input gradients equal a clean run's
    from dropless_mixture_experts_gb300 import abi
    from dropless_mixture_experts_gb300.layer import MoELayer
    cfg = MoEConfig(300, 128, 64, 8, 2, 64, dtype, "rejected_index")
    inp = make_inputs(cfg)
    dev = to_dev(inp, dtype)
    p = {k: dev[k] for k in params_of(inp)}
    runs = []
    for corrupt in (False, True):
        layer = MoELayer(cfg.tokens, cfg.d_model, cfg.d_hidden, cfg.experts, cfg.top_k,
                         cfg.shared_hidden, dtype, train=True)
        layer.route(dev["x"], p["w_router"])
        if corrupt:
            layer.idx[5, 1] = 99
            layer.idx[17, 0] = -3
        layer.permute()
        layer.grouped_ffn_fwd(dev["x"], p, abi.MOE_SAVE_FOR_BWD)
        layer.combine(dev["x"], p, abi.MOE_SAVE_FOR_BWD, upstream=dev["upstream"])
        layer.backward(dev["x"], p, dev["upstream"])
        torch.cuda.synchronize()
        status, _ = layer.device_status()
        runs.append((status, layer.y.clone(), layer.dx.clone()))
    assert runs[0][0] == 0
    assert runs[1][0] == abi.MOE_ERR_DEVICE_CHECK
    keep = torch.ones(cfg.tokens, dtype=torch.bool, device="cuda")
    keep[[5, 17]] = False
    assert torch.equal(runs[0][1][keep], runs[1][1][keep])
    assert torch.equal(runs[0][2][keep], runs[1][2][keep])


def test_train_step_from_host_matches_device_inputs():
    # the host-input step (upstream copied on a side stream behind the
    # forward) gives the device-input step's results bit for bit
    cfg = MoEConfig(777, 128, 128, 8, 3, 128, "bf16", "host_inputs")
    inp = make_inputs(cfg)
    dev = to_dev(inp, "bf16")
    p = {k: dev[k] for k in params_of(inp)}
    from dropless_mixture_experts_gb300.layer import MoELayer
    layer = MoELayer(cfg.tokens, cfg.d_model, cfg.d_hidden, cfg.experts, cfg.top_k,
                     cfg.shared_hidden, "bf16", train=True)
    loss, dx, g = layer.train_step(dev["x"], p, dev["upstream"])
    torch.cuda.synchronize()
    ref = (loss.clone(), dx.clone(), {k: v.clone() for k, v in g.items() if v is not None})
    xh = dev["x"].cpu().pin_memory()
    gh = dev["upstream"].cpu().pin_memory()
    lh = torch.empty(1, dtype=torch.float32).pin_memory()
    for _ in range(2):  # the second call reuses the layer's input buffers
        loss2, dx2, g2 = layer.train_step_from_host(xh, p, gh, lh)
        torch.cuda.synchronize()
        assert torch.equal(loss2, ref[0]) and float(lh[0]) == float(ref[0][0])
        assert torch.equal(dx2, ref[1])
        for k, v in ref[2].items():
            assert torch.equal(g2[k], v), k


@pytest.mark.parametrize("shared_sms", [0, 48])
def test_pipelined_host_steps_match_single_steps(shared_sms):
    # the pipelined host-input steps (inputs of the next step copied in and
    # results of the previous one copied out while a step runs, two device
    # slots alternating) give each batch's single-step results bit for bit
    cfg = MoEConfig(1500, 256, 256, 8, 2, 512, "bf16", "pipelined")
    inp = make_inputs(cfg)
    dev = to_dev(inp, "bf16")
    p = {k: dev[k] for k in params_of(inp)}
    from dropless_mixture_experts_gb300.layer import MoELayer
    layer = MoELayer(cfg.tokens, cfg.d_model, cfg.d_hidden, cfg.experts, cfg.top_k,
                     cfg.shared_hidden, "bf16", train=True, shared_sms=shared_sms)
    n = 5
    gen = torch.Generator().manual_seed(11)
    xs = [(dev["x"].cpu().float() + 0.05 * i * torch.randn(dev["x"].shape, generator=gen))
          .to(torch.bfloat16) for i in range(n)]
    dys = [(dev["upstream"].cpu().float() * (1 + 0.1 * i)).to(torch.bfloat16) for i in range(n)]
    refs = []
    for i in range(n):
        loss, dx, g = layer.train_step(xs[i].cuda(), p, dys[i].cuda())
        torch.cuda.synchronize()
        refs.append((loss.clone().cpu(), dx.clone().cpu(), g["dw_gate"].clone()))
    xh = [x.pin_memory() for x in xs]
    gh = [d.pin_memory() for d in dys]
    lh = [torch.empty(1, dtype=torch.float32).pin_memory() for _ in range(n)]
    dxh = [torch.empty(cfg.tokens, cfg.d_model, dtype=torch.bfloat16).pin_memory()
           for _ in range(n)]
    for _ in range(2):  # the second call reuses the slots
        for t in lh + dxh:
            t.zero_()
        layer.train_steps_from_host(xh, p, gh, lh, dxh)
        torch.cuda.synchronize()
        for i in range(n):
            assert torch.equal(lh[i], refs[i][0]), i
            assert torch.equal(dxh[i], refs[i][1]), i
        assert torch.equal(layer.grads["dw_gate"], refs[-1][2])
    # a CUDA graph of the pipelined steps (copies and cross-stream events
    # recorded with the kernels) replays the same results
    replay = layer.capture(lambda: layer.train_steps_from_host(xh, p, gh, lh, dxh))
    for _ in range(2):
        for t in lh + dxh:
            t.zero_()
        replay()
        torch.cuda.synchronize()
        for i in range(n):
            assert torch.equal(lh[i], refs[i][0]), i
            assert torch.equal(dxh[i], refs[i][1]), i
    assert layer.device_status()[0] == 0


def test_captured_train_step_replays_the_eager_results():
    # a CUDA graph of the train step (and of the host-input step) gives the
    # eager step's results bit for bit on every replay
    cfg = MoEConfig(1500, 512, 1024, 4, 2, 1024, "bf16", "graph")
    inp = make_inputs(cfg)
    dev = to_dev(inp, "bf16")
    p = {k: dev[k] for k in params_of(inp)}
    from dropless_mixture_experts_gb300.layer import MoELayer
    layer = MoELayer(cfg.tokens, cfg.d_model, cfg.d_hidden, cfg.experts, cfg.top_k,
                     cfg.shared_hidden, "bf16", train=True)
    loss, dx, g = layer.train_step(dev["x"], p, dev["upstream"])
    torch.cuda.synchronize()
    ref = (loss.clone(), dx.clone(), {k: v.clone() for k, v in g.items() if v is not None})
    replay = layer.capture(lambda: layer.train_step(dev["x"], p, dev["upstream"]))
    xh = dev["x"].cpu().pin_memory()
    gh = dev["upstream"].cpu().pin_memory()
    lh = torch.empty(1, dtype=torch.float32).pin_memory()
    replay_host = layer.capture(lambda: layer.train_step_from_host(xh, p, gh, lh))
    for run in (replay, replay, replay_host):
        layer.loss.zero_()
        layer.dx.zero_()
        for v in layer.grads.values():
            if v is not None:
                v.zero_()
        run()
        torch.cuda.synchronize()
        assert torch.equal(layer.loss, ref[0])
        assert torch.equal(layer.dx, ref[1])
        for k, v in ref[2].items():
            assert torch.equal(layer.grads[k], v), k
    assert float(lh[0]) == float(ref[0][0])


# The shared expert on a side stream beside the routed experts (SM-capped
# persistent kernels on both streams): the same results, bit for bit, as the
# serial composition, in the train step, the forward pass and a CUDA-graph
# replay of the train step.
OVERLAP = [
    MoEConfig(2050, 256, 128, 64, 8, 256, "bf16", "overlap_decoder_small"),
    MoEConfig(1100, 512, 1024, 4, 2, 1024, "bf16", "overlap_pairs_shared"),
    MoEConfig(300, 64, 64, 5, 5, 64, "f32", "overlap_f32"),
]


@pytest.mark.parametrize("cfg", OVERLAP, ids=[c.name for c in OVERLAP])
def test_shared_expert_side_stream_matches_serial(cfg):
    from dropless_mixture_experts_gb300.layer import MoELayer
    inp = make_inputs(cfg)
    dev = to_dev(inp, cfg.dtype)
    p = {k: dev[k] for k in params_of(inp)}
    outs = []
    for shared_sms in (0, 40):
        layer = MoELayer(cfg.tokens, cfg.d_model, cfg.d_hidden, cfg.experts, cfg.top_k,
                         cfg.shared_hidden, cfg.dtype, train=True, shared_sms=shared_sms)
        loss, dx, g = layer.train_step(dev["x"], p, dev["upstream"])
        torch.cuda.synchronize()
        assert layer.device_status()[0] == 0
        res = {"loss": loss.clone(), "dx": dx.clone(), "y": layer.y.clone()}
        res.update({k: v.clone() for k, v in g.items() if v is not None})
        fwd = MoELayer(cfg.tokens, cfg.d_model, cfg.d_hidden, cfg.experts, cfg.top_k,
                       cfg.shared_hidden, cfg.dtype, train=False, shared_sms=shared_sms)
        res["y_fwd"] = fwd.forward(dev["x"], p).clone()
        if shared_sms:
            replay = layer.capture(lambda: layer.train_step(dev["x"], p, dev["upstream"]))
            layer.dx.zero_()
            for v in layer.grads.values():
                if v is not None:
                    v.zero_()
            replay()
            torch.cuda.synchronize()
            res["dx_graph"] = layer.dx.clone()
            res["dws_down_graph"] = layer.grads["dws_down"].clone()
        outs.append(res)
    serial, over = outs
    for k, v in serial.items():
        assert torch.equal(v, over[k]), k
    assert torch.equal(serial["dx"], over["dx_graph"])
    assert torch.equal(serial["dws_down"], over["dws_down_graph"])
    assert torch.equal(serial["y"], serial["y_fwd"])
