#!/usr/bin/env python
"""Throughput of the GB300 dropless MoE layer: one step = the train step
(route, permute, grouped SwiGLU experts, combine with the loss value, and the
full backward) over one batch of seeded synthetic tokens.

Prints ONE JSON line on rank 0.  ``--impl reference`` times the float64 CPU
oracle instead (a deliberately slow baseline on the host cores).

Multi-GPU (torchrun): every rank runs its own batch (independent problems,
weak scaling); the only collectives are the barrier and the max-over-ranks
timing reduction, outside the data path.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer tokens/s fwd and train step (bf16), % of dense BF16 tensor peak"
DEFAULT_CONFIG = "decoder_bf16_128k"
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--launch", default="graph", choices=["graph", "stream"],
                    help="graph: each timed step replays a CUDA graph of the whole step; "
                         "stream: the library's launches are issued one by one")
    ap.add_argument("--skew", type=float, default=0.0,
                    help="router bias ramp: skew * 4 logit std from expert 0 down to expert E-1")
    ap.add_argument("--capacity-factor", type=float, default=0.0,
                    help="capacity routing: each expert keeps ceil(F * T * k / E) pairs (0: dropless)")
    ap.add_argument("--also", default=None,
                    help="comma-separated further workloads measured in the same run and "
                         "reported under 'also' (default: e8k2_bf16_128k beside the default "
                         "workload, none otherwise)")
    ap.add_argument("--shared-sms", type=int, default=-1,
                    help="SMs of the side stream that runs the shared expert beside the routed "
                         "experts (0: one stream; default: 48 of 152, scaled to the device, "
                         "for workloads with a shared expert)")
    ap.add_argument("--sweep", default="", choices=["", "maxtok"],
                    help="maxtok: the largest train-step token count that fits in free HBM")
    return ap.parse_args()


def with_routing(cfg, args):
    """The workload with the command line's skew and capacity."""
    import dataclasses
    import math
    cap = 0
    if args.capacity_factor > 0:
        cap = math.ceil(args.capacity_factor * cfg.tokens * cfg.top_k / cfg.experts)
    return dataclasses.replace(cfg, skew=args.skew, capacity=cap)


# Kernel names of each piece of the pages' pieces suite (route, sort_permute,
# experts_grouped_swiglu, unpermute_combine); the rest of a train step is
# the backward.
PIECES = {
    "route": ("tc_router", "router_fused", "topk_softmax", "simt_logits"),
    "sort_permute": ("perm_hist", "perm_colscan", "perm_finalize", "perm_scatter", "zero_fill"),
    "experts": ("scatter_rows", "tc_gateup", "tc_gateup_sh", "tc_down", "tc_down_sh",
                "simt_gateup", "simt_gateup_sh", "simt_down", "simt_down_sh"),
    "combine": ("combine", "loss_reduce"),
}


def pieces_of(fwd_rec, train_rec, steps):
    """ms per step of each piece: the forward's pieces from a forward-only
    record, the backward as the train step's remainder."""
    def total(rec, names=None):
        return sum(t for n, (_, t) in rec.items() if names is None or n in names) / steps
    out = {k: total(fwd_rec, v) for k, v in PIECES.items()}
    out["forward_total"] = total(fwd_rec)
    out["backward"] = total(train_rec) - out["forward_total"]
    out["train_total"] = total(train_rec)
    return out


# ---------------------------------------------------------------------------
# algorithmic work per step
# ---------------------------------------------------------------------------
def step_flops(cfg, kept_frac=1.0):
    """Algorithmic FLOPs of one forward and one train step (router, routed
    and shared SwiGLU experts; the backward is twice the forward).  With
    capacity routing the routed experts count the kept pairs only."""
    T, d, h, E, k, hs = cfg.tokens, cfg.d_model, cfg.d_hidden, cfg.experts, cfg.top_k, cfg.shared_hidden
    fwd = T * (2 * d * E + kept_frac * k * 6 * d * h + 6 * d * hs)
    return fwd, 3 * fwd


# The pages' train-step times (ms) for the bf16 workloads: the RTX 3090 layer
# runs of kernel_gmm_gpu.json (pallas, dispatch sorted) and the H100 NVL
# decoder rows of gpu_moe_h100.json (pallas, sorted).  Another machine's
# numbers: context for the ratio, not a target.
PAGE_TRAIN_MS = {
    "e8k2_bf16_32k": (16.02, "RTX 3090, pallas sorted bf16, 32768 tokens (kernel_gmm_gpu.json)"),
    "e8k2_bf16_128k": (65.46, "RTX 3090, pallas sorted bf16, 131072 tokens (kernel_gmm_gpu.json)"),
    "e64k4_bf16_32k": (13.37, "RTX 3090, pallas sorted bf16, E64 k4 h256 (kernel_gmm_gpu.json)"),
    "decoder_bf16_16k": (2.628, "H100 NVL, pallas sorted, decoder 16384 tokens (gpu_moe_h100.json)"),
    "decoder_bf16_128k": (19.126, "H100 NVL, pallas sorted, decoder 131072 tokens (gpu_moe_h100.json)"),
}


def vs_page(cfg, value):
    """value / the pages' train-step tokens/s for the same workload (None
    without one; skewed or capacity routing has none)."""
    ent = PAGE_TRAIN_MS.get(cfg.name)
    if ent is None or cfg.skew or cfg.capacity:
        return None, None
    return value / (cfg.tokens / (ent[0] / 1e3)), ent[1]


def kernel_work(cfg, kept=None):
    """Algorithmic work per step of each kernel name: {"flop": f, "byte": b}.
    f = 2*M*N*K over real rows (routed launches count the kept pairs; the
    shared expert's launches carry the suffix _sh); b = every operand and
    result read or written once (real rows only, no padding rows, no
    split-K partials; weights once per launch).  The train step saves the
    pre-activations, so gate/up counts three [rows, h] outputs."""
    T, d, h, E, k, hs = cfg.tokens, cfg.d_model, cfg.d_hidden, cfg.experts, cfg.top_k, cfg.shared_hidden
    P = T * k if kept is None else kept
    el = 2 if cfg.dtype == "bf16" else 4
    w = {}
    router_b = T * d * el + d * E * el
    w["router"] = {"flop": 2 * T * d * E, "byte": router_b + T * k * 8}
    w["logits"] = {"flop": 2 * T * d * E, "byte": router_b + T * E * 4}
    # x and the dense bf16 logit gradient in, the f32 [d, E] gradient out
    w["router_dw"] = {"flop": 2 * T * d * E, "byte": T * d * el + T * E * el + d * E * 4}

    def ffn(tag, M, hh, n_w):
        # M rows through one SwiGLU expert stack of hidden hh (n_w weight sets)
        wb = d * hh * el * n_w  # one [d, hh] matrix per weight set
        w["gateup" + tag] = {"flop": 4 * M * d * hh,
                             "byte": M * d * el + 2 * wb + 3 * M * hh * el}
        w["down" + tag] = {"flop": 2 * M * d * hh, "byte": M * hh * el + wb + M * d * el}
        # the (gate-scaled) dy rows and the saved a_g, a_u in; dA [M, 2hh]
        # out (the float32 path also writes gate*H for its W_down gradient)
        n_out = 3 if cfg.dtype == "f32" else 2
        w["dz" + tag] = {"flop": 2 * M * d * hh,
                         "byte": M * d * el + wb + 2 * M * hh * el + n_out * M * hh * el}
        w["dx" + tag] = {"flop": 4 * M * d * hh, "byte": 2 * M * hh * el + 2 * wb + M * d * el}
        w["dw_down" + tag] = {"flop": 2 * M * d * hh,
                              "byte": M * hh * el + M * d * el + d * hh * 4 * n_w}
        w["dw_gateup" + tag] = {"flop": 4 * M * d * hh,
                                "byte": M * d * el + 2 * M * hh * el + 2 * d * hh * 4 * n_w}

    ffn("", P, h, E)
    if hs:
        ffn("_sh", T, hs, 1)
    shared_rows = T if hs else 0
    # x -> xs and dy -> dys: each token row read once, written to its k rows
    w["scatter_rows"] = {"flop": 0, "byte": 2 * (T + P) * d * el}
    # pair rows + shared rows + upstream read, y written
    w["combine"] = {"flop": 0, "byte": (P + shared_rows + T + T) * d * el}
    # pair rows + shared rows read, dx written
    w["router_dx"] = {"flop": 0, "byte": (P + shared_rows + T) * d * el}
    return w


def kernel_bound(name, wk, peaks):
    """The roofline a kernel sits under: the larger of its time at the
    compute peak (bf16 tensor, or FP32 FFMA for the SIMT kernels) and its
    time at the HBM peak.  Returns (bound, compute peak TFLOP/s, hbm GB/s)."""
    hbm = float(peaks.get("hbm_gbs", 6800.0))
    if name.startswith("simt_"):
        # FP32 FFMA: 152 SMs x 128 lanes x 2 flop x max SM clock
        comp, cb = 152 * 128 * 2 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12, "alu"
    else:
        comp, cb = float(peaks.get("bf16_tflops", 1900.0)), "tensor"
    t_c = wk["flop"] / (comp * 1e12)
    t_m = wk["byte"] / (hbm * 1e9)
    return (cb if t_c >= t_m else "hbm"), comp, hbm


def code_text(text):
    """CUDA/C++ source with comments and blank space removed (what a
    compiler sees); string literals are kept as they are."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':  # a string literal, escapes included
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


# The strict-float32 GEMMs: no bf16 step launches code from this file.
FP32_ONLY_SOURCES = ("gemm_simt.cu",)


def src_hash(csrc=None):
    """Hash of the CUDA sources' code (comments and blank space ignored): the
    key under which per-launch DRAM traffic counters stay valid.  Every
    counter kept is of a bf16 train step's launch, so the strict-float32
    GEMMs' file, which no bf16 step runs, is left out."""
    h = hashlib.sha256()
    csrc = csrc or os.path.join(ROOT, "dropless_mixture_experts_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")) and f not in FP32_ONLY_SOURCES:
            h.update(f.encode())
            h.update(code_text(open(os.path.join(csrc, f), encoding="utf-8").read()).encode())
    return h.hexdigest()[:16]


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


class ClockSampler:
    def __init__(self, index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.p = subprocess.Popen(
                ["nvidia-smi", f"--id={index}", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None
        self.t0 = self.t1 = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()

    def finish(self):
        if self.p is None:
            return None
        time.sleep(0.25)
        self.p.terminate()
        self.p.wait()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.f.name)
        sms, mx, reasons = [], None, set()
        for r in rows:
            r = [c.strip() for c in r]
            try:
                ts = time.mktime(time.strptime(r[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
            except Exception:
                ts = None
            if ts is not None and self.t0 is not None and not (self.t0 - 1.5 <= ts <= self.t1 + 1.0):
                continue
            try:
                sms.append(float(r[2]))
                mx = float(r[3])
            except ValueError:
                continue
            for name, v in zip(REASONS, r[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sms)}


# ---------------------------------------------------------------------------
# CPU oracle timing (baseline / reference arm)
# ---------------------------------------------------------------------------
def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count()


def oracle_tokens_per_s(cfg, inputs, target_s=10.0, max_tokens=None):
    """Times the oracle train step (as it stands) on the first S tokens of
    the workload, S grown until one run takes about target_s."""
    import oracle
    from dropless_mixture_experts_gb300.synthetic import params_of

    p = params_of(inputs)
    S = min(cfg.tokens, 1024)
    cap = cfg.tokens if max_tokens is None else min(cfg.tokens, max_tokens)
    while True:
        # capacity scales with the sample: the same share of each expert kept
        c_s = -(-cfg.capacity * S // cfg.tokens) if cfg.capacity else None
        t0 = time.perf_counter()
        oracle.train_step(inputs["x"][:S], p, cfg.top_k, inputs["upstream"][:S], capacity=c_s)
        dt = time.perf_counter() - t0
        if dt >= target_s * 0.5 or S >= cap:
            return S / dt, S, dt
        S = min(cap, int(S * max(2.0, target_s / max(dt, 1e-3) * 0.8)))


# ---------------------------------------------------------------------------
# ranks (torchrun): independent batches, the job's time is its slowest rank's
# ---------------------------------------------------------------------------
def rank_info():
    """(world size, rank, local rank) from the launcher's environment."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed_offset(rank):
    """Each rank draws its own batch (and weights) from the seeded generator."""
    return 100 * rank


def max_over_ranks(values, device):
    """Each value's maximum over the ranks of the process group (times: the
    job waits for its slowest rank); the values themselves without one."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def job_tokens_per_s(world, tokens, seconds):
    """Whole-job throughput: every rank processes its own batch of `tokens`,
    the job takes the slowest rank's `seconds` (weak scaling)."""
    return world * tokens / seconds


def reference_arm(args, cfg):
    _, rank, _ = rank_info()
    if rank != 0:  # rank 0 alone times the oracle; the others leave without work
        return
    from dropless_mixture_experts_gb300.synthetic import make_inputs, params_of
    import oracle

    inputs = make_inputs(cfg)
    p = params_of(inputs)
    S = min(cfg.tokens, 1024)
    c_s = -(-cfg.capacity * S // cfg.tokens) if cfg.capacity else None  # same kept share
    for _ in range(args.warmup):
        oracle.train_step(inputs["x"][:S], p, cfg.top_k, inputs["upstream"][:S], capacity=c_s)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.train_step(inputs["x"][:S], p, cfg.top_k, inputs["upstream"][:S], capacity=c_s)
        times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    v = S / (ms / 1e3)
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": cfg.name, "tokens": cfg.tokens, "d_model": cfg.d_model,
                   "d_hidden": cfg.d_hidden, "experts": cfg.experts, "top_k": cfg.top_k,
                   "shared_hidden": cfg.shared_hidden, "storage": cfg.dtype,
                   "routing": {"skew": cfg.skew, "capacity": cfg.capacity}},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": f"train step on the first {S} of {cfg.tokens} tokens per step"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# maximum tokens of one train step (the pages' maxtok suite)
# ---------------------------------------------------------------------------
def layer_device_bytes(cfg, tokens):
    """Device bytes of one train-step invocation at ``tokens``: the layer's
    buffers and workspace as the library sizes them (counted on torch's meta
    device, nothing allocated), the token inputs, the weights and their
    gradients' inputs."""
    import torch
    from dropless_mixture_experts_gb300.layer import MoELayer
    L = MoELayer(tokens, cfg.d_model, cfg.d_hidden, cfg.experts, cfg.top_k, cfg.shared_hidden,
                 cfg.dtype, device="meta", train=True, capacity=cfg.capacity)
    b = 0
    for v in vars(L).values():
        if isinstance(v, torch.Tensor):
            b += v.nbytes
        elif isinstance(v, dict):
            b += sum(x.nbytes for x in v.values() if isinstance(x, torch.Tensor))
    el = 2 if cfg.dtype == "bf16" else 4
    d, h, E, hs = cfg.d_model, cfg.d_hidden, cfg.experts, cfg.shared_hidden
    b += 2 * tokens * d * el                        # x and the upstream gradient
    b += (d * E + 3 * E * d * h + 3 * d * hs) * el  # weights
    return b


def maxtok_sweep(args, cfg):
    """Largest train-step token count that fits in the free HBM of this GPU,
    by the library's own sizes (a doubling then bisection search on
    ``layer_device_bytes``), bounded by the C ABI's index range; then one
    real train step at that size is run and timed to show it fits."""
    import dataclasses
    import torch
    from dropless_mixture_experts_gb300 import abi
    from dropless_mixture_experts_gb300.layer import MoELayer

    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    abi.load()
    free, total = torch.cuda.mem_get_info()
    budget = int(free * 0.92)  # room for the allocator's rounding and the context

    def abi_ok(T):
        return T <= (1 << 31) // 64 and T * cfg.top_k + cfg.experts * 256 < (1 << 31)

    def fits(T):
        return abi_ok(T) and layer_device_bytes(cfg, T) <= budget

    lo = 1024
    hi = lo
    while fits(hi * 2):
        hi *= 2
    lo, hi = hi, hi * 2
    while hi - lo > 1024:
        mid = (lo + hi) // 2 // 1024 * 1024
        lo, hi = (mid, hi) if fits(mid) else (lo, mid)
    T = lo
    binding = "memory" if abi_ok(hi) else "index range"

    # one real step at that size, inputs drawn on the device (seeded)
    td = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    d, h, E, hs = cfg.d_model, cfg.d_hidden, cfg.experts, cfg.shared_hidden
    g = torch.Generator(device="cuda")

    def normal(seed, shape, std):
        g.manual_seed(seed)
        return (torch.randn(shape, generator=g, device="cuda", dtype=torch.float32) * std).to(td)

    p = {"w_router": normal(1, (d, E), d ** -0.5), "w_gate": normal(2, (E, d, h), d ** -0.5),
         "w_up": normal(3, (E, d, h), d ** -0.5), "w_down": normal(4, (E, h, d), h ** -0.5),
         "ws_gate": None, "ws_up": None, "ws_down": None}
    if hs:
        p.update(ws_gate=normal(5, (d, hs), d ** -0.5), ws_up=normal(6, (d, hs), d ** -0.5),
                 ws_down=normal(7, (hs, d), hs ** -0.5))
    x = normal(0, (T, d), 1.0)
    G = normal(8, (T, d), 1.0)
    layer = MoELayer(T, d, h, E, cfg.top_k, hs, cfg.dtype, train=True, capacity=cfg.capacity)
    for _ in range(2):
        layer.train_step(x, p, G)
    torch.cuda.synchronize()
    st, _ = layer.device_status()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(3)]
    for a, b in evs:
        a.record()
        layer.train_step(x, p, G)
        b.record()
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    line = {
        "metric": "max train-step tokens in HBM", "value": T, "unit": "tokens", "n_gpus": 1,
        "higher_is_better": True, "dtype": "bf16" if cfg.dtype == "bf16" else "f32",
        "data": "synthetic (drawn on the device)",
        "config": {"workload": cfg.name, "d_model": d, "d_hidden": h, "experts": E,
                   "top_k": cfg.top_k, "shared_hidden": hs, "step": "train (value_and_grad)"},
        "binding": binding, "device_bytes": layer_device_bytes(cfg, T),
        # the pages' maxtok rows give peak MB per doubling of the tokens
        "ladder_mb": {str(t): layer_device_bytes(cfg, t) / 2 ** 20
                      for t in (131072 << i for i in range(12)) if t <= T},
        "bytes_per_token": layer_device_bytes(cfg, T) / T, "free_bytes": free,
        "total_bytes": total, "peak_allocated": torch.cuda.max_memory_allocated(),
        "device_status": st, "ms_per_step": ms, "tokens_per_s": T / (ms / 1e3),
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
NOMINAL_BF16_TFLOPS = 2250.0  # GB300 dense bf16 tensor peak (NVIDIA's published, no sparsity)


def also_default(name):
    """The second 131072-token bf16 workload reported beside the default one."""
    return "e8k2_bf16_128k" if name == DEFAULT_CONFIG else ""


def shared_sms_of(cfg, args):
    """SMs of the shared expert's side stream: the command line's, else 48 of
    152 (the best of a sweep at the decoder workloads), scaled to the
    device; 0 without a shared expert."""
    import torch
    if not cfg.shared_hidden:
        return 0
    if args.shared_sms >= 0:
        return args.shared_sms
    n = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return max(1, round(n * 48 / 152))


def measure(cfg, args, world, rank, local, barrier, peaks, cpu_baseline):
    """Times one workload: the train step and the forward (graph replays by
    default), the end-to-end host-input step, and the per-kernel split.
    Returns the bench line's fields for it (rank 0 prints them)."""
    import torch

    from dropless_mixture_experts_gb300 import abi
    from dropless_mixture_experts_gb300.layer import MoELayer
    from dropless_mixture_experts_gb300.synthetic import make_inputs, params_of

    td = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    inputs = make_inputs(cfg, seed_offset=rank_seed_offset(rank))
    host = {k: (None if v is None else
                torch.from_numpy(v).to(torch.float32 if k == "router_bias" else td).pin_memory())
            for k, v in inputs.items()}
    dev = {k: (None if v is None else v.to("cuda", non_blocking=True)) for k, v in host.items()}
    p = {k: dev[k] for k in params_of(inputs)}
    shared_sms = shared_sms_of(cfg, args)
    layer = MoELayer(cfg.tokens, cfg.d_model, cfg.d_hidden, cfg.experts, cfg.top_k,
                     cfg.shared_hidden, cfg.dtype, train=True, capacity=cfg.capacity,
                     shared_sms=shared_sms)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()

    def train():
        layer.train_step(dev["x"], p, dev["upstream"])

    def fwd():
        layer.forward(dev["x"], p)

    def timed(fn, K):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        for a, b in evs:
            flush.zero_()
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    for _ in range(args.warmup):
        train()
        fwd()
    torch.cuda.synchronize()
    st, _ = layer.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} after warm-up")
    # routing statistics as the pages record them, and the pairs kept
    per_expert = torch.bincount(layer.idx.reshape(-1).long(), minlength=cfg.experts).cpu()
    P = cfg.tokens * cfg.top_k
    kept = int(layer.counts.sum().item())
    routing = {"skew": cfg.skew, "max_expert_frac": float(per_expert.max()) / P,
               "empty_experts": int((per_expert == 0).sum()), "capacity": cfg.capacity,
               "kept_pairs_frac": kept / P}

    run_train, run_fwd = train, fwd
    if args.launch == "graph":
        # the same passes recorded once; each timed step replays all of it
        run_train, run_fwd = layer.capture(train), layer.capture(fwd)
        for _ in range(args.warmup):
            run_train()
            run_fwd()
        torch.cuda.synchronize()

    clocks = ClockSampler(local)
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    clocks.mark_start()
    train_ms = timed(run_train, args.steps)
    torch.cuda.synchronize()
    barrier()
    clocks.mark_stop()
    fwd_ms = timed(run_fwd, args.steps)
    clk = clocks.finish()

    ms = statistics.mean(train_ms)
    fms = statistics.mean(fwd_ms)
    ms, fms = max_over_ranks([ms, fms], "cuda")
    value = job_tokens_per_s(world, cfg.tokens, ms / 1e3)
    fwd_value = job_tokens_per_s(world, cfg.tokens, fms / 1e3)

    # end to end through the public API with host buffers: every step's H2D
    # of its batch (x and the upstream gradient) and D2H of its value and of
    # the input gradient dx, in a pipelined sequence of steps (the copies of
    # step i + 1's inputs and step i - 1's results run while step i computes);
    # the weight gradients stay on the device for an optimizer step
    loss_h = [torch.empty(1, dtype=torch.float32).pin_memory() for _ in range(2)]
    dx_h = [torch.empty(cfg.tokens, cfg.d_model, dtype=td).pin_memory() for _ in range(2)]
    n_e2e = max(4, args.steps)

    def e2e_steps(n):
        layer.train_steps_from_host([host["x"]] * n, p, [host["upstream"]] * n,
                                    [loss_h[i % 2] for i in range(n)],
                                    [dx_h[i % 2] for i in range(n)])

    e2e_steps(2)  # first-call setup
    # one pipelined sequence of all the timed steps, as a training loop runs
    # them (the first step's input copy and the last step's result copy are
    # the only ones not hidden behind a step); graph mode: the sequence
    # captured as one CUDA graph and replayed (the copies and the
    # cross-stream events record into it like the kernels)
    per_run = n_e2e
    runs = 1
    run_steps = layer.capture(lambda: e2e_steps(per_run)) if args.launch == "graph" else \
        (lambda: e2e_steps(per_run))
    torch.cuda.synchronize()
    e2e_times = []
    for _ in range(3):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(runs):
            run_steps()
        torch.cuda.synchronize()
        e2e_times.append((time.perf_counter() - t0) / (runs * per_run))
    e2e_s = statistics.median(e2e_times)
    h2d = host["x"].numel() * host["x"].element_size() * 2
    d2h = loss_h[0].numel() * loss_h[0].element_size() + dx_h[0].numel() * dx_h[0].element_size()
    (e2e_s,) = max_over_ranks([e2e_s], "cuda")
    e2e = {"value": job_tokens_per_s(world, cfg.tokens, e2e_s), "unit": "tokens/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "copies": "per step: H2D x and the upstream gradient, D2H the value and dx",
           "steps": f"{runs * per_run} steps of train_steps_from_host per timing, pipelined "
                    f"in runs of {per_run}" + (" (each run a replayed CUDA graph)"
                                               if args.launch == "graph" else "") +
                    "; each step's working set is larger than L2"}

    # per-kernel device time and launch count of the forward and of the step
    # (stream launches with an event pair around each launch: a little
    # slower than the graph-replayed step, so each fraction is a lower bound;
    # every kernel on one stream, so that each is timed alone)
    layer.shared_sms = 0
    prof_steps = 3
    abi.moe_profile_enable(True)
    for _ in range(prof_steps):
        flush.zero_()
        fwd()
    fwd_rec = abi.moe_profile_read()
    abi.moe_profile_enable(False)
    abi.moe_profile_enable(True)
    for _ in range(prof_steps):
        flush.zero_()
        train()
    rec = abi.moe_profile_read()
    abi.moe_profile_enable(False)
    layer.shared_sms = shared_sms
    pieces = pieces_of(fwd_rec, rec, prof_steps)
    launches_per_step = sum(n for n, _ in rec.values()) / prof_steps
    work = kernel_work(cfg, kept)

    # the dominant kernel with a known algorithmic amount of work, under
    # whichever of its compute and HBM rooflines is the binding one
    def work_of(name):
        return work.get(name.split("_", 1)[1] if name.startswith(("tc_", "simt_")) else name)
    known = [kv for kv in rec.items() if work_of(kv[0])]
    tname, (tn, tms) = max(known, key=lambda kv: kv[1][1])
    wk = work_of(tname)
    bound, comp_peak, hbm_peak = kernel_bound(tname, wk, peaks)
    secs = tms / prof_steps / 1e3
    if bound == "hbm":
        achieved, peak, runit = wk["byte"] / secs / 1e9 if secs > 0 else 0.0, hbm_peak, "GB/s"
    else:
        achieved, peak, runit = wk["flop"] / secs / 1e12 if secs > 0 else 0.0, comp_peak, "TFLOP/s"
    traffic = None
    try:
        tr = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
        ent = tr.get(cfg.name, {}).get(tname)
        if ent and ent.get("src_sha") == src_hash():
            traffic = ent["bytes_per_launch"]
    except Exception:
        pass
    roofline = {"bound": bound, "achieved": achieved, "peak": peak, "unit": runit,
                "frac": achieved / peak if peak else None, "traffic": traffic,
                "kernel": tname, "launch_ms": tms / tn,
                "algorithmic": {"flop": wk["flop"], "byte": wk["byte"]},
                "peak_source": {"tensor": "measured bf16 burst", "hbm": "measured HBM copy",
                                "alu": "derived: 152 SMs x 128 FP32 lanes x 2 x max SM clock"}[bound]}
    kernels = {}
    for k_, (n, t) in sorted(rec.items(), key=lambda kv: -kv[1][1]):
        ent = {"launches_per_step": n / prof_steps, "ms_per_step": t / prof_steps}
        wk = work_of(k_)
        if wk and t > 0:
            secs = t / prof_steps / 1e3
            bnd, comp_peak, hbm_peak = kernel_bound(k_, wk, peaks)
            ent["bound"] = bnd
            if wk["flop"]:
                ent["tflops"] = wk["flop"] / secs / 1e12
                ent["frac_" + ("alu" if k_.startswith("simt_") else "bf16")] = ent["tflops"] / comp_peak
            ent["gbs"] = wk["byte"] / secs / 1e9
            ent["frac_hbm"] = ent["gbs"] / hbm_peak
        kernels[k_] = ent

    f_fwd, f_train = step_flops(cfg, kept / P)
    measured_bf16 = float(peaks.get("bf16_tflops", 1900.0))
    cpu = None
    if cpu_baseline and rank == 0 and world == 1:
        v, S, dt = oracle_tokens_per_s(cfg, inputs)
        cpu = {"value": v, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
               "sample": f"float64 train step on the first {S} of {cfg.tokens} tokens ({dt:.1f} s)"}
    out = {
        "value": value, "ms_per_step": ms, "fwd_tokens_per_s": fwd_value, "fwd_ms": fms,
        "config": {"workload": cfg.name, "tokens": cfg.tokens, "d_model": cfg.d_model,
                   "d_hidden": cfg.d_hidden, "experts": cfg.experts, "top_k": cfg.top_k,
                   "shared_hidden": cfg.shared_hidden, "step": "train (value_and_grad)",
                   "routing": routing,
                   "l2": "flushed between timed steps (256 MiB write)",
                   "launch": ("a CUDA graph of the whole step, replayed per step"
                              if args.launch == "graph" else "stream launches"),
                   "shared_expert_stream": (f"side stream, {shared_sms} SMs" if shared_sms
                                            else "same stream"),
                   "kernel_timing": ("pieces_ms, kernels and roofline: a separate pass of "
                                     "stream launches on one stream with an event pair "
                                     "around each launch"),
                   "parallelism": f"independent batch per GPU x{world}"},
        # the dense bf16 tensor peak of the part, and the measured cuBLAS
        # matmul rate (the roofline denominator) beside it
        "pct_bf16_peak": {"train": f_train / (ms / 1e3) / 1e12 / NOMINAL_BF16_TFLOPS,
                          "fwd": f_fwd / (fms / 1e3) / 1e12 / NOMINAL_BF16_TFLOPS,
                          "peak_tflops": NOMINAL_BF16_TFLOPS,
                          "peak_source": "GB300 dense bf16 tensor peak, published (2.25 PFLOP/s)"},
        "pct_of_measured_matmul": {"train": f_train / (ms / 1e3) / 1e12 / measured_bf16,
                                   "fwd": f_fwd / (fms / 1e3) / 1e12 / measured_bf16,
                                   "peak_tflops": measured_bf16,
                                   "peak_source": "measured bf16 matmul burst"},
        "clocks": clk, "e2e": e2e, "gpu_launches": int(round(launches_per_step * args.steps)),
        "roofline": roofline, "cpu_baseline": cpu, "pieces_ms": pieces, "kernels": kernels,
    }
    del layer, dev, host, flush
    torch.cuda.empty_cache()
    return out


def main():
    args = parse()
    from dropless_mixture_experts_gb300.synthetic import CONFIGS

    cfg = with_routing(CONFIGS[args.config], args)
    if args.impl == "reference":
        reference_arm(args, cfg)
        return
    if args.sweep == "maxtok":
        maxtok_sweep(args, cfg)
        return

    import torch
    import torch.distributed as dist

    from dropless_mixture_experts_gb300 import abi

    world, rank, local = rank_info()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")

    def barrier():
        if world > 1:
            dist.barrier()

    abi.load()
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        pass
    main_res = measure(cfg, args, world, rank, local, barrier, peaks, not args.no_cpu_baseline)
    also = {}
    also_name = args.also if args.also is not None else also_default(args.config)
    for name in [n for n in also_name.split(",") if n]:
        r = measure(with_routing(CONFIGS[name], args), args, world, rank, local, barrier, peaks,
                    False)
        also[name] = {k: r[k] for k in ("value", "ms_per_step", "fwd_tokens_per_s", "fwd_ms",
                                        "pct_bf16_peak", "pct_of_measured_matmul", "roofline",
                                        "e2e", "clocks", "pieces_ms", "kernels")}

    if rank == 0:
        vs, vs_basis = vs_page(cfg, main_res["value"])
        line = {
            "metric": METRIC, "value": main_res["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": main_res["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": vs,
            "vs_baseline_basis": vs_basis,
            "dtype": "bf16" if cfg.dtype == "bf16" else "f32",
            "data": "synthetic",
        }
        line.update({k: v for k, v in main_res.items() if k not in line})
        if also:
            line["also"] = also
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
