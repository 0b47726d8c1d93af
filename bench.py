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
DEFAULT_CONFIG = "e8k2_bf16_32k"
L2_BYTES = 129 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# algorithmic work per step
# ---------------------------------------------------------------------------
def step_flops(cfg):
    """Algorithmic FLOPs of one forward and one train step (router, routed
    and shared SwiGLU experts; the backward is twice the forward)."""
    T, d, h, E, k, hs = cfg.tokens, cfg.d_model, cfg.d_hidden, cfg.experts, cfg.top_k, cfg.shared_hidden
    fwd = T * (2 * d * E + k * 6 * d * h + 6 * d * hs)
    return fwd, 3 * fwd


def kernel_work(cfg):
    """Algorithmic work per step of each kernel name: ("flop", n) for the
    contractions (2*M*N*K over real rows; the routed experts' launches, and
    the shared expert's with suffix _sh), ("byte", n) for the row streams
    (each row read or written once)."""
    T, d, h, E, k, hs = cfg.tokens, cfg.d_model, cfg.d_hidden, cfg.experts, cfg.top_k, cfg.shared_hidden
    P = T * k
    el = 2 if cfg.dtype == "bf16" else 4
    w = {"logits": ("flop", 2 * T * d * E), "router": ("flop", 2 * T * d * E),
         "router_dw": ("flop", 2 * T * d * E)}
    for name, n in (("gateup", 2), ("down", 1), ("dz", 1), ("dx", 2), ("dw_down", 1),
                    ("dw_gateup", 2)):
        w[name] = ("flop", 2 * P * d * h * n)
        if hs:
            w[name + "_sh"] = ("flop", 2 * T * d * hs * n)
    shared_rows = T if hs else 0
    # x -> xs and dy -> dys: each token row read once, written to its k rows
    w["scatter_rows"] = ("byte", 2 * (T + P) * d * el)
    # pair rows + shared rows + upstream read, y written
    w["combine"] = ("byte", (P + shared_rows + T + T) * d * el)
    # pair rows + shared rows read, dx written
    w["router_dx"] = ("byte", (P + shared_rows + T) * d * el)
    return w


def src_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dropless_mixture_experts_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh")):
            h.update(open(os.path.join(csrc, f), "rb").read())
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
        t0 = time.perf_counter()
        oracle.train_step(inputs["x"][:S], p, cfg.top_k, inputs["upstream"][:S])
        dt = time.perf_counter() - t0
        if dt >= target_s * 0.5 or S >= cap:
            return S / dt, S, dt
        S = min(cap, int(S * max(2.0, target_s / max(dt, 1e-3) * 0.8)))


def reference_arm(args, cfg):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from dropless_mixture_experts_gb300.synthetic import make_inputs, params_of
    import oracle

    inputs = make_inputs(cfg)
    p = params_of(inputs)
    S = min(cfg.tokens, 1024)
    for _ in range(args.warmup):
        oracle.train_step(inputs["x"][:S], p, cfg.top_k, inputs["upstream"][:S])
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.train_step(inputs["x"][:S], p, cfg.top_k, inputs["upstream"][:S])
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
                   "shared_hidden": cfg.shared_hidden, "storage": cfg.dtype},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
                         "sample": f"train step on the first {S} of {cfg.tokens} tokens per step"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def main():
    args = parse()
    from dropless_mixture_experts_gb300.synthetic import CONFIGS

    cfg = CONFIGS[args.config]
    if args.impl == "reference":
        reference_arm(args, cfg)
        return

    import numpy as np
    import torch
    import torch.distributed as dist

    from dropless_mixture_experts_gb300 import abi
    from dropless_mixture_experts_gb300.layer import MoELayer
    from dropless_mixture_experts_gb300.synthetic import make_inputs, params_of

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")

    def barrier():
        if world > 1:
            dist.barrier()

    abi.load()
    td = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    inputs = make_inputs(cfg, seed_offset=100 * rank)
    host = {k: (None if v is None else
                torch.from_numpy(v).to(torch.float32 if k == "router_bias" else td).pin_memory())
            for k, v in inputs.items()}
    dev = {k: (None if v is None else v.to("cuda", non_blocking=True)) for k, v in host.items()}
    p = {k: dev[k] for k in params_of(inputs)}
    layer = MoELayer(cfg.tokens, cfg.d_model, cfg.d_hidden, cfg.experts, cfg.top_k,
                     cfg.shared_hidden, cfg.dtype, train=True)
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

    clocks = ClockSampler(local)
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    clocks.mark_start()
    train_ms = timed(train, args.steps)
    torch.cuda.synchronize()
    barrier()
    clocks.mark_stop()
    fwd_ms = timed(fwd, args.steps)
    clk = clocks.finish()

    ms = statistics.mean(train_ms)
    fms = statistics.mean(fwd_ms)
    if world > 1:
        t = torch.tensor([ms, fms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms, fms = float(t[0]), float(t[1])
    value = world * cfg.tokens / (ms / 1e3)
    fwd_value = world * cfg.tokens / (fms / 1e3)

    # end to end through the public API with host buffers: H2D of the batch
    # (x and the upstream gradient) and D2H of the loss inside the timed region
    loss_host = torch.empty(1, dtype=torch.float32).pin_memory()
    e2e_times = []
    for _ in range(max(3, args.steps // 2)):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        dev["x"].copy_(host["x"], non_blocking=True)
        dev["upstream"].copy_(host["upstream"], non_blocking=True)
        loss, _, _ = layer.train_step(dev["x"], p, dev["upstream"])
        loss_host.copy_(loss, non_blocking=True)
        torch.cuda.synchronize()
        e2e_times.append(time.perf_counter() - t0)
    e2e_s = statistics.median(e2e_times)
    h2d = host["x"].numel() * host["x"].element_size() * 2
    e2e = {"value": world * cfg.tokens / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": 4}

    # per-kernel device time and launch count of the step
    abi.moe_profile_enable(True)
    prof_steps = 3
    for _ in range(prof_steps):
        flush.zero_()
        train()
    rec = abi.moe_profile_read()
    abi.moe_profile_enable(False)
    launches_per_step = sum(n for n, _ in rec.values()) / prof_steps
    work = kernel_work(cfg)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        pass
    # the dominant kernel with a known algorithmic amount of work
    def work_of(name):
        return work.get(name.split("_", 1)[1] if name.startswith(("tc_", "simt_")) else name)
    known = [kv for kv in rec.items() if work_of(kv[0])]
    tname, (tn, tms) = max(known, key=lambda kv: kv[1][1])
    unit, amount = work_of(tname)
    amount *= prof_steps
    alu = tname.startswith("simt_")
    if unit == "byte":
        achieved = amount / (tms / 1e3) / 1e9 if tms > 0 else 0.0
        peak = float(peaks.get("hbm_gbs", 6800.0))
        bound, runit = "hbm", "GB/s"
    elif alu:
        achieved = amount / (tms / 1e3) / 1e12 if tms > 0 else 0.0
        # FP32 FFMA: 152 SMs x 128 lanes x 2 flop x max SM clock
        peak = 152 * 128 * 2 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12
        bound, runit = "alu", "TFLOP/s"
    else:
        achieved = amount / (tms / 1e3) / 1e12 if tms > 0 else 0.0
        peak = float(peaks.get("bf16_tflops", 1900.0))
        bound, runit = "tensor", "TFLOP/s"
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
                "peak_source": {"tensor": "measured bf16 burst", "hbm": "measured HBM copy",
                                "alu": "derived: 152 SMs x 128 FP32 lanes x 2 x max SM clock"}[bound]}
    kernels = {}
    for k_, (n, t) in sorted(rec.items(), key=lambda kv: -kv[1][1]):
        ent = {"launches_per_step": n / prof_steps, "ms_per_step": t / prof_steps}
        wk = work_of(k_)
        if wk and t > 0:
            u, a = wk
            if u == "byte":
                ent["gbs"] = a / (t / prof_steps / 1e3) / 1e9
                ent["frac_hbm"] = ent["gbs"] / float(peaks.get("hbm_gbs", 6800.0))
            elif not k_.startswith("simt_"):
                ent["tflops"] = a / (t / prof_steps / 1e3) / 1e12
                ent["frac_bf16"] = ent["tflops"] / float(peaks.get("bf16_tflops", 1900.0))
        kernels[k_] = ent

    f_fwd, f_train = step_flops(cfg)
    bf16_peak = float(peaks.get("bf16_tflops", 1900.0))
    cpu = None
    if rank == 0 and not args.no_cpu_baseline and world == 1:
        v, S, dt = oracle_tokens_per_s(cfg, inputs)
        cpu = {"value": v, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
               "sample": f"float64 train step on the first {S} of {cfg.tokens} tokens ({dt:.1f} s)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if cfg.dtype == "bf16" else "f32",
            "data": "synthetic",
            "config": {"workload": cfg.name, "tokens": cfg.tokens, "d_model": cfg.d_model,
                       "d_hidden": cfg.d_hidden, "experts": cfg.experts, "top_k": cfg.top_k,
                       "shared_hidden": cfg.shared_hidden, "step": "train (value_and_grad)",
                       "l2": "flushed between timed steps (256 MiB write)",
                       "parallelism": f"independent batch per GPU x{world}"},
            "fwd_tokens_per_s": fwd_value, "fwd_ms": fms,
            "pct_bf16_peak": {"train": f_train / (ms / 1e3) / 1e12 / bf16_peak,
                              "fwd": f_fwd / (fms / 1e3) / 1e12 / bf16_peak},
            "clocks": clk, "e2e": e2e, "gpu_launches": int(round(launches_per_step * args.steps)),
            "roofline": roofline, "cpu_baseline": cpu, "kernels": kernels,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
