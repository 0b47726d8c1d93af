"""Host-side accounting of bench.py: the per-kernel algorithmic work adds
up to the layer's FLOP count, and each kernel's roofline is the binding one."""

import bench
from dropless_mixture_experts_gb300.synthetic import CONFIGS

PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "sm_max_mhz": 2070.0}


def test_kernel_flops_add_up_to_the_train_step():
    for name, cfg in CONFIGS.items():
        w = bench.kernel_work(cfg)
        gemm = sum(v["flop"] for k, v in w.items() if k not in ("router", "logits", "router_dw"))
        # the router's three contractions: x W_r, x^T dl, and dl W_r^T (inside router_dx)
        router = 3 * w["router"]["flop"]
        _, train = bench.step_flops(cfg)
        assert gemm + router == train, name


def test_capacity_counts_kept_pairs_only():
    cfg = CONFIGS["e8k2_bf16_32k"]
    full = bench.kernel_work(cfg)
    half = bench.kernel_work(cfg, kept=cfg.tokens * cfg.top_k // 2)
    assert half["gateup"]["flop"] * 2 == full["gateup"]["flop"]
    assert half["router"] == full["router"]


def test_binding_roofline():
    w = bench.kernel_work(CONFIGS["e8k2_bf16_32k"])
    # h = 1024: the saved-activation traffic of dZ outweighs its FLOPs
    assert bench.kernel_bound("tc_dz", w["dz"], PEAKS)[0] == "hbm"
    assert bench.kernel_bound("tc_gateup", w["gateup"], PEAKS)[0] == "tensor"
    assert bench.kernel_bound("tc_router", w["router"], PEAKS)[0] == "hbm"
    assert bench.kernel_bound("combine", w["combine"], PEAKS)[0] == "hbm"
    assert bench.kernel_bound("simt_gateup", w["gateup"], PEAKS)[0] == "alu"
    # fine-grained experts (h = 128): every routed GEMM is HBM-bound
    wd = bench.kernel_work(CONFIGS["decoder_bf16_128k"])
    for k in ("gateup", "down", "dz", "dx", "dw_down", "dw_gateup"):
        assert bench.kernel_bound("tc_" + k, wd[k], PEAKS)[0] == "hbm", k


def test_vs_baseline_uses_the_pages_train_time_for_the_same_workload():
    cfg = CONFIGS["e8k2_bf16_32k"]
    v, basis = bench.vs_page(cfg, 32768 / 16.02e-3)  # the page's own tokens/s
    assert abs(v - 1.0) < 1e-12 and "RTX 3090" in basis
    # no page number: float32 workloads, skewed or capacity routing
    assert bench.vs_page(CONFIGS["e8k2_f32_4k"], 1.0) == (None, None)
    import dataclasses
    assert bench.vs_page(dataclasses.replace(cfg, skew=0.9), 1.0) == (None, None)
    assert bench.vs_page(dataclasses.replace(cfg, capacity=100), 1.0) == (None, None)


def test_traffic_key_ignores_comments_only():
    a = 'int f() { return 1; } // note\n/* block */ const char* s = "x // y";'
    b = 'int f() {\n  return 1;  // another note\n}\nconst char* s = "x // y";'
    assert bench.code_text(a) == bench.code_text(b)
    assert bench.code_text(a) != bench.code_text(a.replace("return 1", "return 2"))
    assert bench.code_text('"a /* b */"') == '"a /* b */"'  # inside a string: code


def test_traffic_key_covers_every_source_but_the_fp32_gemms(tmp_path):
    # the key changes with any .cu / .cuh file's code except the strict-fp32
    # GEMMs' file, which no bf16 step runs
    for name, body in (("a.cu", "int a;"), ("b.cuh", "int b;"), ("gemm_simt.cu", "int c;"),
                       ("notes.txt", "x")):
        (tmp_path / name).write_text(body)
    key = bench.src_hash(str(tmp_path))
    (tmp_path / "gemm_simt.cu").write_text("int c2;")
    (tmp_path / "notes.txt").write_text("y")
    assert bench.src_hash(str(tmp_path)) == key
    (tmp_path / "b.cuh").write_text("int b2;")
    assert bench.src_hash(str(tmp_path)) != key
