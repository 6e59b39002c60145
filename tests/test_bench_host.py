"""Host-side arithmetic of bench.py (CPU): algorithmic bytes and FLOPs per launch, the ncu traffic
lookup keyed to the kernel source, the config record and the argument checks."""
import json
import os
import shutil

import numpy as np
import pytest

import bench
import moe_inputs as mi


def test_layer_work_closed_forms():
    cfg = mi.CONFIGS["qwen3_decode"]
    counts = np.full(cfg.E, cfg.T * cfg.k // cfg.E)
    counts[5] = 0                                        # one idle expert streams no weights
    w = bench.layer_work(cfg, counts)
    A = cfg.E - 1
    assert w["active_experts"] == A
    assert w["gemm_w13"]["bytes"] == A * 2 * 1536 * 4096 * 2
    assert w["gemm_down"]["bytes"] == A * 4096 * 1536 * 2
    P = cfg.T * cfg.k
    assert w["gemm_w13"]["flops"] == 2 * P * 4096 * 2 * 1536
    assert w["gemm_down"]["flops"] == 2 * P * 1536 * 4096
    # the shared expert adds its weights once and its FLOPs over all T rows
    hy = mi.CONFIGS["hy3_decode"]
    wh = bench.layer_work(hy, np.ones(hy.E))
    assert wh["gemm_w13"]["bytes"] == hy.E * 2 * hy.I * hy.H * 2 + 2 * hy.I_s * hy.H * 2
    assert wh["gemm_down"]["flops"] == 2 * hy.T * hy.k * hy.I * hy.H + 2 * hy.T * hy.I_s * hy.H


def test_traffic_lookup_is_keyed_to_the_kernel_source(tmp_path, monkeypatch):
    # a committed record is used exactly when it was taken on the current kernel source
    import hashlib
    recs = json.load(open(os.path.join(bench.ROOT, "profiles", "dram_traffic.json")))
    for wl, kernels in recs.items():
        for kern, rec in kernels.items():
            src = rec.get("src", "grouped_gemm.cu")
            with open(os.path.join(bench.ROOT, "moe_expert_layer_fwd_gb300", "csrc", src), "rb") as f:
                sha = hashlib.sha256(f.read()).hexdigest()[:16]
            want = rec["bytes_per_launch"] if rec["src_sha"] == sha else None
            assert bench._traffic(wl, kern, src) == want
    assert bench._traffic("qwen3_decode", "no_such_kernel") is None
    assert bench._traffic("no_such_workload", "gemm_w13_swiglu") is None
    # an edited kernel source voids the record
    root = tmp_path / "root"
    (root / "profiles").mkdir(parents=True)
    (root / "moe_expert_layer_fwd_gb300" / "csrc").mkdir(parents=True)
    shutil.copy(os.path.join(bench.ROOT, "profiles", "dram_traffic.json"), root / "profiles")
    src = os.path.join(bench.ROOT, "moe_expert_layer_fwd_gb300", "csrc", "grouped_gemm.cu")
    dst = root / "moe_expert_layer_fwd_gb300" / "csrc" / "grouped_gemm.cu"
    shutil.copy(src, dst)
    monkeypatch.setattr(bench, "ROOT", str(root))
    rec = json.load(open(root / "profiles" / "dram_traffic.json"))["qwen3_decode"]["gemm_w13_swiglu"]
    with open(dst, "rb") as f:
        rec["src_sha"] = hashlib.sha256(f.read()).hexdigest()[:16]
    json.dump({"qwen3_decode": {"gemm_w13_swiglu": rec}}, open(root / "profiles" / "dram_traffic.json", "w"))
    assert bench._traffic("qwen3_decode", "gemm_w13_swiglu") == rec["bytes_per_launch"]
    with open(dst, "a") as f:
        f.write("\n// edited\n")
    assert bench._traffic("qwen3_decode", "gemm_w13_swiglu") is None


def test_config_record_and_overrides():
    a = bench._args(["--workload", "qwen3_decode", "--override", "E=32,T=16"])
    cfg = bench.workload(a)
    assert (cfg.E, cfg.T, cfg.H) == (32, 16, 4096)
    c = bench._config(cfg, 1)
    assert c["workload"] == "qwen3_decode (overridden shape)" and c["global_batch"] == 16
    c = bench._config(mi.CONFIGS["long_prefill"], 4)
    assert c["workload"] == "long_prefill" and c["global_batch"] == 4 * 16384 and c["parallelism"] == "replicas x4"


def test_arguments():
    with pytest.raises(SystemExit):
        bench._args(["--warmup", "2"])
    a = bench._args([])
    assert a.workload == bench.DEFAULT_WORKLOAD and a.warmup >= 3 and a.impl == "gb300"


def test_per_config_selection():
    a = bench._args([])
    assert bench.per_config_names(a) == ["tiny", "hy3_decode", "hy3_prefill", "long_prefill"]
    assert bench.per_config_names(bench._args(["--workload", "long_prefill"])) == []
    assert bench.per_config_names(bench._args(["--override", "E=32"])) == []
    assert bench.per_config_names(bench._args(["--per-config", "none"])) == []
    assert bench.per_config_names(bench._args(["--per-config", "tiny,qwen3_decode"])) == ["tiny"]


def test_oracle_inputs_generate_exactly_the_needed_experts():
    """The CPU legs' inputs: the sampled tokens' experts carry the generated weights (bit for bit
    those of the full generation), and the oracle's result on them equals the one on full inputs."""
    import oracle
    cfg = mi.CONFIGS["hy3_decode"].with_(T=6, H=128, E=12, k=3, I=64, I_s=64)
    full = mi.generate(cfg)
    toks = np.arange(4)
    lazy = bench.oracle_inputs(cfg, toks)
    _, idx = oracle.gating_topk(full.logits, cfg.k, cfg.gate, full.bias, cfg.routed_scaling_factor, cfg.eps)
    for e in np.unique(idx[toks]):
        assert (lazy.w13[e] == full.w13[e]).all() and (lazy.w2[e] == full.w2[e]).all()
    assert (lazy.w13_s == full.w13_s).all() and (lazy.w2_s == full.w2_s).all()
    args = (cfg.k, cfg.gate)
    kw = dict(routed_scaling_factor=cfg.routed_scaling_factor, eps=cfg.eps)
    a = oracle.moe_layer_forward_tokens(toks, full.x, full.logits, *args, full.w13, full.w2, full.bias,
                                        w13_s=full.w13_s, w2_s=full.w2_s, **kw)
    b = oracle.moe_layer_forward_tokens(toks, lazy.x, lazy.logits, *args, lazy.w13, lazy.w2, lazy.bias,
                                        w13_s=lazy.w13_s, w2_s=lazy.w2_s, **kw)
    assert (a["y"] == b["y"]).all()


def test_w4a8_leg_shapes_and_bound():
    """Every workload fits the W4A8 layer's shape limits; its gate/up GEMM is HBM-bound at decode
    sizes and tensor-bound (against the fp8-rate peak) at prefill sizes, by arithmetic intensity."""
    assert all(bench._w4a8_fits(c) for c in mi.CONFIGS.values())
    assert not bench._w4a8_fits(mi.CONFIGS["tiny"].with_(H=192))
    assert not bench._w4a8_fits(mi.CONFIGS["hy3_decode"].with_(I_s=192))
    peaks = {"hbm_gbs": 6788.6, "bf16_tflops": 1855.6}
    ridge = peaks["bf16_tflops"] * bench.FP8_OVER_BF16 * 1e12 / (peaks["hbm_gbs"] * 1e9)
    per_w = 0.5 + 1.0 / 32
    for name, tensor in [("qwen3_decode", False), ("hy3_decode", False), ("hy3_prefill", True), ("long_prefill", True)]:
        c = mi.CONFIGS[name]
        f1 = 2.0 * c.T * c.k * c.H * 2 * c.I + (2.0 * c.T * c.H * 2 * c.I_s if c.n_shared else 0.0)
        b1 = (c.E + (1 if c.n_shared else 0)) * 2 * c.I * c.H * per_w  # every expert active: the lowest intensity
        assert (f1 / b1 >= ridge) == tensor, name
