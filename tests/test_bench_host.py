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
    # the committed records match the committed sources
    assert bench._traffic("qwen3_decode", "gemm_w13_swiglu") is not None
    assert bench._traffic("qwen3_decode", "gemm_w13_swiglu_mxfp4", "grouped_gemm_mxfp4.cu") is not None
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
