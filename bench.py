#!/usr/bin/env python3
"""Benchmark of the GB300 MoE expert-layer forward; rank 0 prints one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference] [--workload NAME]

A step is one full layer forward (gating top-k, init-routing, gate/up grouped
GEMM + SwiGLU, down grouped GEMM + routing weight, finalize) through the C ABI
(moe_layer_forward), on seeded synthetic inputs already resident in HBM.
`value` times K plain calls; a second timed loop of K moe_layer_forward_events
calls gives each step's duration (CUDA events on the launching stream), from
which the dominant kernel's roofline is computed.
The default workload is the Qwen3-MoE-style decode layer (T=64, H=4096,
E=128, k=8, I=1536).  Its 4.75 GB of active expert weights per step exceed the
129 MB L2, so no L2 flush is needed between steps.

Multi-GPU: the layer does not shard here; --gpus N (under torchrun) runs N
independent replicas, one per GPU, and reports the whole-job throughput with
the max time over ranks (weak scaling, no data-path collective).

--impl reference times the CPU oracle (the only reference this path has) on a
bounded sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s on 1 GB300; % of HBM BW (decode) / % BF16 TC peak (prefill)"
DEFAULT_WORKLOAD = "qwen3_decode"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def _args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-front-end", action="store_true", help="skip timing the front end (norm + router GEMM)")
    ap.add_argument("--no-mxfp4", action="store_true", help="skip timing the W4A8 layer (MXFP8 x MXFP4 weights)")
    ap.add_argument("--mxfp4-f16", action="store_true",
                    help="also time the 4-bit-weight layer on f16 operands (software-decoded weights)")
    ap.add_argument("--profile-mxfp4", action="store_true",
                    help="with --profile-steps: the MXFP4-weight layer loop on f16 operands instead")
    ap.add_argument("--profile-w4a8", action="store_true",
                    help="with --profile-steps: the W4A8 layer loop instead (for ncu launch lists and captures)")
    ap.add_argument("--cpu-baseline-child", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--sample-tokens", type=int, default=0,
                    help="tokens of the CPU-baseline sample (0: as many as fit about --cpu-seconds of oracle time)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target oracle time of the CPU-baseline sample when --sample-tokens is 0")
    ap.add_argument("--profile-steps", action="store_true",
                    help="plain moe_layer_forward loop only (for ncu launch lists)")
    ap.add_argument("--override", default="",
                    help="shape overrides of the workload for small profiling captures, e.g. E=32,T=16")
    ap.add_argument("--per-config", default="auto",
                    help="workloads measured beside the headline one, each in its own record: 'auto' (all other "
                         "workloads when the headline is the default one), 'none', or a comma-separated list")
    a = ap.parse_args(argv)
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    return a


# ------------------------------------------------------------------ clocks
class Clocks:
    """nvidia-smi sampling of SM clock and throttle reasons every 200 ms."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_id: str):
        self.device_id = device_id
        self.proc = None
        self.file = None
        self.window = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", self.device_id], stdout=self.file,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        out = {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        if self.proc is None:
            out["note"] = "nvidia-smi unavailable"
            return out
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = []
        for line in self.file.read().splitlines():
            c = [x.strip() for x in line.split(",")]
            if len(c) < 10:
                continue
            try:
                ts = _dt.datetime.strptime(c[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(c[2]), float(c[3]), c[4], c[6:10]))
            except ValueError:
                continue
        os.unlink(self.file.name)
        if not rows:
            out["note"] = "no samples"
            return out
        inwin = [r for r in rows if self.window and self.window[0] - 0.2 <= r[0] <= self.window[1] + 0.2]
        use = inwin if inwin else rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[4]) if v.lower() == "active"})
        out.update(sm_mhz=statistics.median(r[1] for r in use), sm_max_mhz=max(r[2] for r in use),
                   reasons=reasons, samples=len(use), samples_in_timed_region=len(inwin))
        try:
            out["power_w_max"] = max(float(r[3]) for r in use)
        except ValueError:
            pass
        return out


# ------------------------------------------------------------------ distributed plumbing
def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def _barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ work accounting
def layer_work(cfg, counts):
    """Algorithmic bytes and FLOPs of the two grouped GEMMs for one step."""
    import numpy as np
    A = int((np.asarray(counts) > 0).sum())
    P = cfg.T * cfg.k
    w13_b = A * 2 * cfg.I * cfg.H * 2 + (2 * cfg.I_s * cfg.H * 2 if cfg.n_shared else 0)
    w2_b = A * cfg.H * cfg.I * 2 + (cfg.H * cfg.I_s * 2 if cfg.n_shared else 0)
    f1 = 2 * P * cfg.H * 2 * cfg.I + (2 * cfg.T * cfg.H * 2 * cfg.I_s if cfg.n_shared else 0)
    f2 = 2 * P * cfg.I * cfg.H + (2 * cfg.T * cfg.I_s * cfg.H if cfg.n_shared else 0)
    return dict(active_experts=A, gemm_w13=dict(bytes=w13_b, flops=f1), gemm_down=dict(bytes=w2_b, flops=f2))


def _traffic(workload, kernel, src_file="grouped_gemm.cu"):
    """DRAM bytes per launch from the committed ncu summary, if it matches the current kernel source."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(kernel)
    if not e:
        return None
    src = os.path.join(ROOT, "moe_expert_layer_fwd_gb300", "csrc", src_file)
    with open(src, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    return e.get("bytes_per_launch") if e.get("src_sha") == sha else None


# ------------------------------------------------------------------ CPU oracle timing
def workload(args):
    import moe_inputs as mi
    cfg = mi.CONFIGS[args.workload]
    if args.override:
        kw = {}
        for item in args.override.split(","):
            key, val = item.split("=")
            kw[key.strip()] = type(getattr(cfg, key.strip()))(val)
        cfg = cfg.with_(**kw)
    return cfg


def oracle_inputs(cfg, tokens):
    """The workload's inputs for the oracle on `tokens`: x, logits and bias in full, and the expert
    weights of the experts those tokens are routed to (the oracle's own routing), each generated from
    its slice of the seeded weight stream; the other experts' rows are never touched (the arrays are
    allocated, not filled)."""
    import numpy as np
    import moe_inputs as mi
    import oracle
    inp = mi.generate(cfg, weights=False)
    _, idx = oracle.gating_topk(inp.logits, cfg.k, cfg.gate, inp.bias, cfg.routed_scaling_factor, cfg.eps)
    w13 = np.empty((cfg.E, 2 * cfg.I, cfg.H), np.uint16)
    w2 = np.empty((cfg.E, cfg.H, cfg.I), np.uint16)
    for e in np.unique(idx[np.asarray(tokens)]):
        w13[e], w2[e] = mi.expert_weights(cfg, int(e))
    inp.w13, inp.w2 = w13, w2
    if cfg.n_shared:
        full = mi.generate(cfg.with_(E=1, T=1))  # the shared expert's streams do not depend on E or T
        inp.w13_s, inp.w2_s = full.w13_s, full.w2_s
    return inp


def _spread(n, T):
    """n token indices spread evenly over [0, T)."""
    import numpy as np
    return np.unique(np.linspace(0, T - 1, n).round().astype(np.int64))


def cpu_baseline_child(args):
    """Runs in a subprocess with the BLAS thread count fixed: times the oracle on a token sample --
    args.sample_tokens tokens, or (0) a sample grown 4x at a time from 8 tokens until one run takes at
    least half of args.cpu_seconds or covers the batch (the oracle's time grows with the experts a
    sample touches, not in proportion to its tokens); tokens spread evenly over the batch.  Input
    generation is outside the timed region."""
    import numpy as np
    import oracle
    cfg = workload(args)

    def run(toks):
        inp = oracle_inputs(cfg, toks)
        t0 = time.perf_counter()
        oracle.moe_layer_forward_tokens(toks, inp.x, inp.logits, cfg.k, cfg.gate, inp.w13, inp.w2, inp.bias,
                                        cfg.routed_scaling_factor, cfg.eps, inp.w13_s, inp.w2_s)
        return time.perf_counter() - t0

    if args.sample_tokens > 0:
        toks = _spread(min(args.sample_tokens, cfg.T), cfg.T)
        dt = run(toks)
    else:
        n = min(8, cfg.T)
        while True:
            toks = _spread(n, cfg.T)
            dt = run(toks)
            if dt >= args.cpu_seconds / 2 or n >= cfg.T:
                break
            n = min(cfg.T, 4 * n)
    print(json.dumps({"tokens": int(len(toks)), "seconds": dt}))


def cpu_baseline(args, cores=None, workload_name=None, override=None):
    """The oracle timed on a sample of a workload's tokens (cpu_baseline_child), in a child process on
    `cores` host threads (default: all of this process's affinity set)."""
    workload_name = workload_name or args.workload
    override = args.override if override is None else override
    cores = cores or len(os.sched_getaffinity(0))
    env = dict(os.environ, OMP_NUM_THREADS=str(cores), OPENBLAS_NUM_THREADS=str(cores), MKL_NUM_THREADS=str(cores))
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    cmd = [sys.executable, os.path.join(ROOT, "bench.py"), "--cpu-baseline-child", "--workload", workload_name,
           "--sample-tokens", str(args.sample_tokens), "--cpu-seconds", str(args.cpu_seconds), "--override", override]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        return {"value": None, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                "error": r.stderr.strip().splitlines()[-1:] }
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": d["tokens"] / d["seconds"], "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{d['tokens']} tokens spread over the {workload_name} workload (routing of all tokens, "
                      f"expert FFNs of the sampled tokens, float64 numpy with BLAS on {cores} "
                      f"thread{'s' if cores > 1 else ''}): {d['seconds']:.2f} s"}


# ------------------------------------------------------------------ reference arm (the oracle)
def run_reference(args, rank, world):
    if rank != 0:
        return
    import numpy as np
    import moe_inputs as mi
    import oracle
    cfg = workload(args)
    inp = oracle_inputs(cfg, np.arange(args.warmup + args.steps) % cfg.T)
    cores = len(os.sched_getaffinity(0))

    def step(i):
        oracle.moe_layer_forward_tokens(np.array([i % cfg.T]), inp.x, inp.logits, cfg.k, cfg.gate, inp.w13, inp.w2,
                                        inp.bias, cfg.routed_scaling_factor, cfg.eps, inp.w13_s, inp.w2_s)

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    v = args.steps / dt
    line = {
        "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded Philox inputs, random-init weights)",
        "impl": "reference",
        "config": _config(cfg, world),
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"1 token of the {args.workload} workload per step (routing of all tokens, its "
                                   f"{cfg.k} expert FFNs in float64 numpy)"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _config(cfg, world):
    import moe_inputs as mi
    name = cfg.name if cfg == mi.CONFIGS.get(cfg.name) else cfg.name + " (overridden shape)"
    return {"workload": name, "T": cfg.T, "H": cfg.H, "E": cfg.E, "k": cfg.k, "I": cfg.I, "gate": cfg.gate,
            "routed_scaling_factor": cfg.routed_scaling_factor, "n_shared": cfg.n_shared, "I_s": cfg.I_s,
            "zipf_s": cfg.zipf_s, "global_batch": cfg.T * world,
            "l2": "inputs larger than L2 (the active expert weights read each step exceed 129 MB)",
            "parallelism": f"replicas x{world}"}


# ------------------------------------------------------------------ front end (the step before gating)
def front_end(args, cfg, K, W, moe, mi, d16):
    """Times the fused residual add + RMSNorm + cast and the router gate GEMM on the workload's
    [T, H] hidden state and E experts (synthetic bf16 hidden state, residual, norm and gate weights).
    Reported beside the layer, not part of its value."""
    import torch
    T, H, E = cfg.T, cfg.H, cfg.E
    h = d16(mi.normal_bf16(cfg.seed, 101, (T, H)))
    res = d16(mi.normal_bf16(cfg.seed, 102, (T, H)))
    w = d16(mi.normal_bf16(cfg.seed, 103, (H,), 1.0, 0.1))
    wg = d16(mi.normal_bf16(cfg.seed, 104, (E, H), 0.0, 0.02))
    y32 = torch.empty((T, H), dtype=torch.float32, device="cuda")
    y16 = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    r_out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
    ws = torch.empty(moe.lib().moe_router_logits_workspace_size(T, H, E), dtype=torch.uint8, device="cuda")
    for _ in range(W):
        moe.moe_add_rms_norm_cast(h, res, w, 1e-6, y32, y16, r_out)
        moe.moe_router_logits(y32, wg, logits, ws)
    torch.cuda.synchronize()
    codes = torch.empty((T, H), dtype=torch.uint8, device="cuda")
    scales = torch.empty((T, H // 32), dtype=torch.uint8, device="cuda")

    def mx():
        moe.lib().moe_add_rms_norm_mxfp8(h.data_ptr(), res.data_ptr(), w.data_ptr(), T, H, 1e-6, codes.data_ptr(),
                                         scales.data_ptr(), None, r_out.data_ptr(), None)

    for _ in range(W):
        mx()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    n_ms, r_ms, m_ms = 0.0, 0.0, 0.0
    for _ in range(K):
        ev[0].record()
        mx()
        ev[1].record()
        torch.cuda.synchronize()
        m_ms += ev[0].elapsed_time(ev[1])
    for _ in range(K):
        ev[0].record()
        moe.moe_add_rms_norm_cast(h, res, w, 1e-6, y32, y16, r_out)
        ev[1].record()
        moe.moe_router_logits(y32, wg, logits, ws)
        ev[2].record()
        torch.cuda.synchronize()
        n_ms += ev[0].elapsed_time(ev[1])
        r_ms += ev[1].elapsed_time(ev[2])
    return {"what": "fused residual add + RMSNorm + cast (fp32 and bf16 out), then the fp32 router gate GEMM; "
                    "separately the fused add + RMSNorm + MXFP8 quantisation (E4M3 codes, E8M0 scales); "
                    "synthetic bf16 inputs of the workload's T, H, E; CUDA events per kernel, mean of K",
            "norm_ms": n_ms / K, "router_ms": r_ms / K, "norm_mxfp8_ms": m_ms / K,
            "gpu_launches": (2 + (2 if ws.numel() > moe.lib().moe_status_bytes() else 1)) * K,
            "norm_bytes": T * H * 2 * 2 + H * 2 + T * H * (4 + 2 + 2), "router_flops": 2 * T * H * E,
            "mx_bytes": T * H * 2 * 2 + H * 2 + T * H * (1 + 2) + T * H // 32}


# ------------------------------------------------------------------ the layer on MXFP4 expert weights
def mxfp4_leg(args, cfg, K, W, moe, inp, t, d16, peaks, peak_src, y_bf16):
    """Times moe.Mxfp4Layer (gating, routing, f16 row gather, the two 4-bit grouped GEMMs, finalize)
    on the workload with its expert weights quantised to MXFP4 on the GPU (one-time, not timed).
    Reported beside the bf16 layer, not part of its value (a lower weight precision)."""
    import torch
    w13q = moe.moe_mxfp4_prepack(*moe.moe_mxfp4_quantize(d16(inp.w13)), gate_up=True)
    w2q = moe.moe_mxfp4_prepack(*moe.moe_mxfp4_quantize(t["w2"]), gate_up=False)
    torch.cuda.empty_cache()
    layer = moe.Mxfp4Layer(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.gate, cfg.routed_scaling_factor, cfg.eps)
    args_fw = dict(x=t["x"], logits=t["logits"], w13=w13q, w2=w2q, bias=t["bias"])
    for _ in range(W):
        layer.forward(**args_fw)
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record()
    for _ in range(K):
        layer.forward(**args_fw)
    s1.record()
    torch.cuda.synchronize()
    ms = s0.elapsed_time(s1) / K
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    for i in range(K):
        layer.forward(events=evs[i], **args_fw)
    torch.cuda.synchronize()
    names = ["gating_routing_gather", "gemm_w13_swiglu_mxfp4", "gemm_down_mxfp4", "finalize"]
    kern = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K)) for j, n in enumerate(names)}
    for w_ in (layer.ws, layer.routing_ws):
        st = moe.moe_get_device_status(w_)
        if st != moe.MOE_OK:
            raise SystemExit(f"MXFP4 layer device status: {moe.status_string(st)}")
    A = int((layer.routing["counts"].cpu() > 0).sum())
    per_w = 0.5 + 1.0 / 32  # code + scale bytes per weight
    b1 = A * 2 * cfg.I * cfg.H * per_w + A * 2 * cfg.I * 4   # + the per-row fp32 exponent offsets
    b2 = A * cfg.H * cfg.I * per_w + A * cfg.H * 4
    t1 = kern["gemm_w13_swiglu_mxfp4"] * 1e-3
    y = layer.y.float()
    return {
        "value": cfg.T / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms, "kernels_ms": kern,
        "gpu_launches": moe.Mxfp4Layer.KERNELS_PER_FORWARD * K,
        "weights": "MXFP4 (E2M1 codes, E8M0 scale per 32 along K), quantised on the GPU from the bf16 weights; "
                   "token rows and act in f16",
        "roofline": {"bound": "hbm", "kernel": "gemm_w13_swiglu_mxfp4", "achieved": b1 / t1 / 1e9,
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": b1 / t1 / 1e9 / peaks["hbm_gbs"],
                     "peak_source": f"{peak_src} (hbm_gbs)", "algorithmic_bytes_per_launch": b1,
                     "per_unit": f"{2 * cfg.I * cfg.H} weights x {per_w} B + {2 * cfg.I} x 4 B row offsets per "
                                 f"active expert (x {A})",
                     "traffic": _traffic(cfg.name, "gemm_w13_swiglu_mxfp4", "grouped_gemm_mxfp4.cu")},
        "gemm_down_mxfp4_gbs": b2 / (kern["gemm_down_mxfp4"] * 1e-3) / 1e9,
        "max_rel_diff_vs_bf16_layer": float((y - y_bf16).abs().max() / y_bf16.abs().max()),
    }


# ------------------------------------------------------------------ the W4A8 layer (MXFP8 x MXFP4)
class W4a8Weights:
    """The MXFP4-quantised, prepacked expert weights, kept for the next workload with the same weights."""

    def __init__(self):
        self.key = None
        self.w = None

    def get(self, cfg, moe, mi, d16, t):
        import torch
        key = (cfg.seed, cfg.E, cfg.H, cfg.I, cfg.w_std, cfg.n_shared, cfg.I_s)
        if key != self.key:
            self.w = None
            torch.cuda.empty_cache()
            w13_raw = d16(mi.normal_bf16(cfg.seed, mi.TID_W13, (cfg.E, 2 * cfg.I, cfg.H), 0.0, cfg.w_std))
            w13 = moe.moe_w4a8_prepack(*moe.moe_mxfp4_quantize(w13_raw), gate_up=True)
            del w13_raw
            w2 = moe.moe_w4a8_prepack(*moe.moe_mxfp4_quantize(t["w2"]), gate_up=False)
            w13_s = w2_s = None
            if cfg.n_shared:
                sh = mi.generate(cfg.with_(E=1, T=1))
                w13_s = moe.moe_w4a8_prepack(*moe.moe_mxfp4_quantize(d16(sh.w13_s)), gate_up=True)
                w2_s = moe.moe_w4a8_prepack(*moe.moe_mxfp4_quantize(d16(sh.w2_s)), gate_up=False)
            torch.cuda.empty_cache()
            self.w = (w13, w2, w13_s, w2_s)
            self.key = key
        return self.w


W4A8_WEIGHTS = W4a8Weights()
# dense tensor rate of the block-scaled MXFP8 x MXFP4 MMA over bf16 (nominal 4.5 / 2.25 PFLOP/s)
FP8_OVER_BF16 = 2.0


def w4a8_leg(args, cfg, K, W, moe, mi, d16, t, peaks, peak_src, y_bf16):
    """Times moe_layer_forward_w4a8 (gating, routing, MXFP8 row gather, the two block-scaled W4A8 GEMMs,
    finalize; the shared expert as one more GEMM segment) on the workload: the expert weights quantised
    to MXFP4 on the GPU and the hidden state to MXFP8 by the fused RMSNorm + MX quantisation (both
    one-time, not timed).  Reported beside the bf16 layer (a lower precision), not part of its value."""
    import torch
    w13, w2, w13_s, w2_s = W4A8_WEIGHTS.get(cfg, moe, mi, d16, t)
    ones = torch.ones(cfg.H, dtype=torch.bfloat16, device="cuda")
    xc, xs, _, _ = moe.moe_add_rms_norm_mxfp8(t["x"], None, ones, 1e-6, with_fp32=False)
    layer = moe.W4a8Layer(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.gate, cfg.routed_scaling_factor, cfg.eps,
                          cfg.n_shared, cfg.I_s)
    fw = dict(x_codes=xc, x_scales=xs, logits=t["logits"], w13=w13, w2=w2, bias=t["bias"], w13_s=w13_s, w2_s=w2_s)
    for _ in range(W):
        layer.forward(**fw)
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record()
    for _ in range(K):
        layer.forward(**fw)
    s1.record()
    torch.cuda.synchronize()
    ms = s0.elapsed_time(s1) / K
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    for i in range(K):
        layer.forward_events(evs[i], **fw)
    torch.cuda.synchronize()
    st = moe.moe_get_device_status(layer.ws)
    if st != moe.MOE_OK:
        raise SystemExit(f"{cfg.name}: W4A8 layer device status: {moe.status_string(st)}")
    names = ["gating", "init_routing_and_row_gather", "gemm_w13_swiglu_w4a8", "gemm_down_w4a8", "finalize"]
    kern = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K)) for j, n in enumerate(names)}
    A = int((layer.counts.cpu() > 0).sum())
    per_w = 0.5 + 1.0 / 32  # code + scale bytes per weight
    n_units = A + (1 if cfg.n_shared else 0)
    b1 = n_units * 2 * cfg.I * cfg.H * per_w
    b2 = n_units * cfg.H * cfg.I * per_w
    f1 = 2.0 * cfg.T * cfg.k * cfg.H * 2 * cfg.I + (2.0 * cfg.T * cfg.H * 2 * cfg.I_s if cfg.n_shared else 0.0)
    f2 = f1 / 2  # down: the same rows times I instead of 2I columns
    t1 = kern["gemm_w13_swiglu_w4a8"] * 1e-3
    t2 = kern["gemm_down_w4a8"] * 1e-3
    y = layer.y.float()
    # bound of the gate/up GEMM: HBM below the ridge of the fp8-rate tensor peak and HBM, tensor above
    tc_peak = peaks["bf16_tflops"] * FP8_OVER_BF16
    if f1 / b1 < tc_peak * 1e12 / (peaks["hbm_gbs"] * 1e9):
        roof = {"bound": "hbm", "kernel": "gemm_w13_swiglu_w4a8", "achieved": b1 / t1 / 1e9,
                "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": b1 / t1 / 1e9 / peaks["hbm_gbs"],
                "peak_source": f"{peak_src} (hbm_gbs)"}
    else:
        roof = {"bound": "tensor", "kernel": "gemm_w13_swiglu_w4a8", "achieved": f1 / t1 / 1e12,
                "peak": tc_peak, "unit": "TFLOP/s", "frac": f1 / t1 / 1e12 / tc_peak,
                "peak_source": f"{peak_src} (bf16_tflops) x {FP8_OVER_BF16} (nominal fp8 / bf16 dense ratio)"}
    roof.update(algorithmic_bytes_per_launch=b1, flops_per_launch=f1,
                per_unit=f"{2 * cfg.I * cfg.H} weights x {per_w} B per streamed expert (x {A} active"
                         + (" + the shared expert)" if cfg.n_shared else ")"),
                traffic=_traffic(cfg.name, "gemm_w13_swiglu_w4a8", "grouped_gemm_w4a8.cu"))
    return {
        "value": cfg.T / (ms * 1e-3), "unit": "tokens/s", "ms_per_step": ms, "kernels_ms": kern,
        "gpu_launches": layer.launches * K,
        "precision": "W4A8: MXFP8 hidden state and act (E4M3, E8M0 scale per 32), MXFP4 expert weights (E2M1, E8M0 "
                     "scale per 32) quantised on the GPU from the bf16 weights; block-scaled tcgen05 MMA "
                     "(kind::mxf8f6f4), fp32 accumulation",
        "roofline": roof,
        "gemm_down_w4a8": {"achieved_gbs": b2 / t2 / 1e9, "frac": b2 / t2 / 1e9 / peaks["hbm_gbs"],
                           "achieved_tflops": f2 / t2 / 1e12, "tc_frac": f2 / t2 / 1e12 / tc_peak},
        "layer_hbm_frac_of_measured": (b1 + b2) / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
        "layer_tc_frac_of_fp8_peak": (f1 + f2) / (ms * 1e-3) / 1e12 / tc_peak,
        "max_rel_diff_vs_bf16_layer": float((y - y_bf16).abs().max() / y_bf16.abs().max()),
    }


# ------------------------------------------------------------------ GB300 arm
# the workloads measured beside the default one (hy3_decode and hy3_prefill share their weights)
OTHER_WORKLOADS = ["tiny", "hy3_decode", "hy3_prefill", "long_prefill"]


def _w4a8_fits(cfg):
    """The W4A8 layer's shape limits: H a multiple of 256, I and I_s of 128."""
    return cfg.H % 256 == 0 and cfg.I % 128 == 0 and (not cfg.n_shared or cfg.I_s % 128 == 0)


def _decode_sized(cfg):
    """Decode-shaped problems (at most 32 token rows per expert on average, no more than 32 tokens for a
    shared expert), the shapes the f16-operand 4-bit layer's 32-column tiles are built for."""
    return cfg.T * cfg.k <= 32 * cfg.E and cfg.T <= 64 and cfg.E >= 16


def per_config_names(args):
    if args.per_config == "none":
        return []
    if args.per_config == "auto":
        if args.workload != DEFAULT_WORKLOAD or args.override:
            return []
        return [n for n in OTHER_WORKLOADS if n != args.workload]
    return [n for n in args.per_config.split(",") if n and n != args.workload]


class DeviceWeights:
    """Expert weights resident in HBM, kept for the next workload when it has the same weights
    (the weights depend only on the seed, E, H, I, the shared expert and their spread)."""

    def __init__(self):
        self.key = None
        self.t = None

    def get(self, cfg, moe, mi, d16):
        import torch
        key = (cfg.seed, cfg.E, cfg.H, cfg.I, cfg.w_std, cfg.n_shared, cfg.I_s)
        if key != self.key:
            self.t = None
            torch.cuda.empty_cache()
            inp = mi.generate(cfg)
            # weights are loaded once: w13 goes through the one-time gate/up packing (not timed)
            w13_raw = d16(inp.w13)
            self.t = dict(w13=moe.moe_prepack_w13(w13_raw), w2=d16(inp.w2),
                          w13_s=moe.moe_prepack_w13(d16(inp.w13_s)) if inp.w13_s is not None else None,
                          w2_s=d16(inp.w2_s) if inp.w2_s is not None else None)
            del w13_raw, inp
            self.key = key
        return self.t


def measure(args, cfg, K, W, world, rank, local, moe, mi, d16, weights, peaks, peak_src, dev_id):
    """One workload: the headline timed loop, per-step events, e2e, clocks, roofline, CPU baseline."""
    import numpy as np
    import torch

    inp = mi.generate(cfg, weights=False)
    t = dict(weights.get(cfg, moe, mi, d16))
    t.update(x=d16(inp.x), logits=torch.from_numpy(inp.logits).cuda(),
             bias=torch.from_numpy(inp.bias).cuda() if inp.bias is not None else None)
    layer = moe.MoELayer(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.gate, cfg.routed_scaling_factor, cfg.eps,
                         cfg.n_shared, cfg.I_s)
    launches = moe.moe_layer_kernel_launches(layer.desc)

    clocks = Clocks(dev_id) if rank == 0 else None
    if clocks:
        clocks.start()
    # the first (cold) call, timed on its own: tensor-map encoding, first launches, cold L2 and TLBs
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    c0.record()
    layer.forward(**t)
    c1.record()
    torch.cuda.synchronize()
    cold_ms = c0.elapsed_time(c1)
    for _ in range(W):
        layer.forward(**t)
    torch.cuda.synchronize()
    status = moe.moe_get_device_status(layer.ws)
    if status != moe.MOE_OK:
        raise SystemExit(f"{cfg.name}: device status after warm-up: {moe.status_string(status)}")
    counts = layer.counts.cpu().numpy()
    # timed region 1 (the value): K plain moe_layer_forward calls
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    _barrier(world)
    torch.cuda.synchronize()
    w0 = time.time()
    start.record()
    for _ in range(K):
        layer.forward(**t)
    end.record()
    torch.cuda.synchronize()
    w1 = time.time()
    if clocks:
        clocks.mark(w0, w1)
    _barrier(world)
    ms_total = _max_over_ranks(start.elapsed_time(end), world)
    status = moe.moe_get_device_status(layer.ws)
    if status != moe.MOE_OK:
        raise SystemExit(f"{cfg.name}: device status after the timed region: {moe.status_string(status)}")
    # timed region 2 (per-kernel durations): K moe_layer_forward_events calls, six events
    # recorded on the launching stream around the steps of every call
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    for row in evs:
        for e in row:
            e.record()
    torch.cuda.synchronize()
    for i in range(K):
        layer.forward_events(evs[i], **t)
    torch.cuda.synchronize()
    names = ["gating", "init_routing", "gemm_w13_swiglu", "gemm_down", "finalize"]
    kern_ms = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(K))
               for j, n in enumerate(names)}
    step_ms = sorted(evs[i][0].elapsed_time(evs[i][5]) for i in range(K))

    # end to end: pinned host inputs -> device, forward, result -> pinned host, every step.  Served
    # as a pipeline: two buffer sets (inputs, layer outputs, pinned results) and three streams, so
    # step i+1's inputs are copied in and step i-1's result copied out while step i computes; the
    # host reads every step's result (waiting for it two steps later, before reusing its buffer).
    e2e = None
    if not args.no_e2e:
        NB = 2
        hx = torch.from_numpy(np.ascontiguousarray(inp.x).view(np.int16)).pin_memory()
        hl = torch.from_numpy(inp.logits).pin_memory()
        layers = [layer] + [moe.MoELayer(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.gate, cfg.routed_scaling_factor,
                                         cfg.eps, cfg.n_shared, cfg.I_s) for _ in range(NB - 1)]
        hys = [torch.empty((cfg.T, cfg.H), dtype=torch.int16).pin_memory() for _ in range(NB)]
        dxs = [torch.empty((cfg.T, cfg.H), dtype=torch.int16, device="cuda") for _ in range(NB)]
        dls = [torch.empty_like(t["logits"]) for _ in range(NB)]
        s_in, s_comp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(NB)]
        ev_comp = [torch.cuda.Event() for _ in range(NB)]
        ev_out = [torch.cuda.Event() for _ in range(NB)]
        pending = [False] * NB
        checksum = [0]

        def take(b):
            # the host reads the result that buffer set b holds (waiting for its copy-out)
            if pending[b]:
                ev_out[b].synchronize()
                checksum[0] ^= int(hys[b][0, 0]) ^ int(hys[b][-1, -1])
                pending[b] = False

        def e2e_step(i):
            b = i % NB
            take(b)
            s_in.wait_event(ev_comp[b])      # the forward that read these input buffers is done
            with torch.cuda.stream(s_in):
                dxs[b].copy_(hx, non_blocking=True)
                dls[b].copy_(hl, non_blocking=True)
                ev_in[b].record(s_in)
            s_comp.wait_event(ev_in[b])
            s_comp.wait_event(ev_out[b])     # this layer's output was copied out
            te = dict(t)
            te["x"] = dxs[b].view(torch.bfloat16)
            te["logits"] = dls[b]
            layers[b].forward(stream=s_comp, **te)
            ev_comp[b].record(s_comp)
            s_out.wait_event(ev_comp[b])
            with torch.cuda.stream(s_out):
                hys[b].copy_(layers[b].y.view(torch.int16), non_blocking=True)
                ev_out[b].record(s_out)
            pending[b] = True

        def drain():
            for b in range(NB):
                take(b)

        for i in range(W):
            e2e_step(i)
        drain()
        torch.cuda.synchronize()
        _barrier(world)
        c0 = time.perf_counter()
        for i in range(K):
            e2e_step(i)
        drain()
        c1 = time.perf_counter()
        _barrier(world)
        e2e_s = _max_over_ranks(c1 - c0, world)
        e2e = {"value": world * cfg.T * K / e2e_s, "unit": "tokens/s",
               "h2d_bytes_per_step": hx.numel() * 2 + hl.numel() * 4, "d2h_bytes_per_step": hys[0].numel() * 2,
               "ms_per_step": e2e_s / K * 1e3,
               "sync": "pipelined over 2 buffer sets and 3 streams: inputs copied in and results copied out "
                       "while the neighbouring step computes; every result read on the host"}
        ref_y = layer.y.view(torch.int16).cpu().numpy()
        for b in range(NB):
            if not np.array_equal(hys[b].numpy(), ref_y):
                raise SystemExit(f"{cfg.name}: end-to-end result differs from the device-resident run")
        del layers, dxs, dls

    clk = clocks.stop() if clocks else None

    work = layer_work(cfg, counts)
    ms = ms_total / K
    # dominant kernel: the gate/up grouped GEMM (2/3 of the weight bytes and FLOPs)
    dom = "gemm_w13_swiglu"
    dom_work = work["gemm_w13"]
    t_dom = kern_ms[dom] * 1e-3
    bw = dom_work["bytes"] / t_dom / 1e9
    tf = dom_work["flops"] / t_dom / 1e12
    ridge = peaks["bf16_tflops_sustained"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    ai = dom_work["flops"] / dom_work["bytes"]
    if ai < ridge:
        roof = {"bound": "hbm", "achieved": bw, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": bw / peaks["hbm_gbs"]}
    else:
        roof = {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops_sustained"], "unit": "TFLOP/s",
                "frac": tf / peaks["bf16_tflops_sustained"]}
    roof["traffic"] = _traffic(cfg.name, dom)
    roof.update(kernel=dom, peak_source=f"{peak_src} ({'hbm_gbs' if roof['bound'] == 'hbm' else 'bf16_tflops_sustained'})",
                algorithmic_bytes_per_launch=dom_work["bytes"], flops_per_launch=dom_work["flops"],
                per_unit=f"{2 * cfg.I * cfg.H * 2} weight bytes per active expert "
                         f"(x {work['active_experts']} active experts" + (" + the shared expert)" if cfg.n_shared else ")"),
                launch_ms=kern_ms[dom])
    tot_b = work["gemm_w13"]["bytes"] + work["gemm_down"]["bytes"]
    tot_f = work["gemm_w13"]["flops"] + work["gemm_down"]["flops"]
    layer_roof = {"weight_bytes": tot_b, "flops": tot_f,
                  "hbm_frac_of_measured": tot_b / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                  "tc_frac_of_measured_burst": tot_f / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                  "tc_frac_of_measured_sustained": tot_f / (ms * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"],
                  "how": "the two grouped GEMMs' weight bytes and FLOPs over ms_per_step (the whole layer)"}
    t_down = kern_ms["gemm_down"] * 1e-3
    rec = {
        "value": world * cfg.T * K / (ms_total * 1e-3),
        "unit": "tokens/s",
        "ms_per_step": ms,
        "step_ms": {"median": statistics.median(step_ms), "min": step_ms[0], "cold_first_call": cold_ms,
                    "how": "median and minimum of the K per-call durations of the events loop; the first call "
                           "of the process timed alone"},
        "roofline": roof,
        "roofline_layer": layer_roof,
        "roofline_gemm_down": {"achieved_gbs": work["gemm_down"]["bytes"] / t_down / 1e9,
                               "achieved_tflops": work["gemm_down"]["flops"] / t_down / 1e12},
        "kernels_ms": kern_ms,
        "routing": {"active_experts": work["active_experts"], "max_over_mean": float(counts.max() / counts.mean()),
                    "empty_experts": int((counts == 0).sum())},
        "gpu_launches": launches * K,
        "clocks": clk,
    }
    if e2e:
        rec["e2e"] = e2e
    rec["_y"] = layer.y.float()
    rec["_t"] = t
    rec["_inp"] = inp
    return rec


def run_gb300(args, rank, world, local):
    import numpy as np
    import torch

    import moe_expert_layer_fwd_gb300 as moe
    import moe_inputs as mi
    from moe_expert_layer_fwd_gb300 import build as moe_build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl gb300")
    torch.cuda.set_device(local)
    moe_build.build()
    cfg = workload(args)
    K, W = args.steps, args.warmup

    def d16(u):
        return torch.from_numpy(np.ascontiguousarray(u).view(np.int16)).cuda().view(torch.bfloat16)

    weights = DeviceWeights()
    if args.profile_steps:
        inp = mi.generate(cfg, weights=False)
        t = dict(weights.get(cfg, moe, mi, d16))
        t.update(x=d16(inp.x), logits=torch.from_numpy(inp.logits).cuda(),
                 bias=torch.from_numpy(inp.bias).cuda() if inp.bias is not None else None)
        if args.profile_w4a8:
            w13, w2, w13_s, w2_s = W4A8_WEIGHTS.get(cfg, moe, mi, d16, t)
            ones = torch.ones(cfg.H, dtype=torch.bfloat16, device="cuda")
            xc, xs, _, _ = moe.moe_add_rms_norm_mxfp8(t["x"], None, ones, 1e-6, with_fp32=False)
            l8 = moe.W4a8Layer(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.gate, cfg.routed_scaling_factor, cfg.eps,
                               cfg.n_shared, cfg.I_s)
            for _ in range(W + K):
                l8.forward(xc, xs, t["logits"], w13, w2, t["bias"], w13_s, w2_s)
        elif args.profile_mxfp4:
            full = mi.generate(cfg)
            w13q = moe.moe_mxfp4_prepack(*moe.moe_mxfp4_quantize(d16(full.w13)), gate_up=True)
            w2q = moe.moe_mxfp4_prepack(*moe.moe_mxfp4_quantize(t["w2"]), gate_up=False)
            l4 = moe.Mxfp4Layer(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.gate, cfg.routed_scaling_factor, cfg.eps)
            for _ in range(W + K):
                l4.forward(t["x"], t["logits"], w13q, w2q, t["bias"])
        else:
            layer = moe.MoELayer(cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.gate, cfg.routed_scaling_factor, cfg.eps,
                                 cfg.n_shared, cfg.I_s)
            for _ in range(W + K):
                layer.forward(**t)
        torch.cuda.synchronize()
        return

    dev_id = str(local)
    try:
        dev_id = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        pass
    peaks, src = _peaks()
    rec = measure(args, cfg, K, W, world, rank, local, moe, mi, d16, weights, peaks, src, dev_id)
    y_bf16, t, inp = rec.pop("_y"), rec.pop("_t"), rec.pop("_inp")

    front = None if args.no_front_end else front_end(args, cfg, K, W, moe, mi, d16)
    # the W4A8 layer (its GEMMs walk 32 token columns per tile at decode sizes, 112 at prefill sizes)
    w8 = None
    if not args.no_mxfp4 and _w4a8_fits(cfg):
        w8 = w4a8_leg(args, cfg, K, W, moe, mi, d16, t, peaks, src, y_bf16)
    # the 4-bit-weight layer on f16 operands (routed experts only), on request
    w4 = None
    if args.mxfp4_f16 and cfg.n_shared == 0 and _decode_sized(cfg):
        inp.w13 = mi.normal_bf16(cfg.seed, mi.TID_W13, (cfg.E, 2 * cfg.I, cfg.H), 0.0, cfg.w_std)
        w4 = mxfp4_leg(args, cfg, K, W, moe, inp, t, d16, peaks, src, y_bf16)
        inp.w13 = None
    del t, y_bf16

    others = {}
    for name in per_config_names(args):
        c = mi.CONFIGS[name]
        r = measure(args, c, K, W, world, rank, local, moe, mi, d16, weights, peaks, src, dev_id)
        y_c, t_c = r.pop("_y"), r.pop("_t")
        r.pop("_inp")
        if not args.no_mxfp4 and _w4a8_fits(c):
            r["w4a8"] = w4a8_leg(args, c, K, W, moe, mi, d16, t_c, peaks, src, y_c)
        del y_c, t_c
        r["config"] = _config(c, world)
        others[name] = r
    weights.t = None
    W4A8_WEIGHTS.w = None
    torch.cuda.empty_cache()

    if rank != 0:
        return

    line = {
        "metric": METRIC,
        "value": rec.pop("value"),
        "unit": rec.pop("unit"),
        "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": rec.pop("ms_per_step"),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded Philox inputs, random-init weights)",
        "config": _config(cfg, world),
    }
    line.update(rec)
    if w8:
        line["w4a8"] = w8
    if w4:
        line["mxfp4_weights"] = w4
    if front:
        clk = rec.get("clocks")
        sm_mhz = (clk or {}).get("sm_mhz") or peaks.get("sm_max_mhz", 2070.0)
        fp32_tflops = torch.cuda.get_device_properties(local).multi_processor_count * 128 * 2 * sm_mhz * 1e6 / 1e12
        nb = front.pop("norm_bytes")
        mb = front.pop("mx_bytes")
        front["norm_mxfp8_roofline"] = {"bound": "hbm", "achieved": mb / (front["norm_mxfp8_ms"] * 1e-3) / 1e9,
                                        "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                        "frac": mb / (front["norm_mxfp8_ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"]}
        rf = front.pop("router_flops")
        front["norm_roofline"] = {"bound": "hbm", "achieved": nb / (front["norm_ms"] * 1e-3) / 1e9,
                                  "peak": peaks["hbm_gbs"], "unit": "GB/s",
                                  "frac": nb / (front["norm_ms"] * 1e-3) / 1e9 / peaks["hbm_gbs"]}
        front["router_roofline"] = {"bound": "alu", "achieved": rf / (front["router_ms"] * 1e-3) / 1e12,
                                    "peak": fp32_tflops, "unit": "TFLOP/s",
                                    "frac": rf / (front["router_ms"] * 1e-3) / 1e12 / fp32_tflops,
                                    "peak_source": f"SMs x 128 FP32 lanes x 2 FLOP/FMA x {sm_mhz:.0f} MHz "
                                                   "(median SM clock of the timed region)"}
        line["front_end"] = front
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args)
        if cfg.T * cfg.k <= 32 * cfg.E:  # the small and decode configs: the oracle on one core as well
            line["cpu_baseline_1core"] = cpu_baseline(args, cores=1)
        for name, r in others.items():
            r["cpu_baseline"] = cpu_baseline(args, workload_name=name, override="")
    if others:
        line["per_config"] = others
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = _args(argv)
    if args.cpu_baseline_child:
        cpu_baseline_child(args)
        return
    rank, world, local = _dist()
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_gb300(args, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
