"""GPU parity: every step of the CUDA path, through the C ABI, against the oracle.

Routing (expert choice, counts, offsets, permutation and its inverse, gathered
rows) must be bit-exact; floating-point outputs must meet
max|gpu-oracle|/max|oracle| <= 2e-2 and mean|gpu-oracle|/mean|oracle| <= 5e-3
(single bf16 roundings are also checked element by element).
"""
import numpy as np
import pytest

import moe_inputs as mi
import oracle
from gpu_util import (assert_bf16_rounding_close, assert_close, dev, dev_bf16, host, host_bf16_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    from moe_expert_layer_fwd_gb300 import build
    build.build()
    import moe_expert_layer_fwd_gb300 as m
    return m


def _torch():
    import torch
    return torch


# ---------------------------------------------------------------- a1 gating
GATING_CASES = [
    ("tiny", {}), ("qwen3_decode", {}), ("hy3_decode", {}), ("hy3_prefill", {}), ("long_prefill", {}),
    ("tiny", dict(T=1, E=1, k=1)),
    ("tiny", dict(T=37, E=1024, k=32)),
    ("hy3_decode", dict(T=33, E=200, k=8, bias_std=0.0)),  # sigmoid without bias: many exact key ties
    # the fused op's bias placement (inside the sigmoid)
    ("hy3_decode", dict(gate="sigmoid_inner_bias")),
    ("hy3_prefill", dict(gate="sigmoid_inner_bias", bias_std=0.5)),
    ("tiny", dict(T=37, E=1024, k=32, gate="sigmoid_inner_bias", bias_std=1.0, routed_scaling_factor=2.826)),
]


@pytest.mark.parametrize("name,over", GATING_CASES)
def test_gating_topk_parity(moe, name, over):
    cfg = mi.CONFIGS[name].with_(**over)
    inp = mi.generate(cfg, weights=False)
    w_ref, idx_ref = oracle.gating_topk(inp.logits, cfg.k, cfg.gate, inp.bias, cfg.routed_scaling_factor, cfg.eps)
    w, idx = moe.moe_gating_topk(dev(inp.logits), cfg.k, cfg.gate, dev(inp.bias) if inp.bias is not None else None,
                                 cfg.routed_scaling_factor, cfg.eps)
    _torch().cuda.synchronize()
    assert (host(idx) == idx_ref).all(), "expert choice differs"
    np.testing.assert_allclose(host(w), w_ref, rtol=2e-6, atol=1e-7)


def test_gating_ties_on_coarse_grid(moe):
    rng = np.random.default_rng(0)
    logits = (np.round(rng.normal(size=(300, 64)) * 4) / 4).astype(np.float32)
    logits[:10] = 0.0
    logits[10:20, :7] = -0.0
    # a bias on a coarse grid keeps l + b on the grid: exact ties inside the sigmoid too
    bias = (np.round(rng.normal(size=64) * 2) / 4).astype(np.float32)
    for gate, b in (("softmax", None), ("sigmoid", None), ("sigmoid_inner_bias", None),
                    ("sigmoid_inner_bias", bias)):
        rsf = 1.0 if gate == "softmax" else 2.826
        w_ref, idx_ref = oracle.gating_topk(logits, 6, gate, b, rsf)
        w, idx = moe.moe_gating_topk(dev(logits), 6, gate, dev(b) if b is not None else None, rsf)
        assert (host(idx) == idx_ref).all()
        np.testing.assert_allclose(host(w), w_ref, rtol=2e-6, atol=1e-7)


# ---------------------------------------------------------------- a2 routing
ROUTING_CASES = [(16, 8, 2, 256), (64, 128, 8, 4096), (16, 192, 8, 4096), (4096, 192, 8, 64), (16384, 128, 8, 64),
                 (1, 1, 1, 64), (3, 1024, 32, 128), (20000, 7, 3, 64)]


@pytest.mark.parametrize("T,E,k,H", ROUTING_CASES)
def test_init_routing_parity(moe, T, E, k, H):
    rng = np.random.default_rng(T + E + k)
    # skewed choice: some experts hot, some never chosen
    p = rng.dirichlet(np.full(E, 0.3))
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32) \
        if T * E <= 2_000_000 else rng.integers(0, E, size=(T, k)).astype(np.int32)
    x = mi.normal_bf16(1, 1, (T, H))
    counts, offsets, sp, pp = oracle.init_routing(idx, E)
    o = moe.moe_init_routing(dev(idx), E, dev_bf16(x))
    _torch().cuda.synchronize()
    assert (host(o["counts"]) == counts).all()
    assert (host(o["offsets"]) == offsets).all()
    assert (host(o["sorted_pair"]) == sp).all()
    assert (host(o["pair_pos"]) == pp).all()
    xe = host(o["x_exp"].view(_torch().int16)).view(np.uint16)
    assert (xe == oracle.expand_rows(x, sp, k)).all()
    assert moe.moe_get_device_status(o["ws"]) == 0


def test_init_routing_all_pairs_one_expert(moe):
    T, E, k = 5000, 16, 1
    idx = np.full((T, k), 11, np.int32)
    counts, offsets, sp, pp = oracle.init_routing(idx, E)
    o = moe.moe_init_routing(dev(idx), E)
    assert (host(o["counts"]) == counts).all() and (host(o["sorted_pair"]) == sp).all()
    assert (host(o["offsets"]) == offsets).all() and (host(o["pair_pos"]) == pp).all()


def test_init_routing_flags_bad_index(moe):
    idx = np.array([[0, 1], [2, 9]], np.int32)  # 9 >= E
    o = moe.moe_init_routing(dev(idx), 4)
    assert moe.moe_get_device_status(o["ws"]) == moe.MOE_ERR_DEVICE_CHECK


# ---------------------------------------------------------------- a3 / a4 grouped GEMMs
def _segments(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


GEMM_CASES = [
    # (counts per expert, H, I): narrow instance (few rows per expert) ...
    ([3, 0, 1, 7, 16, 17, 0, 32], 256, 128),
    ([1] * 40 + [0] * 24, 512, 192),
    ([5, 2, 0, 9], 4096, 1536),
    ([4, 0, 20, 3], 192, 64),
    # ... and the 256-wide instance (many rows per expert, ragged tails)
    ([300, 0, 1, 255, 256, 257, 40, 600], 256, 128),
    ([513, 64, 0, 1000], 1024, 256),
    ([400, 3, 0, 700, 17], 384, 192),  # feature tiles cut by I and by N
    # >= 256 rows per expert: compute-bound instance with 128-deep stages; K = 320 and 192
    # leave a last stage holding a single 64-deep chunk
    ([600, 0, 900, 257], 320, 192),
    # 240 experts: too many for the expert tables beside seven weight-streaming stages, so six
    ([40] * 120 + [37] * 100 + [0] * 20, 256, 128),
]


def _pack_ref(w13):
    """The packed gate/up layout written out from its definition (numpy indexing)."""
    E, twoI, H = w13.shape
    I = twoI // 2
    r = np.arange(twoI)
    g, q = r // 32, r % 32
    src = np.where(q < 16, 16 * g + q, I + 16 * g + q - 16)
    return w13[:, src, :]


@pytest.mark.parametrize("E,I,H", [(3, 128, 256), (2, 1536, 64), (1, 64, 128)])
def test_prepack_w13_is_the_packed_permutation(moe, E, I, H):
    w13 = mi.normal_bf16(E + I, 2, (E, 2 * I, H), 0.0, 0.02)
    got = moe.moe_prepack_w13(dev_bf16(w13))
    assert (host(got.view(_torch().int16)).view(np.uint16) == _pack_ref(w13)).all()


@pytest.mark.parametrize("counts,H,I", GEMM_CASES)
def test_grouped_gemm_swiglu_parity(moe, counts, H, I):
    E = len(counts)
    off = _segments(counts)
    M = int(off[-1])
    rng_seed = M + H + I
    x = mi.normal_bf16(rng_seed, 1, (M, H))
    w13 = mi.normal_bf16(rng_seed, 2, (E, 2 * I, H), 0.0, 0.02)
    ref = oracle.grouped_gemm_swiglu(x, w13, off)
    act = moe.moe_grouped_gemm_swiglu(dev_bf16(x), moe.moe_prepack_w13(dev_bf16(w13)), dev(off))
    got = host_bf16_f64(act)
    assert_close(got, ref, "act")
    assert_bf16_rounding_close(got, ref, "act")


# (T, k, E, H, I, zipf-like skew): the gate/up GEMM gathering its own rows through row_src, on
# each instance family: decode (<= 32 rows per expert, a separate gather kernel first),
# weight-streaming and compute-bound CTA pairs (< / >= 256 rows per expert, the gather inside the GEMM)
GATHER_CASES = [(16, 2, 8, 256, 128, 0.0), (300, 4, 16, 512, 128, 0.0), (1000, 4, 8, 512, 256, 0.3),
                (3000, 2, 6, 256, 128, 0.0), (37, 8, 64, 4096, 1536, 0.0), (1100, 8, 240, 256, 128, 0.0)]


@pytest.mark.parametrize("T,k,E,H,I,skew", GATHER_CASES)
def test_grouped_gemm_swiglu_gathers_its_rows(moe, T, k, E, H, I, skew):
    """act through row_src (the call gathers x[sorted_pair[pos] // k]) equals the oracle's GEMM on the
    oracle's expanded rows, and equals the call on pre-expanded rows bit for bit."""
    seed = T + E + H
    rng = np.random.default_rng(seed)
    p = np.exp(skew * rng.normal(size=E) * 3)
    p /= p.sum()
    idx = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]).astype(np.int32)
    counts, off, sp, _ = oracle.init_routing(idx, E)
    x = mi.normal_bf16(seed, 1, (T, H))
    w13 = mi.normal_bf16(seed, 2, (E, 2 * I, H), 0.0, 0.02)
    ref = oracle.grouped_gemm_swiglu(oracle.expand_rows(x, sp, k), w13, off)
    w13p = moe.moe_prepack_w13(dev_bf16(w13))
    ws = _torch().zeros(moe.lib().moe_grouped_gemm_swiglu_workspace_size(T * k, H, 1), dtype=_torch().uint8,
                        device="cuda")
    act = moe.moe_grouped_gemm_swiglu(dev_bf16(x), w13p, dev(off), ws=ws, row_src=dev(sp), k=k)
    assert moe.moe_get_device_status(ws) == moe.MOE_OK
    got = host_bf16_f64(act)
    assert_close(got, ref, "act (row_src)")
    assert_bf16_rounding_close(got, ref, "act (row_src)")
    pre = moe.moe_grouped_gemm_swiglu(dev_bf16(oracle.expand_rows(x, sp, k)), w13p, dev(off))
    assert _torch().equal(act.view(_torch().int16), pre.view(_torch().int16))


@pytest.mark.parametrize("T,E,bad", [(8, 4, 21), (300, 4, -1), (1200, 4, 2405)],
                         ids=["decode", "streaming", "compute-bound"])
def test_grouped_gemm_swiglu_flags_bad_row_src(moe, T, E, bad):
    """A source row outside [0, T*k) is reported (its row of act is unspecified) on each instance
    family, by the separate gather kernel (decode) or the gather inside the GEMM (CTA pairs),
    without stalling the GEMM; every other row is still right."""
    torch = _torch()
    k, H, I = 2, 256, 128
    idx = np.array([[e % E, (e + 1) % E] for e in range(T)], np.int32)
    _, off, sp, _ = oracle.init_routing(idx, E)
    sp = sp.copy()
    sp[3] = bad  # outside [0, T*k)
    x = mi.normal_bf16(3, 1, (T, H))
    w13 = mi.normal_bf16(3, 2, (E, 2 * I, H), 0.0, 0.02)
    ws = torch.zeros(moe.lib().moe_grouped_gemm_swiglu_workspace_size(T * k, H, 1), dtype=torch.uint8, device="cuda")
    act = moe.moe_grouped_gemm_swiglu(dev_bf16(x), moe.moe_prepack_w13(dev_bf16(w13)), dev(off), ws=ws,
                                      row_src=dev(sp), k=k)
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_DEVICE_CHECK
    sp_ok = sp.copy()
    sp_ok[3] = 0
    ref = oracle.grouped_gemm_swiglu(oracle.expand_rows(x, sp_ok, k), w13, off)
    keep = np.arange(T * k) != 3
    assert_close(host_bf16_f64(act)[keep], ref[keep], "act rows with a valid source")


@pytest.mark.parametrize("counts,H,I", GEMM_CASES)
def test_grouped_gemm_down_parity(moe, counts, H, I):
    E = len(counts)
    off = _segments(counts)
    M = int(off[-1])
    seed = 7 + M + H
    a = mi.normal_bf16(seed, 1, (M, I), 0.0, 0.5)
    w2 = mi.normal_bf16(seed, 3, (E, H, I), 0.0, 0.02)
    T = M
    topk_w = (np.abs(mi.normal_f32(seed, 5, (T, 1))) + 0.1).astype(np.float32)
    sorted_pair = np.random.default_rng(seed).permutation(M).astype(np.int32)
    ref = oracle.grouped_gemm(a, w2, off, topk_w.reshape(-1)[sorted_pair])
    out = moe.moe_grouped_gemm(dev_bf16(a), dev_bf16(w2), dev(off), dev(topk_w), dev(sorted_pair))
    got = host_bf16_f64(out)
    assert_close(got, ref, "y_perm")
    assert_bf16_rounding_close(got, ref, "y_perm")
    # without routing weights
    ref1 = oracle.grouped_gemm(a, w2, off)
    got1 = host_bf16_f64(moe.moe_grouped_gemm(dev_bf16(a), dev_bf16(w2), dev(off)))
    assert_bf16_rounding_close(got1, ref1, "plain")


def test_grouped_gemm_rejects_inconsistent_offsets(moe):
    torch = _torch()
    off = np.array([0, 5, 3, 8], np.int32)  # decreasing: invalid
    x = mi.normal_bf16(0, 1, (8, 256))
    w13 = mi.normal_bf16(0, 2, (3, 256, 256), 0.0, 0.02)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    act = torch.full((8, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_gemm_swiglu(dev_bf16(x), dev_bf16(w13), dev(off), act=act, ws=ws)
    assert moe.moe_get_device_status(ws) == moe.MOE_ERR_DEVICE_CHECK
    assert (act.float() == 7.0).all()  # nothing written


# ---------------------------------------------------------------- a6 finalize
@pytest.mark.parametrize("T,k,H,shared", [(16, 2, 256, False), (64, 8, 4096, False), (16, 8, 4096, True),
                                          (1000, 3, 192, True), (1, 1, 64, False)])
def test_finalize_parity(moe, T, k, H, shared):
    P = T * k
    y_perm = mi.normal_bf16(T, 1, (P, H))
    pair_pos = np.random.default_rng(T).permutation(P).astype(np.int32)
    s = mi.normal_bf16(T, 2, (T, H)) if shared else None
    ref = oracle.finalize_routing(y_perm, pair_pos, T, k, s)
    y = moe.moe_finalize_routing(dev_bf16(y_perm), dev(pair_pos), T, k, dev_bf16(s) if shared else None)
    got = host_bf16_f64(y)
    assert_close(got, ref, "y")
    assert_bf16_rounding_close(got, ref, "y")
