"""The C-ABI library builds, loads and exports every symbol include/moe.h declares.

No compute call here: only host-side queries and argument validation, which
returns before anything touches a GPU.
"""
import ctypes
import os
import re
import subprocess

import pytest

import moe_inputs as mi
import moe_expert_layer_fwd_gb300 as moe
from moe_expert_layer_fwd_gb300 import build as moe_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def L():
    moe_build.build()
    return moe.lib()


def _declared():
    with open(HEADER) as f:
        return re.findall(r"^MOE_API [^(]*?\b(moe_\w+)\(", f.read(), flags=re.M)


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert len(names) >= 15
    out = subprocess.run(["nm", "-D", "--defined-only", moe.LIB_PATH], capture_output=True, text=True, check=True)
    exported = set(re.findall(r"\bT (moe_\w+)", out.stdout))
    assert set(names) <= exported, set(names) - exported
    for n in names:
        assert hasattr(L, n)
    # the binding declares a signature for every symbol of the header
    assert set(names) == set(moe._SIGS)


def test_version_and_status_strings(L):
    assert moe.lib().moe_abi_version() == 200
    assert moe.status_string(0) == "MOE_OK"
    assert moe.status_string(-1) == "MOE_ERR_INVALID_ARG"
    assert moe.status_string(-5) == "MOE_ERR_TIMEOUT"
    assert moe.status_string(123) == "MOE_ERR_UNKNOWN"
    assert moe.lib().moe_status_bytes() == 256


@pytest.mark.parametrize("name", list(mi.CONFIGS))
def test_workspace_sizes(L, name):
    c = mi.CONFIGS[name]
    d = moe.make_desc(c.T, c.H, c.E, c.k, c.I, c.gate, c.routed_scaling_factor, c.eps, c.n_shared, c.I_s)
    n = moe.moe_layer_workspace_size(d)
    P = c.T * c.k
    # at least x_exp, act, y_perm and the permutation
    assert n >= P * (2 * c.H + c.I) * 2 + 2 * P * 4
    offs = moe.moe_layer_workspace_offsets(d)
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert L.moe_init_routing_workspace_size(c.T, c.E, c.k) >= 256


def test_layer_kernel_launches(L):
    # decode-sized (T*k <= 4096): gating + routing in one kernel, row gather, two GEMMs, finalize
    assert L.moe_layer_kernel_launches(ctypes.byref(moe.make_desc(64, 4096, 128, 8, 1536))) == 5
    # larger: gating, routing (3), two GEMMs (the gate/up GEMM gathers its own rows), finalize
    assert L.moe_layer_kernel_launches(ctypes.byref(moe.make_desc(4096, 4096, 192, 8, 1536))) == 7
    # compute-bound (>= 256 rows per expert): the gate/up GEMM gathers its own rows
    assert L.moe_layer_kernel_launches(ctypes.byref(moe.make_desc(16384, 2048, 128, 8, 768))) == 7
    assert L.moe_layer_kernel_launches(ctypes.byref(moe.make_desc(1024, 256, 8, 4, 128))) == 7
    # shared expert with I_s != I: one more down GEMM launch
    d = moe.make_desc(16, 4096, 192, 8, 1536, gate="sigmoid", n_shared=1, I_s=1024)
    assert L.moe_layer_kernel_launches(ctypes.byref(d)) == 6


def test_desc_validation(L):
    bad = [moe.make_desc(16, 100, 8, 2, 128),      # H % 64
           moe.make_desc(16, 256, 8, 9, 128),      # k > E
           moe.make_desc(16, 256, 2000, 2, 128),   # E > 1024
           moe.make_desc(16, 256, 8, 2, 96),       # I % 64
           moe.make_desc(-1, 256, 8, 2, 128)]
    for d in bad:
        assert L.moe_layer_workspace_size(ctypes.byref(d)) == 0
    d = moe.make_desc(16, 256, 8, 2, 128, gate=7)
    assert L.moe_layer_workspace_size(ctypes.byref(d)) == 0


def test_gating_validation_returns_before_launch(L):
    P16 = 16  # an aligned non-null dummy address: never dereferenced since validation fails first
    assert L.moe_gating_topk(P16, None, 4, 8, 9, 0, 1.0, 1e-20, P16, P16, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_gating_topk(P16, None, 4, 8, 2, 5, 1.0, 1e-20, P16, P16, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_gating_topk(P16, None, 4, 8, 2, 3, 1.0, 1e-20, P16, P16, None) == moe.MOE_ERR_INVALID_ARG
    # the three gates pass validation (an empty batch then returns without a launch)
    for gate in (0, 1, 2):
        assert L.moe_gating_topk(None, None, 0, 8, 2, gate, 1.0, 1e-20, None, None, None) == moe.MOE_OK
    assert L.moe_gating_topk(None, P16, 0, 8, 2, 2, 2.826, 1e-20, None, None, None) == moe.MOE_OK
    assert L.moe_gating_topk(P16, P16, 4, 8, 2, 0, 1.0, 1e-20, P16, P16, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_gating_topk(None, None, 4, 8, 2, 0, 1.0, 1e-20, P16, P16, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_gating_topk(P16 + 4, None, 4, 8, 2, 0, 1.0, 1e-20, P16, P16, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_gating_topk(P16, None, 4, 0, 1, 0, 1.0, 1e-20, P16, P16, None) == moe.MOE_ERR_INVALID_ARG
    # empty input: nothing to do
    assert L.moe_gating_topk(None, None, 0, 8, 2, 0, 1.0, 1e-20, None, None, None) == moe.MOE_OK


def test_routing_and_gemm_validation(L):
    P16 = 16
    small = L.moe_init_routing_workspace_size(4, 8, 2)
    assert L.moe_init_routing(P16, 4, 8, 2, None, 0, None, P16, P16, P16, P16, P16, small - 1, None) == \
        moe.MOE_ERR_WORKSPACE
    assert L.moe_init_routing(P16, 4, 8, 2, P16, 0, None, P16, P16, P16, P16, P16, small, None) == \
        moe.MOE_ERR_INVALID_ARG  # x without x_exp
    # moe_grouped_gemm_swiglu(x, row_src, k, T, w13, offsets, E, M, H, I, act, ws, ws_bytes, stream)
    assert L.moe_grouped_gemm_swiglu(P16, None, 1, 0, P16, P16, 8, 32, 100, 128, P16, P16, 256, None) == \
        moe.MOE_ERR_UNSUPPORTED
    assert L.moe_grouped_gemm_swiglu(P16, None, 1, 0, P16, P16, 8, 32, 256, 128, P16, P16, 255, None) == \
        moe.MOE_ERR_WORKSPACE
    # with row_src the workspace also holds the gathered rows and their flags
    need = L.moe_grouped_gemm_swiglu_workspace_size(32, 256, 1)
    assert need >= L.moe_status_bytes() + 32 * 256 * 2 + 8
    assert L.moe_grouped_gemm_swiglu_workspace_size(32, 256, 0) == L.moe_status_bytes()
    assert L.moe_grouped_gemm_swiglu(P16, P16, 8, 4, P16, P16, 8, 32, 256, 128, P16, P16, need - 1, None) == \
        moe.MOE_ERR_WORKSPACE
    assert L.moe_grouped_gemm_swiglu(P16, P16, 0, 4, P16, P16, 8, 32, 256, 128, P16, P16, need, None) == \
        moe.MOE_ERR_INVALID_ARG  # k < 1
    assert L.moe_grouped_gemm_swiglu(P16, P16 + 4, 8, 4, P16, P16, 8, 32, 256, 128, P16, P16, need, None) == \
        moe.MOE_ERR_INVALID_ARG  # misaligned row_src
    assert L.moe_grouped_gemm(P16, P16, P16, P16, None, 8, 32, 256, 128, P16, P16, 256, None) == \
        moe.MOE_ERR_INVALID_ARG  # topk_w without sorted_pair
    assert L.moe_grouped_gemm(P16, P16, P16, None, None, 8, 0, 256, 128, P16, P16, 256, None) == moe.MOE_OK
    assert L.moe_finalize_routing(P16, P16, None, 4, 33, 256, P16, None) == moe.MOE_ERR_UNSUPPORTED


def test_layer_forward_validation(L):
    d = moe.make_desc(16, 256, 8, 2, 128)
    need = L.moe_layer_workspace_size(ctypes.byref(d))
    P16 = 16
    args = [P16] * 11
    args[2] = None  # no bias (softmax)
    assert L.moe_layer_forward(ctypes.byref(d), *args, P16, need - 1, None) == moe.MOE_ERR_WORKSPACE
    a = list(args)
    a[2] = P16  # bias given with softmax gating
    assert L.moe_layer_forward(ctypes.byref(d), *a, P16, need, None) == moe.MOE_ERR_INVALID_ARG
    a = list(args)
    a[2] = None
    a[3] = None  # w13 missing
    assert L.moe_layer_forward(ctypes.byref(d), *a, P16, need, None) == moe.MOE_ERR_INVALID_ARG
    ds = moe.make_desc(16, 256, 8, 2, 128, gate="sigmoid", n_shared=1, I_s=128)
    need_s = L.moe_layer_workspace_size(ctypes.byref(ds))
    a = list(args)
    a[5] = None  # shared expert weights missing
    assert L.moe_layer_forward(ctypes.byref(ds), *a, P16, need_s, None) == moe.MOE_ERR_INVALID_ARG


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(moe, "LIB_PATH", str(tmp_path / "nope.so"))
    monkeypatch.setattr(moe, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        moe.lib()


def test_front_end_validation_returns_before_launch(L):
    P16 = 16  # an aligned non-null dummy address: never dereferenced since validation fails first
    # moe_add_rms_norm_cast(hidden, residual, weight, T, H, eps, y32, y16, residual_out, stream)
    assert L.moe_add_rms_norm_cast(P16, None, P16, 4, 100, 1e-6, P16, P16, None, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_add_rms_norm_cast(P16, None, P16, 4, 16384, 1e-6, P16, P16, None, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_add_rms_norm_cast(P16, P16, P16, 4, 256, 1e-6, P16, P16, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_add_rms_norm_cast(P16, None, P16, 4, 256, -1.0, P16, P16, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_add_rms_norm_cast(P16 + 4, None, P16, 4, 256, 1e-6, P16, P16, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_add_rms_norm_cast(None, None, None, 0, 256, 1e-6, None, None, None, None) == moe.MOE_OK
    # moe_router_logits(y32, w_gate, T, H, E, logits, stream)
    assert L.moe_router_logits(P16, P16, 4, 100, 8, P16, P16, 1 << 20, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_router_logits(P16, P16, 4, 256, 2000, P16, P16, 1 << 20, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_router_logits(P16, None, 4, 256, 8, P16, P16, 1 << 20, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_router_logits(P16, P16, 4, 256, 8, P16, P16, 0, None) == moe.MOE_ERR_WORKSPACE
    assert L.moe_router_logits(None, None, 0, 256, 8, None, None, 0, None) == moe.MOE_OK
    assert L.moe_router_logits_workspace_size(64, 4096, 128) >= L.moe_status_bytes()


def test_debug_set_validation(L):
    assert L.moe_debug_set(3, 0) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_debug_set(1, 0) == moe.MOE_OK and L.moe_debug_set(2, 0) == moe.MOE_OK


def test_mxfp4_validation_returns_before_launch(L):
    P16 = 1 << 20
    E = moe.MOE_ERR_INVALID_ARG
    U = moe.MOE_ERR_UNSUPPORTED
    assert L.moe_mxfp4_quantize(P16, 4, 48, P16, P16, None) == U            # K % 32
    assert L.moe_mxfp4_quantize(P16, -1, 64, P16, P16, None) == E
    assert L.moe_mxfp4_quantize(P16 + 4, 4, 64, P16, P16, None) == E        # misaligned weights
    assert L.moe_mxfp4_quantize(P16, 0, 64, None, None, None) == moe.MOE_OK  # nothing to do
    assert L.moe_mxfp4_prepack(P16, P16, 2, 192, 256, 1, P16 * 2, P16 * 3, P16 * 4, None) == U  # n_out % 128
    assert L.moe_mxfp4_prepack(P16, P16, 2, 256, 96, 1, P16 * 2, P16 * 3, P16 * 4, None) == U   # K % 64
    assert L.moe_mxfp4_prepack(P16, P16, 2, 256, 256, 1, P16, P16 * 3, P16 * 4, None) == E      # in place
    assert L.moe_gather_rows_f16(P16, P16, 4, 2, 100, 8, P16, P16, 256, None) == U             # H % 64
    assert L.moe_gather_rows_f16(P16, P16, 4, 2, 128, 8, P16, P16, 16, None) == moe.MOE_ERR_WORKSPACE
    assert L.moe_grouped_gemm_swiglu_mxfp4(P16, P16, P16, P16, P16, 8, 32, 100, 128, P16, P16, 256, None) == U
    assert L.moe_grouped_gemm_swiglu_mxfp4(P16, P16, P16, P16, P16, 2000, 32, 256, 128, P16, P16, 256, None) == U
    assert L.moe_grouped_gemm_mxfp4(P16, P16, P16, P16, P16, P16, None, 8, 32, 256, 128, P16, P16, 256, None) == E
    assert L.moe_grouped_gemm_mxfp4(P16, P16, P16, P16, P16, None, None, 8, 32, 192, 128, P16, P16, 256, None) == U
    assert L.moe_grouped_gemm_mxfp4(P16, P16, P16, None, P16, None, None, 8, 32, 256, 128, P16, P16, 256, None) == E


def test_mxfp4_weights_expert_slice_is_a_view_of_the_local_rows():
    import torch
    E, n_out, K = 5, 256, 128
    codes = torch.arange(E * n_out * K // 2, dtype=torch.int64).to(torch.uint8).view(E * n_out, K // 2)
    scales = torch.arange(E * n_out * K // 32, dtype=torch.int64).to(torch.uint8).view(E * n_out // 128, K // 32, 128)
    omega = torch.arange(E * n_out, dtype=torch.float32)
    w = moe.Mxfp4Weights(codes, scales, omega, E, n_out, K)
    loc = w.experts(1, 3)
    assert (loc.E, loc.n_out, loc.K) == (2, n_out, K)
    assert loc.codes.data_ptr() == codes.data_ptr() + 1 * n_out * (K // 2)
    assert loc.scales.data_ptr() == scales.data_ptr() + 1 * n_out * (K // 32)
    assert loc.omega.data_ptr() == omega.data_ptr() + 1 * n_out * 4
    assert loc.codes.is_contiguous() and loc.scales.is_contiguous() and loc.omega.is_contiguous()
    assert torch.equal(loc.omega, omega[n_out:3 * n_out])
    with pytest.raises(ValueError):
        w.experts(3, 3)
    with pytest.raises(ValueError):
        w.experts(0, 6)


def test_w4a8_validation_returns_before_launch(L):
    P16 = 1 << 20
    E = moe.MOE_ERR_INVALID_ARG
    U = moe.MOE_ERR_UNSUPPORTED
    # moe_w4a8_prepack(codes, scales, E, n_out, K, gate_up, codes_p, sf_p, stream)
    assert L.moe_w4a8_prepack(P16, P16, 2, 128, 256, 1, P16 * 2, P16 * 3, None) == U   # n_out % 256
    assert L.moe_w4a8_prepack(P16, P16, 2, 256, 192, 0, P16 * 2, P16 * 3, None) == U   # K % 128
    assert L.moe_w4a8_prepack(P16, P16, 2, 256, 256, 0, P16, P16 * 3, None) == E       # in place
    # moe_gather_rows_mx(x_codes, x_scales, sorted_pair, T, k, H, M, out_codes, out_sf, ws, ws_bytes, stream)
    assert L.moe_gather_rows_mx(P16, P16, P16, 4, 2, 192, 8, P16, P16, P16, 256, None) == U        # H % 128
    assert L.moe_gather_rows_mx(P16, P16, None, 4, 1, 256, 8, None, P16, P16, 256, None) == E      # M > T, identity
    assert L.moe_gather_rows_mx(P16, P16, P16, 4, 2, 256, 8, P16, P16, P16, 16, None) == moe.MOE_ERR_WORKSPACE
    # moe_grouped_gemm_swiglu_w4a8(x, x_sf, codes, sf, offsets, E, M, H, I, act, act_sf, ws, ws_bytes, stream)
    assert L.moe_grouped_gemm_swiglu_w4a8(P16, P16, P16, P16, P16, 8, 32, 192, 128, P16, P16, P16, 256, None) == U
    assert L.moe_grouped_gemm_swiglu_w4a8(P16, P16, P16, P16, P16, 8, 32, 256, 64, P16, P16, P16, 256, None) == U
    assert L.moe_grouped_gemm_swiglu_w4a8(P16, P16, P16, P16, P16, 8, 32, 256, 128, None, P16, P16, 256, None) == E
    # moe_grouped_gemm_w4a8(a, a_sf, codes, sf, offsets, topk_w, sorted_pair, E, M, N, K, out, ws, ws_bytes, stream)
    assert L.moe_grouped_gemm_w4a8(P16, P16, P16, P16, P16, P16, None, 8, 32, 256, 128, P16, P16, 256, None) == E
    assert L.moe_grouped_gemm_w4a8(P16, P16, P16, P16, P16, None, None, 8, 32, 192, 128, P16, P16, 256, None) == U
    assert L.moe_grouped_gemm_w4a8(P16, P16, P16, P16, P16, None, None, 8, 0, 256, 128, None, P16, 256, None) == \
        moe.MOE_OK
    # the layer: H, I, I_s multiples of 128
    d = moe.make_desc(16, 256, 8, 2, 192)
    assert L.moe_w4a8_layer_workspace_size(ctypes.byref(d)) == 0
    d = moe.make_desc(16, 256, 8, 2, 128, gate="sigmoid", n_shared=1, I_s=128)
    need = L.moe_w4a8_layer_workspace_size(ctypes.byref(d))
    assert need > 16 * 2 * (256 + 128 + 512)
    # a small batch is gated and sorted by one kernel: 1 + row gathers 2 + GEMMs 2 + finalize 1
    assert L.moe_w4a8_layer_kernel_launches(ctypes.byref(d)) == 6
    big = moe.make_desc(4096, 256, 8, 2, 128, gate="sigmoid", n_shared=1, I_s=128)
    assert L.moe_w4a8_layer_kernel_launches(ctypes.byref(big)) == 9
    args = [P16] * 16  # x_codes ... counts (the workspace pointer follows)
    args[3] = None  # no bias
    assert L.moe_layer_forward_w4a8(ctypes.byref(d), *args, P16, need - 1, None) == moe.MOE_ERR_WORKSPACE
    a = list(args)
    a[8] = None  # shared expert weights missing
    assert L.moe_layer_forward_w4a8(ctypes.byref(d), *a, P16, need, None) == E
