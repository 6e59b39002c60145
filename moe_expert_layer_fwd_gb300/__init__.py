"""GB300 (sm_103a) sparse MoE expert-layer forward: Python binding of ``libmoe_gb300.so``.

Argument marshalling only: every step of the forward pass runs in the CUDA
kernels behind the C ABI declared in ``include/moe.h``.  PyTorch supplies
device memory and streams; there is no CPU fallback -- if the library is not
built, every call raises.

Functions carry the C names:

    moe_gating_topk, moe_init_routing, moe_grouped_gemm_swiglu, moe_grouped_gemm,
    moe_finalize_routing, moe_layer_forward (+ MoELayer, which owns a workspace); the front end
    moe_add_rms_norm_cast and moe_router_logits; moe_init_routing_range.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import NamedTuple, Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_gb300.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_WORKSPACE = -3
MOE_ERR_CUDA = -4
MOE_ERR_TIMEOUT = -5
MOE_ERR_DEVICE_CHECK = -6
GATES = {"softmax": 0, "sigmoid": 1, "sigmoid_inner_bias": 2}

_lib = None
_lock = threading.Lock()


class MoEError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what} failed: {status_string(status)} ({status})")


class moe_layer_desc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("I", ctypes.c_int32), ("gate", ctypes.c_int32), ("routed_scaling_factor", ctypes.c_float),
                ("eps", ctypes.c_float), ("n_shared", ctypes.c_int32), ("I_s", ctypes.c_int32)]


_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "moe_abi_version": (ctypes.c_int, []),
    "moe_status_bytes": (ctypes.c_size_t, []),
    "moe_workspace_init": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "moe_get_device_status": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p]),
    "moe_gating_topk": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_float, ctypes.c_float, ctypes.c_void_p,
                                       ctypes.c_void_p, ctypes.c_void_p]),
    "moe_init_routing_workspace_size": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "moe_init_routing": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                        ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                        ctypes.c_void_p]),
    "moe_init_routing_range": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "moe_init_routing_static_scratch": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                       ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p,
                                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                       ctypes.c_void_p, ctypes.c_void_p]),
    "moe_mxfp4_quantize": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_void_p]),
    "moe_mxfp4_prepack": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                         ctypes.c_void_p]),
    "moe_gather_rows_f16": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                           ctypes.c_void_p]),
    "moe_grouped_gemm_swiglu_mxfp4": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                     ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                                     ctypes.c_size_t, ctypes.c_void_p]),
    "moe_grouped_gemm_mxfp4": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "moe_w4a8_prepack": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "moe_gather_rows_mx": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                          ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "moe_grouped_gemm_swiglu_w4a8": (ctypes.c_int, [ctypes.c_void_p] * 5 + [ctypes.c_int] * 4 +
                                     [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t,
                                      ctypes.c_void_p]),
    "moe_grouped_gemm_w4a8": (ctypes.c_int, [ctypes.c_void_p] * 7 + [ctypes.c_int] * 4 +
                              [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "moe_w4a8_layer_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(moe_layer_desc)]),
    "moe_layer_forward_w4a8": (ctypes.c_int, [ctypes.POINTER(moe_layer_desc)] + [ctypes.c_void_p] * 17 +
                               [ctypes.c_size_t, ctypes.c_void_p]),
    "moe_layer_forward_w4a8_events": (ctypes.c_int, [ctypes.POINTER(moe_layer_desc)] + [ctypes.c_void_p] * 17 +
                                      [ctypes.c_size_t, ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p),
                                       ctypes.c_int]),
    "moe_w4a8_layer_kernel_launches": (ctypes.c_int, [ctypes.POINTER(moe_layer_desc)]),
    "moe_debug_set": (ctypes.c_int, [ctypes.c_int, ctypes.c_ulonglong]),
    "moe_add_rms_norm_cast": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                             ctypes.c_void_p, ctypes.c_void_p]),
    "moe_add_rms_norm_mxfp8": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p,
                                              ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]),
    "moe_router_logits_workspace_size": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "moe_router_logits": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "moe_prepack_w13": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                       ctypes.c_void_p]),
    "moe_grouped_gemm_workspace_size": (ctypes.c_size_t, []),
    "moe_grouped_gemm_swiglu_workspace_size": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int, ctypes.c_int]),
    "moe_grouped_gemm_swiglu": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                               ctypes.c_size_t, ctypes.c_void_p]),
    "moe_grouped_gemm": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                        ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "moe_finalize_routing": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]),
    "moe_layer_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(moe_layer_desc)]),
    "moe_layer_workspace_offsets": (ctypes.c_int, [ctypes.POINTER(moe_layer_desc),
                                                   ctypes.POINTER(ctypes.c_size_t), ctypes.c_int]),
    "moe_layer_forward": (ctypes.c_int, [ctypes.POINTER(moe_layer_desc)] + [ctypes.c_void_p] * 11 +
                          [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "moe_layer_forward_events": (ctypes.c_int, [ctypes.POINTER(moe_layer_desc)] + [ctypes.c_void_p] * 11 +
                                 [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                  ctypes.POINTER(ctypes.c_void_p), ctypes.c_int]),
    "moe_layer_kernel_launches": (ctypes.c_int, [ctypes.POINTER(moe_layer_desc)]),
}


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m moe_expert_layer_fwd_gb300.build`"
                                   " (there is no CPU fallback)")
            l = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                f = getattr(l, name)
                f.restype = res
                f.argtypes = args
            _lib = l
    return _lib


def status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def _check(status: int, what: str) -> None:
    if status != MOE_OK:
        raise MoEError(status, what)


# ------------------------------------------------------------------ torch glue
def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _ws(nbytes: int, device, ws=None):
    torch = _torch()
    nbytes = max(int(nbytes), 256)
    if ws is None or ws.numel() < nbytes:
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=device)
    return ws


def moe_gating_topk(logits, k: int, gate: str = "softmax", bias=None, routed_scaling_factor: float = 1.0,
                    eps: float = 1e-20, topk_w=None, topk_idx=None, stream=None):
    """a1: returns (topk_w [T,k] fp32, topk_idx [T,k] int32)."""
    torch = _torch()
    T, E = logits.shape
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    if topk_idx is None:
        topk_idx = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    _check(lib().moe_gating_topk(_ptr(logits), _ptr(bias), T, E, k, GATES[gate], routed_scaling_factor, eps,
                                 _ptr(topk_w), _ptr(topk_idx), _stream(stream)), "moe_gating_topk")
    return topk_w, topk_idx


def moe_init_routing(topk_idx, E: int, x=None, ws=None, out: Optional[dict] = None, stream=None) -> dict:
    """a2: returns dict(counts, offsets, sorted_pair, pair_pos, x_exp (if x given), ws)."""
    torch = _torch()
    T, k = topk_idx.shape
    P = T * k
    dev = topk_idx.device
    o = dict(out or {})
    o.setdefault("counts", torch.empty(E, dtype=torch.int32, device=dev))
    o.setdefault("offsets", torch.empty(E + 1, dtype=torch.int32, device=dev))
    o.setdefault("sorted_pair", torch.empty(P, dtype=torch.int32, device=dev))
    o.setdefault("pair_pos", torch.empty(P, dtype=torch.int32, device=dev))
    H = 0
    if x is not None:
        H = x.shape[1]
        o.setdefault("x_exp", torch.empty((P, H), dtype=x.dtype, device=dev))
    need = lib().moe_init_routing_workspace_size(T, E, k)
    ws = _ws(need, dev, ws)
    _check(lib().moe_init_routing(_ptr(topk_idx), T, E, k, _ptr(x), H, _ptr(o.get("x_exp")), _ptr(o["counts"]),
                                  _ptr(o["offsets"]), _ptr(o["sorted_pair"]), _ptr(o["pair_pos"]), _ptr(ws),
                                  ws.numel(), _stream(stream)), "moe_init_routing")
    o["ws"] = ws
    return o


def moe_add_rms_norm_cast(hidden, residual, norm_weight, eps: float, y_fp32=None, y_bf16=None, residual_out=None,
                          stream=None):
    """Front end: returns (y_fp32 [T,H] fp32, y_bf16 [T,H] bf16, residual_out [T,H] bf16 or None)."""
    torch = _torch()
    T, H = hidden.shape
    dev = hidden.device
    if y_fp32 is None:
        y_fp32 = torch.empty((T, H), dtype=torch.float32, device=dev)
    if y_bf16 is None:
        y_bf16 = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    if residual is not None and residual_out is None:
        residual_out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    _check(lib().moe_add_rms_norm_cast(_ptr(hidden), _ptr(residual), _ptr(norm_weight), T, H, eps, _ptr(y_fp32),
                                       _ptr(y_bf16), _ptr(residual_out), _stream(stream)), "moe_add_rms_norm_cast")
    return y_fp32, y_bf16, residual_out


def moe_add_rms_norm_mxfp8(hidden, residual, norm_weight, eps: float, with_fp32: bool = True, stream=None):
    """W4A8 front end: returns (codes [T,H] uint8 E4M3, scales [T,H/32] uint8 E8M0, y_fp32 or None,
    residual_out or None)."""
    torch = _torch()
    T, H = hidden.shape
    dev = hidden.device
    codes = torch.empty((T, H), dtype=torch.uint8, device=dev)
    scales = torch.empty((T, H // 32), dtype=torch.uint8, device=dev)
    y32 = torch.empty((T, H), dtype=torch.float32, device=dev) if with_fp32 else None
    r_out = torch.empty((T, H), dtype=torch.bfloat16, device=dev) if residual is not None else None
    _check(lib().moe_add_rms_norm_mxfp8(_ptr(hidden), _ptr(residual), _ptr(norm_weight), T, H, eps, _ptr(codes),
                                        _ptr(scales), _ptr(y32), _ptr(r_out), _stream(stream)),
           "moe_add_rms_norm_mxfp8")
    return codes, scales, y32, r_out


def moe_router_logits(y_fp32, w_gate, logits=None, ws=None, stream=None):
    """Router gate GEMM: logits[T,E] = y_fp32 . w_gate^T in fp32 (w_gate [E,H] bf16)."""
    torch = _torch()
    T, H = y_fp32.shape
    E = w_gate.shape[0]
    if logits is None:
        logits = torch.empty((T, E), dtype=torch.float32, device=y_fp32.device)
    ws = _ws(lib().moe_router_logits_workspace_size(T, H, E), y_fp32.device, ws)
    _check(lib().moe_router_logits(_ptr(y_fp32), _ptr(w_gate), T, H, E, _ptr(logits), _ptr(ws), ws.numel(),
                                   _stream(stream)), "moe_router_logits")
    return logits


def moe_init_routing_range(topk_idx, E: int, e0: int, e1: int, x=None, ws=None, out: Optional[dict] = None,
                           stream=None) -> dict:
    """a2 restricted to the local experts [e0, e1): counts/offsets over e1-e0 experts, sorted_pair
    holding the local pairs first (offsets[-1] of them), pair_pos -1 for pairs routed elsewhere."""
    torch = _torch()
    T, k = topk_idx.shape
    P = T * k
    EL = e1 - e0
    dev = topk_idx.device
    o = dict(out or {})
    o.setdefault("counts", torch.empty(max(EL, 0), dtype=torch.int32, device=dev))
    o.setdefault("offsets", torch.empty(max(EL, 0) + 1, dtype=torch.int32, device=dev))
    o.setdefault("sorted_pair", torch.empty(P, dtype=torch.int32, device=dev))
    o.setdefault("pair_pos", torch.empty(P, dtype=torch.int32, device=dev))
    H = 0
    if x is not None:
        H = x.shape[1]
        o.setdefault("x_exp", torch.empty((P, H), dtype=x.dtype, device=dev))
    need = lib().moe_init_routing_workspace_size(T, E, k)
    ws = _ws(need, dev, ws)
    _check(lib().moe_init_routing_range(_ptr(topk_idx), T, E, k, e0, e1, _ptr(x), H, _ptr(o.get("x_exp")),
                                        _ptr(o["counts"]), _ptr(o["offsets"]), _ptr(o["sorted_pair"]),
                                        _ptr(o["pair_pos"]), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_init_routing_range")
    o["ws"] = ws
    return o


def moe_init_routing_static_scratch(topk_idx, E: int, x=None, out: Optional[dict] = None, stream=None) -> dict:
    """a2 without a workspace (scratch in a fixed device array inside the library; see include/moe.h).
    Only the output tensors passed in `out` are used as given; missing ones are created here."""
    torch = _torch()
    T, k = topk_idx.shape
    P = T * k
    dev = topk_idx.device
    o = dict(out or {})
    o.setdefault("counts", torch.empty(E, dtype=torch.int32, device=dev))
    o.setdefault("offsets", torch.empty(E + 1, dtype=torch.int32, device=dev))
    o.setdefault("sorted_pair", torch.empty(P, dtype=torch.int32, device=dev))
    o.setdefault("pair_pos", torch.empty(P, dtype=torch.int32, device=dev))
    H = 0
    if x is not None:
        H = x.shape[1]
        o.setdefault("x_exp", torch.empty((P, H), dtype=x.dtype, device=dev))
    _check(lib().moe_init_routing_static_scratch(_ptr(topk_idx), T, E, k, _ptr(x), H, _ptr(o.get("x_exp")),
                                                 _ptr(o["counts"]), _ptr(o["offsets"]), _ptr(o["sorted_pair"]),
                                                 _ptr(o["pair_pos"]), _stream(stream)),
           "moe_init_routing_static_scratch")
    return o


def moe_prepack_w13(w13, out=None, stream=None):
    """w13 [E,2I,H] (or [2I,H]) rows [gate; up] -> the packed gate/up layout the GEMMs read."""
    torch = _torch()
    shape = w13.shape
    E, twoI, H = (1, shape[0], shape[1]) if w13.dim() == 2 else shape
    if out is None:
        out = torch.empty_like(w13)
    _check(lib().moe_prepack_w13(_ptr(w13), E, twoI // 2, H, _ptr(out), _stream(stream)), "moe_prepack_w13")
    return out


def moe_grouped_gemm_swiglu(x, w13, offsets, act=None, ws=None, row_src=None, k: int = 1, M: Optional[int] = None,
                            stream=None):
    """a3: act[M,I] = SwiGLU(row(pos) . w13[e]^T) per expert segment; w13 packed by moe_prepack_w13.

    row_src None: x [M,H] holds the rows in expert-sorted order.  row_src given (sorted_pair of
    init-routing): x [T,H] holds the token rows and row pos is x[row_src[pos] // k], gathered by the
    call (M defaults to row_src's length)."""
    torch = _torch()
    E, twoI, H = w13.shape
    I = twoI // 2
    if row_src is None:
        M, T = x.shape[0], 0
    else:
        T = x.shape[0]
        M = row_src.numel() if M is None else M
    if act is None:
        act = torch.empty((M, I), dtype=torch.bfloat16, device=x.device)
    gather = row_src is not None
    ws = _ws(lib().moe_grouped_gemm_swiglu_workspace_size(M, H, int(gather)), x.device, ws)
    _check(lib().moe_grouped_gemm_swiglu(_ptr(x), _ptr(row_src), k, T, _ptr(w13), _ptr(offsets), E, M, H, I,
                                         _ptr(act), _ptr(ws), ws.numel(), _stream(stream)),
           "moe_grouped_gemm_swiglu")
    return act


def moe_grouped_gemm(a, w, offsets, topk_w=None, sorted_pair=None, out=None, ws=None, stream=None):
    """a4: out[M,N] = scale * (a . w[e]^T) per expert segment."""
    torch = _torch()
    M, K = a.shape
    E, N, _ = w.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    ws = _ws(lib().moe_grouped_gemm_workspace_size(), a.device, ws)
    _check(lib().moe_grouped_gemm(_ptr(a), _ptr(w), _ptr(offsets), _ptr(topk_w), _ptr(sorted_pair), E, M, N, K,
                                  _ptr(out), _ptr(ws), ws.numel(), _stream(stream)), "moe_grouped_gemm")
    return out


# ------------------------------------------------------------------ MXFP4 expert weights (decode)
class Mxfp4Weights(NamedTuple):
    """Expert weights [E, n_out, K] in the kernel layout of moe_mxfp4_prepack."""
    codes: object    # [E*n_out, K/2] uint8
    scales: object   # [E*n_out/128, K/32, 128] uint8
    omega: object    # [E*n_out] float32
    E: int
    n_out: int
    K: int

    def experts(self, e0: int, e1: int) -> "Mxfp4Weights":
        """The local experts [e0, e1) as views (no copy): the weights the 4-bit GEMMs take together
        with the offsets of moe_init_routing_range (every expert owns whole 128-row tiles)."""
        if not 0 <= e0 < e1 <= self.E:
            raise ValueError(f"expert range [{e0}, {e1}) outside [0, {self.E})")
        r0, r1 = e0 * self.n_out, e1 * self.n_out
        return Mxfp4Weights(self.codes[r0:r1], self.scales[r0 // 128:r1 // 128], self.omega[r0:r1], e1 - e0,
                            self.n_out, self.K)


def moe_mxfp4_quantize(w, stream=None):
    """w [..., K] bf16 -> (codes uint8 [..., K/2], scales uint8 [..., K/32]), the OCP MXFP4 encoding."""
    torch = _torch()
    K = w.shape[-1]
    rows = w.numel() // K if K else 0
    codes = torch.empty((*w.shape[:-1], K // 2), dtype=torch.uint8, device=w.device)
    scales = torch.empty((*w.shape[:-1], K // 32), dtype=torch.uint8, device=w.device)
    _check(lib().moe_mxfp4_quantize(_ptr(w), rows, K, _ptr(codes), _ptr(scales), _stream(stream)),
           "moe_mxfp4_quantize")
    return codes, scales


def moe_mxfp4_prepack(codes, scales, gate_up: bool, stream=None) -> Mxfp4Weights:
    """codes [E,n_out,K/2], scales [E,n_out,K/32] -> the layout the 4-bit GEMMs read (gate_up: w13)."""
    torch = _torch()
    if codes.dim() == 2:
        codes, scales = codes.unsqueeze(0), scales.unsqueeze(0)
    E, n_out, K2 = codes.shape
    K = 2 * K2
    dev = codes.device
    cp = torch.empty((E * n_out, K2), dtype=torch.uint8, device=dev)
    sp = torch.empty((E * n_out // 128, K // 32, 128), dtype=torch.uint8, device=dev)
    om = torch.empty((E * n_out,), dtype=torch.float32, device=dev)
    _check(lib().moe_mxfp4_prepack(_ptr(codes), _ptr(scales), E, n_out, K, int(bool(gate_up)), _ptr(cp), _ptr(sp),
                                   _ptr(om), _stream(stream)), "moe_mxfp4_prepack")
    return Mxfp4Weights(cp, sp, om, E, n_out, K)


def moe_gather_rows_f16(x, sorted_pair, k: int, M: Optional[int] = None, out=None, ws=None, stream=None):
    """x_rows16[pos] = f16(x[sorted_pair[pos] // k]) for pos < M (default: all of sorted_pair)."""
    torch = _torch()
    T, H = x.shape
    M = sorted_pair.numel() if M is None else M
    if out is None:
        out = torch.empty((M, H), dtype=torch.float16, device=x.device)
    ws = _ws(lib().moe_grouped_gemm_workspace_size(), x.device, ws)
    _check(lib().moe_gather_rows_f16(_ptr(x), _ptr(sorted_pair), T, k, H, M, _ptr(out), _ptr(ws), ws.numel(),
                                     _stream(stream)), "moe_gather_rows_f16")
    return out


def moe_grouped_gemm_swiglu_mxfp4(x_rows16, w13: Mxfp4Weights, offsets, act=None, ws=None, stream=None):
    """a3 on MXFP4 weights: act16[M,I] = SwiGLU(x_rows16 . dequant(w13[e])^T)."""
    torch = _torch()
    M, H = x_rows16.shape
    I = w13.n_out // 2
    if act is None:
        act = torch.empty((M, I), dtype=torch.float16, device=x_rows16.device)
    ws = _ws(lib().moe_grouped_gemm_workspace_size(), x_rows16.device, ws)
    _check(lib().moe_grouped_gemm_swiglu_mxfp4(_ptr(x_rows16), _ptr(w13.codes), _ptr(w13.scales), _ptr(w13.omega),
                                               _ptr(offsets), w13.E, M, H, I, _ptr(act), _ptr(ws), ws.numel(),
                                               _stream(stream)), "moe_grouped_gemm_swiglu_mxfp4")
    return act


def moe_grouped_gemm_mxfp4(a16, w: Mxfp4Weights, offsets, topk_w=None, sorted_pair=None, out=None, ws=None,
                           stream=None):
    """a4 on MXFP4 weights: out[M,N] (bf16) = scale * (a16 . dequant(w[e])^T)."""
    torch = _torch()
    M, K = a16.shape
    if out is None:
        out = torch.empty((M, w.n_out), dtype=torch.bfloat16, device=a16.device)
    ws = _ws(lib().moe_grouped_gemm_workspace_size(), a16.device, ws)
    _check(lib().moe_grouped_gemm_mxfp4(_ptr(a16), _ptr(w.codes), _ptr(w.scales), _ptr(w.omega), _ptr(offsets),
                                        _ptr(topk_w), _ptr(sorted_pair), w.E, M, w.n_out, K, _ptr(out), _ptr(ws),
                                        ws.numel(), _stream(stream)), "moe_grouped_gemm_mxfp4")
    return out


class Mxfp4Layer:
    """The decode layer on MXFP4 expert weights, composed from the C entry points on one stream:
    moe_gating_topk, moe_init_routing, moe_gather_rows_f16, moe_grouped_gemm_swiglu_mxfp4,
    moe_grouped_gemm_mxfp4, moe_finalize_routing (8 kernels), into buffers allocated once here.
    No shared expert (the 4-bit GEMMs cover the routed experts)."""

    KERNELS_PER_FORWARD = 8

    def __init__(self, T: int, H: int, E: int, k: int, I: int, gate: str = "softmax",
                 routed_scaling_factor: float = 1.0, eps: float = 1e-20, device="cuda"):
        torch = _torch()
        self.T, self.H, self.E, self.k, self.I = T, H, E, k, I
        self.gate, self.rsf, self.eps = gate, routed_scaling_factor, eps
        P = T * k
        self.topk_w = torch.empty((T, k), dtype=torch.float32, device=device)
        self.topk_idx = torch.empty((T, k), dtype=torch.int32, device=device)
        self.routing = dict(counts=torch.empty(E, dtype=torch.int32, device=device),
                            offsets=torch.empty(E + 1, dtype=torch.int32, device=device),
                            sorted_pair=torch.empty(P, dtype=torch.int32, device=device),
                            pair_pos=torch.empty(P, dtype=torch.int32, device=device))
        self.routing_ws = _ws(lib().moe_init_routing_workspace_size(T, E, k), device)
        self.ws = _ws(lib().moe_grouped_gemm_workspace_size(), device)
        self.x16 = torch.empty((P, H), dtype=torch.float16, device=device)
        self.act16 = torch.empty((P, I), dtype=torch.float16, device=device)
        self.y_perm = torch.empty((P, H), dtype=torch.bfloat16, device=device)
        self.y = torch.empty((T, H), dtype=torch.bfloat16, device=device)

    def forward(self, x, logits, w13: Mxfp4Weights, w2: Mxfp4Weights, bias=None, stream=None, events=None):
        """y [T,H] bf16.  events: optional list of 5 CUDA events recorded around the steps
        (gating + routing + gather | gate/up GEMM | down GEMM | finalize)."""
        s = stream
        r = self.routing

        def ev(i):
            if events is not None:
                events[i].record(s if s is not None else _torch().cuda.current_stream())

        ev(0)
        moe_gating_topk(logits, self.k, self.gate, bias, self.rsf, self.eps, self.topk_w, self.topk_idx, stream=s)
        moe_init_routing(self.topk_idx, self.E, ws=self.routing_ws, out=r, stream=s)
        moe_gather_rows_f16(x, r["sorted_pair"], self.k, out=self.x16, ws=self.ws, stream=s)
        ev(1)
        moe_grouped_gemm_swiglu_mxfp4(self.x16, w13, r["offsets"], act=self.act16, ws=self.ws, stream=s)
        ev(2)
        moe_grouped_gemm_mxfp4(self.act16, w2, r["offsets"], self.topk_w, r["sorted_pair"], out=self.y_perm,
                               ws=self.ws, stream=s)
        ev(3)
        moe_finalize_routing(self.y_perm, r["pair_pos"], self.T, self.k, y=self.y, stream=s)
        ev(4)
        return self.y


# ------------------------------------------------------------------ W4A8: MXFP8 x MXFP4 on the block-scaled MMA
class W4a8Weights(NamedTuple):
    """Expert weights [E, n_out, K] in the layout of moe_w4a8_prepack."""
    codes: object    # [E*n_out/256, K/128, 256, 64] uint8 E2M1 codes (gate/up rows regrouped for w13)
    sf: object       # [E*n_out/256, K/128, 2, 512] uint8 scale atoms
    E: int
    n_out: int
    K: int

    def experts(self, e0: int, e1: int) -> "W4a8Weights":
        """The local experts [e0, e1) as views (every expert owns whole 256-row tiles)."""
        if not 0 <= e0 < e1 <= self.E:
            raise ValueError(f"expert range [{e0}, {e1}) outside [0, {self.E})")
        r0, r1 = e0 * self.n_out, e1 * self.n_out
        return W4a8Weights(self.codes[r0 // 256:r1 // 256], self.sf[r0 // 256:r1 // 256], e1 - e0, self.n_out,
                           self.K)


def moe_w4a8_prepack(codes, scales, gate_up: bool, stream=None) -> W4a8Weights:
    """codes [E,n_out,K/2], scales [E,n_out,K/32] (moe_mxfp4_quantize) -> the W4A8 GEMMs' layout."""
    torch = _torch()
    if codes.dim() == 2:
        codes, scales = codes.unsqueeze(0), scales.unsqueeze(0)
    E, n_out, K2 = codes.shape
    K = 2 * K2
    dev = codes.device
    cp = torch.empty((E * n_out // 256, K // 128, 256, 64), dtype=torch.uint8, device=dev)
    sf = torch.empty((E * n_out // 256, K // 128, 2, 512), dtype=torch.uint8, device=dev)
    _check(lib().moe_w4a8_prepack(_ptr(codes), _ptr(scales), E, n_out, K, int(bool(gate_up)), _ptr(cp), _ptr(sf),
                                  _stream(stream)), "moe_w4a8_prepack")
    return W4a8Weights(cp, sf, E, n_out, K)


def moe_gather_rows_mx(x_codes, x_scales, sorted_pair=None, k: int = 1, M: Optional[int] = None, out_codes=None,
                       out_sf=None, ws=None, stream=None):
    """(out_codes [M,H] E4M3, out_sf [M,H/128,16] padded scale rows) of rows x[sorted_pair[pos] // k]
    (sorted_pair None: the first M token rows, scale rows only)."""
    torch = _torch()
    T, H = x_codes.shape
    if M is None:
        M = sorted_pair.numel() if sorted_pair is not None else T
    dev = x_codes.device
    if out_codes is None and sorted_pair is not None:
        out_codes = torch.empty((M, H), dtype=torch.uint8, device=dev)
    if out_sf is None:
        out_sf = torch.empty((M, H // 128, 16), dtype=torch.uint8, device=dev)
    ws = _ws(lib().moe_grouped_gemm_workspace_size(), dev, ws)
    _check(lib().moe_gather_rows_mx(_ptr(x_codes), _ptr(x_scales), _ptr(sorted_pair), T, k, H, M, _ptr(out_codes),
                                    _ptr(out_sf), _ptr(ws), ws.numel(), _stream(stream)), "moe_gather_rows_mx")
    return out_codes, out_sf


def moe_grouped_gemm_swiglu_w4a8(x, x_sf, w13: W4a8Weights, offsets, act=None, act_sf=None, ws=None, stream=None):
    """a3 in W4A8: (act [M,I] E4M3, act_sf [M,I/128,16]) = MXFP8(SwiGLU(x . w13[e]^T))."""
    torch = _torch()
    M, H = x.shape
    I = w13.n_out // 2
    if act is None:
        act = torch.empty((M, I), dtype=torch.uint8, device=x.device)
    if act_sf is None:
        act_sf = torch.empty((M, I // 128, 16), dtype=torch.uint8, device=x.device)
    ws = _ws(lib().moe_grouped_gemm_workspace_size(), x.device, ws)
    _check(lib().moe_grouped_gemm_swiglu_w4a8(_ptr(x), _ptr(x_sf), _ptr(w13.codes), _ptr(w13.sf), _ptr(offsets),
                                              w13.E, M, H, I, _ptr(act), _ptr(act_sf), _ptr(ws), ws.numel(),
                                              _stream(stream)), "moe_grouped_gemm_swiglu_w4a8")
    return act, act_sf


def moe_grouped_gemm_w4a8(a, a_sf, w: W4a8Weights, offsets, topk_w=None, sorted_pair=None, out=None, ws=None,
                          stream=None):
    """a4 in W4A8: out [M,N] bf16 = scale * (a . w[e]^T)."""
    torch = _torch()
    M, K = a.shape
    if out is None:
        out = torch.empty((M, w.n_out), dtype=torch.bfloat16, device=a.device)
    ws = _ws(lib().moe_grouped_gemm_workspace_size(), a.device, ws)
    _check(lib().moe_grouped_gemm_w4a8(_ptr(a), _ptr(a_sf), _ptr(w.codes), _ptr(w.sf), _ptr(offsets), _ptr(topk_w),
                                       _ptr(sorted_pair), w.E, M, w.n_out, K, _ptr(out), _ptr(ws), ws.numel(),
                                       _stream(stream)), "moe_grouped_gemm_w4a8")
    return out


class W4a8Layer:
    """One W4A8 layer shape (moe_layer_forward_w4a8) with its own workspace and output buffers."""

    def __init__(self, T, H, E, k, I, gate="softmax", routed_scaling_factor=1.0, eps=1e-20, n_shared=0, I_s=0,
                 device="cuda"):
        torch = _torch()
        self.desc = make_desc(T, H, E, k, I, gate, routed_scaling_factor, eps, n_shared, I_s)
        n = lib().moe_w4a8_layer_workspace_size(ctypes.byref(self.desc))
        if n == 0:
            raise MoEError(MOE_ERR_UNSUPPORTED, "moe_w4a8_layer_workspace_size")
        self.ws = torch.zeros(n, dtype=torch.uint8, device=device)
        self.y = torch.empty((T, H), dtype=torch.bfloat16, device=device)
        self.topk_w = torch.empty((T, k), dtype=torch.float32, device=device)
        self.topk_idx = torch.empty((T, k), dtype=torch.int32, device=device)
        self.counts = torch.empty(E, dtype=torch.int32, device=device)
        self.launches = lib().moe_w4a8_layer_kernel_launches(ctypes.byref(self.desc))

    def _args(self, x_codes, x_scales, logits, w13, w2, bias, w13_s, w2_s):
        return [_ptr(x_codes), _ptr(x_scales), _ptr(logits), _ptr(bias), _ptr(w13.codes), _ptr(w13.sf),
                _ptr(w2.codes), _ptr(w2.sf), _ptr(w13_s.codes) if w13_s else None, _ptr(w13_s.sf) if w13_s else None,
                _ptr(w2_s.codes) if w2_s else None, _ptr(w2_s.sf) if w2_s else None, _ptr(self.y),
                _ptr(self.topk_w), _ptr(self.topk_idx), _ptr(self.counts), _ptr(self.ws), self.ws.numel()]

    def forward(self, x_codes, x_scales, logits, w13: W4a8Weights, w2: W4a8Weights, bias=None, w13_s=None,
                w2_s=None, stream=None):
        _check(lib().moe_layer_forward_w4a8(ctypes.byref(self.desc),
                                            *self._args(x_codes, x_scales, logits, w13, w2, bias, w13_s, w2_s),
                                            _stream(stream)), "moe_layer_forward_w4a8")
        return self.y

    def forward_events(self, events, x_codes, x_scales, logits, w13, w2, bias=None, w13_s=None, w2_s=None,
                       stream=None):
        handles = (ctypes.c_void_p * 6)()
        for i, ev in enumerate(events):
            if ev.cuda_event == 0:
                ev.record()
            handles[i] = ev.cuda_event
        _check(lib().moe_layer_forward_w4a8_events(ctypes.byref(self.desc),
                                                   *self._args(x_codes, x_scales, logits, w13, w2, bias, w13_s, w2_s),
                                                   _stream(stream), handles, 6), "moe_layer_forward_w4a8_events")
        return self.y


def moe_finalize_routing(y_perm, pair_pos, T: int, k: int, shared=None, y=None, stream=None):
    """a6: y[t] = sum_j y_perm[pair_pos[t*k+j]] (+ shared[t])."""
    torch = _torch()
    H = y_perm.shape[1]
    if y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=y_perm.device)
    _check(lib().moe_finalize_routing(_ptr(y_perm), _ptr(pair_pos), _ptr(shared), T, k, H, _ptr(y),
                                      _stream(stream)), "moe_finalize_routing")
    return y


def make_desc(T, H, E, k, I, gate="softmax", routed_scaling_factor=1.0, eps=1e-20, n_shared=0, I_s=0):
    return moe_layer_desc(T, H, E, k, I, GATES[gate] if isinstance(gate, str) else gate, routed_scaling_factor,
                          eps, n_shared, I_s if n_shared else 0)


def moe_layer_workspace_size(desc: moe_layer_desc) -> int:
    n = lib().moe_layer_workspace_size(ctypes.byref(desc))
    if n == 0:
        raise MoEError(MOE_ERR_INVALID_ARG, "moe_layer_workspace_size")
    return n


def moe_layer_workspace_offsets(desc: moe_layer_desc) -> list:
    arr = (ctypes.c_size_t * 8)()
    lib().moe_layer_workspace_offsets(ctypes.byref(desc), arr, 8)
    return list(arr)


def moe_layer_forward(desc: moe_layer_desc, x, logits, w13, w2, bias=None, w13_s=None, w2_s=None, ws=None,
                      y=None, topk_w=None, topk_idx=None, counts=None, stream=None):
    """The whole layer; returns (y, topk_w, topk_idx, counts, ws)."""
    torch = _torch()
    dev = x.device
    T, k, H, E = desc.T, desc.k, desc.H, desc.E
    y = y if y is not None else torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    topk_w = topk_w if topk_w is not None else torch.empty((T, k), dtype=torch.float32, device=dev)
    topk_idx = topk_idx if topk_idx is not None else torch.empty((T, k), dtype=torch.int32, device=dev)
    counts = counts if counts is not None else torch.empty(E, dtype=torch.int32, device=dev)
    ws = _ws(moe_layer_workspace_size(desc), dev, ws)
    _check(lib().moe_layer_forward(ctypes.byref(desc), _ptr(x), _ptr(logits), _ptr(bias), _ptr(w13), _ptr(w2),
                                   _ptr(w13_s), _ptr(w2_s), _ptr(y), _ptr(topk_w), _ptr(topk_idx), _ptr(counts),
                                   _ptr(ws), ws.numel(), _stream(stream)), "moe_layer_forward")
    return y, topk_w, topk_idx, counts, ws


def moe_layer_forward_events(desc: moe_layer_desc, events, x, logits, w13, w2, bias=None, w13_s=None, w2_s=None,
                             ws=None, y=None, topk_w=None, topk_idx=None, counts=None, stream=None):
    """moe_layer_forward that also records six torch.cuda.Event objects around its steps
    (before gating, routing, gate/up GEMM, down GEMM, finalize; after finalize)."""
    handles = (ctypes.c_void_p * 6)()
    for i, ev in enumerate(events):
        if ev.cuda_event == 0:  # torch creates the event lazily on its first record
            ev.record()
        handles[i] = ev.cuda_event
    _check(lib().moe_layer_forward_events(ctypes.byref(desc), _ptr(x), _ptr(logits), _ptr(bias), _ptr(w13),
                                          _ptr(w2), _ptr(w13_s), _ptr(w2_s), _ptr(y), _ptr(topk_w), _ptr(topk_idx),
                                          _ptr(counts), _ptr(ws), ws.numel(), _stream(stream), handles, 6),
           "moe_layer_forward_events")
    return y


def moe_layer_kernel_launches(desc: moe_layer_desc) -> int:
    return lib().moe_layer_kernel_launches(ctypes.byref(desc))


def moe_get_device_status(ws, stream=None) -> int:
    return lib().moe_get_device_status(_ptr(ws), _stream(stream))


def moe_workspace_init(ws, stream=None) -> None:
    _check(lib().moe_workspace_init(_ptr(ws), ws.numel(), _stream(stream)), "moe_workspace_init")


class MoELayer:
    """One MoE layer shape with its own workspace and output buffers (reused across calls)."""

    def __init__(self, T, H, E, k, I, gate="softmax", routed_scaling_factor=1.0, eps=1e-20, n_shared=0, I_s=0,
                 device="cuda"):
        torch = _torch()
        self.desc = make_desc(T, H, E, k, I, gate, routed_scaling_factor, eps, n_shared, I_s)
        self.device = torch.device(device)
        self.ws = torch.zeros(moe_layer_workspace_size(self.desc), dtype=torch.uint8, device=self.device)
        self.y = torch.empty((T, H), dtype=torch.bfloat16, device=self.device)
        self.topk_w = torch.empty((T, k), dtype=torch.float32, device=self.device)
        self.topk_idx = torch.empty((T, k), dtype=torch.int32, device=self.device)
        self.counts = torch.empty(E, dtype=torch.int32, device=self.device)
        self.offsets_bytes = moe_layer_workspace_offsets(self.desc)

    def forward(self, x, logits, w13, w2, bias=None, w13_s=None, w2_s=None, stream=None):
        """w13 / w13_s in the packed layout of moe_prepack_w13."""
        moe_layer_forward(self.desc, x, logits, w13, w2, bias, w13_s, w2_s, self.ws, self.y, self.topk_w,
                          self.topk_idx, self.counts, stream)
        return self.y

    def forward_events(self, events, x, logits, w13, w2, bias=None, w13_s=None, w2_s=None, stream=None):
        moe_layer_forward_events(self.desc, events, x, logits, w13, w2, bias, w13_s, w2_s, self.ws, self.y,
                                 self.topk_w, self.topk_idx, self.counts, stream)
        return self.y

    def intermediate(self, name: str):
        """View of an intermediate in the workspace: offsets, sorted_pair, pair_pos, x_exp, act, y_perm, act_s, shared."""
        torch = _torch()
        d = self.desc
        P = d.T * d.k
        spec = {
            "offsets": (0, torch.int32, (d.E + 1,)),
            "sorted_pair": (1, torch.int32, (P,)),
            "pair_pos": (2, torch.int32, (P,)),
            "x_exp": (3, torch.bfloat16, (P, d.H)),
            "act": (4, torch.bfloat16, (P, d.I)),
            "y_perm": (5, torch.bfloat16, (P, d.H)),
            "act_s": (6, torch.bfloat16, (d.T, d.I_s)),
            "shared": (7, torch.bfloat16, (d.T, d.H)),
        }[name]
        i, dt, shape = spec
        n = 1
        for s in shape:
            n *= s
        off = self.offsets_bytes[i]
        nbytes = n * (4 if dt == torch.int32 else 2)
        return self.ws[off:off + nbytes].view(dt).view(shape)
