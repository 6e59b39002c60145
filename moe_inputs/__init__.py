"""Seeded synthetic inputs for the MoE expert-layer forward.

This module is shared by the CUDA path's tests and bench and by the CPU oracle.
It holds none of the method's arithmetic: it only defines the workload shapes
and turns (seed, tensor id, element index) into numbers, through the
Philox4x32-10 generator in ``philox_gen.c``.

Workloads (shapes from the Qwen3-MoE and Hy3 serving pages):

* ``tiny``          T=16,    H=256,  E=8,   k=2, I=128,  softmax
* ``qwen3_decode``  T=64,    H=4096, E=128, k=8, I=1536, softmax
* ``hy3_decode``    T=16,    H=4096, E=192, k=8, I=1536, sigmoid+bias x2.826, 1 shared expert
* ``hy3_prefill``   T=4096,  same as hy3_decode, Zipf(1.1) expert popularity
* ``long_prefill``  T=16384, H=2048, E=128, k=8, I=768,  softmax, Zipf(1.2)

Distributions: x ~ N(0,1) -> bf16; weights ~ N(0,0.02) -> bf16; router logits
fp32 = round_{2^-8}(N(0,1) + off_e); bias ~ N(0,0.01) fp32.  ``off_e`` is 0 for
uniform popularity; for the Zipf workloads it is round_{2^-8}(beta*ln(E*p_e))
with p_e proportional to rank_e^-s (ranks from a seeded Fisher-Yates shuffle),
and the four lowest-ranked experts get -16 so that they receive no tokens.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "philox_gen.c")
_LIB_PATH = os.path.join(_HERE, "libmoe_inputs.so")
_lib = None
_lock = threading.Lock()

# tensor ids of the Philox key
TID_X, TID_W13, TID_W2, TID_W13S, TID_W2S, TID_LOGITS, TID_BIAS, TID_SHUFFLE = range(1, 9)


def build(force: bool = False) -> str:
    """Compile ``philox_gen.c`` into ``libmoe_inputs.so`` (plain C, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            u64, u32, i64, dbl = ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int64, ctypes.c_double
            vp = ctypes.c_void_p
            lib.moe_inputs_philox4x32_10.argtypes = [vp, vp, vp]
            lib.moe_inputs_u32.argtypes = [u64, u32, i64, vp]
            lib.moe_inputs_normal_bf16.argtypes = [u64, u32, i64, dbl, dbl, vp]
            lib.moe_inputs_normal_bf16_range.argtypes = [u64, u32, i64, i64, dbl, dbl, vp]
            lib.moe_inputs_normal_f32.argtypes = [u64, u32, i64, dbl, dbl, vp]
            lib.moe_inputs_grid_logits.argtypes = [u64, u32, i64, i64, vp, ctypes.c_int, vp]
            for f in ("moe_inputs_philox4x32_10", "moe_inputs_u32", "moe_inputs_normal_bf16",
                      "moe_inputs_normal_bf16_range",
                      "moe_inputs_normal_f32", "moe_inputs_grid_logits"):
                getattr(lib, f).restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags.c_contiguous
    return a.ctypes.data


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, np.uint32)
    _load().moe_inputs_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform_u32(seed: int, tid: int, n: int) -> np.ndarray:
    out = np.empty(n, np.uint32)
    _load().moe_inputs_u32(seed, tid, n, _ptr(out))
    return out


def normal_bf16(seed: int, tid: int, shape, mean=0.0, std=1.0) -> np.ndarray:
    """bf16 bit patterns (uint16) of mean + std*N(0,1)."""
    out = np.empty(shape, np.uint16)
    _load().moe_inputs_normal_bf16(seed, tid, out.size, float(mean), float(std), _ptr(out))
    return out


def normal_bf16_slice(seed: int, tid: int, start: int, shape, mean=0.0, std=1.0) -> np.ndarray:
    """Elements [start, start + prod(shape)) of the stream normal_bf16 draws for the same tensor id:
    normal_bf16(seed, tid, full_shape).reshape(-1)[start:start + n], without the rest."""
    out = np.empty(shape, np.uint16)
    _load().moe_inputs_normal_bf16_range(seed, tid, int(start), out.size, float(mean), float(std), _ptr(out))
    return out


def expert_weights(cfg: "MoEConfig", e: int):
    """(w13[e] [2I,H], w2[e] [H,I]) of generate(cfg): expert e's slices of the weight streams."""
    n13, n2 = 2 * cfg.I * cfg.H, cfg.H * cfg.I
    return (normal_bf16_slice(cfg.seed, TID_W13, e * n13, (2 * cfg.I, cfg.H), 0.0, cfg.w_std),
            normal_bf16_slice(cfg.seed, TID_W2, e * n2, (cfg.H, cfg.I), 0.0, cfg.w_std))


def normal_f32(seed: int, tid: int, shape, mean=0.0, std=1.0) -> np.ndarray:
    out = np.empty(shape, np.float32)
    _load().moe_inputs_normal_f32(seed, tid, out.size, float(mean), float(std), _ptr(out))
    return out


def grid_logits(seed: int, tid: int, T: int, E: int, off: Optional[np.ndarray], q: int = 8) -> np.ndarray:
    out = np.empty((T, E), np.float32)
    offp = None
    if off is not None:
        off = np.ascontiguousarray(off, dtype=np.float64)
        offp = _ptr(off)
    _load().moe_inputs_grid_logits(seed, tid, T, E, offp, q, _ptr(out))
    return out


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    gate: str  # "softmax" | "sigmoid" | "sigmoid_inner_bias"
    routed_scaling_factor: float = 1.0
    eps: float = 1e-20
    n_shared: int = 0
    I_s: int = 0
    bias_std: float = 0.0
    zipf_s: float = 0.0
    zipf_beta: float = 0.0
    n_dead: int = 0  # lowest-ranked experts pushed to -16 (receive no tokens)
    w_std: float = 0.02
    seed: int = 0

    @property
    def P(self) -> int:
        return self.T * self.k

    def with_(self, **kw) -> "MoEConfig":
        return replace(self, **kw)


# beta of the Zipf workloads was chosen so that the seeded routing gives a
# max/mean expert load near 7.5 (the middle of the 5-10x hot-expert range);
# tests/test_inputs.py checks the ratio lies in [5, 10] with empty experts.
CONFIGS = {
    "tiny": MoEConfig("tiny", T=16, H=256, E=8, k=2, I=128, gate="softmax"),
    "qwen3_decode": MoEConfig("qwen3_decode", T=64, H=4096, E=128, k=8, I=1536, gate="softmax"),
    "hy3_decode": MoEConfig("hy3_decode", T=16, H=4096, E=192, k=8, I=1536, gate="sigmoid",
                            routed_scaling_factor=2.826, n_shared=1, I_s=1536, bias_std=0.01),
    "hy3_prefill": MoEConfig("hy3_prefill", T=4096, H=4096, E=192, k=8, I=1536, gate="sigmoid",
                             routed_scaling_factor=2.826, n_shared=1, I_s=1536, bias_std=0.01,
                             zipf_s=1.1, zipf_beta=0.27, n_dead=4),
    "long_prefill": MoEConfig("long_prefill", T=16384, H=2048, E=128, k=8, I=768, gate="softmax",
                              zipf_s=1.2, zipf_beta=0.34, n_dead=4),
}


def zipf_offsets(cfg: MoEConfig) -> Optional[np.ndarray]:
    """Per-expert logit offsets giving a Zipf(s) popularity profile (None if uniform)."""
    if cfg.zipf_s == 0.0:
        return None
    E = cfg.E
    perm = list(range(E))
    u = uniform_u32(cfg.seed, TID_SHUFFLE, E)
    for i in range(E - 1, 0, -1):  # Fisher-Yates
        j = int(u[i]) % (i + 1)
        perm[i], perm[j] = perm[j], perm[i]
    rank = np.empty(E, np.int64)
    rank[np.array(perm)] = np.arange(1, E + 1)
    p = rank.astype(np.float64) ** (-cfg.zipf_s)
    p /= p.sum()
    off = np.round(cfg.zipf_beta * np.log(E * p) * 256.0) / 256.0
    off[rank > E - cfg.n_dead] = -16.0
    return off


@dataclass
class MoEInputs:
    cfg: MoEConfig
    x: np.ndarray            # [T,H] uint16 (bf16 bits)
    logits: np.ndarray       # [T,E] float32
    bias: Optional[np.ndarray]   # [E] float32
    w13: Optional[np.ndarray]    # [E,2I,H] uint16, rows [gate; up]
    w2: Optional[np.ndarray]     # [E,H,I] uint16
    w13_s: Optional[np.ndarray] = None  # [2I_s,H]
    w2_s: Optional[np.ndarray] = None   # [H,I_s]
    off: Optional[np.ndarray] = field(default=None)


def generate(cfg: MoEConfig, weights: bool = True) -> MoEInputs:
    """All inputs of one layer call, deterministic in (cfg, cfg.seed)."""
    s = cfg.seed
    off = zipf_offsets(cfg)
    x = normal_bf16(s, TID_X, (cfg.T, cfg.H))
    logits = grid_logits(s, TID_LOGITS, cfg.T, cfg.E, off)
    bias = normal_f32(s, TID_BIAS, (cfg.E,), 0.0, cfg.bias_std) \
        if cfg.gate in ("sigmoid", "sigmoid_inner_bias") and cfg.bias_std > 0 else None
    w13 = w2 = w13s = w2s = None
    if weights:
        w13 = normal_bf16(s, TID_W13, (cfg.E, 2 * cfg.I, cfg.H), 0.0, cfg.w_std)
        w2 = normal_bf16(s, TID_W2, (cfg.E, cfg.H, cfg.I), 0.0, cfg.w_std)
        if cfg.n_shared:
            w13s = normal_bf16(s, TID_W13S, (2 * cfg.I_s, cfg.H), 0.0, cfg.w_std)
            w2s = normal_bf16(s, TID_W2S, (cfg.H, cfg.I_s), 0.0, cfg.w_std)
    return MoEInputs(cfg, x, logits, bias, w13, w2, w13s, w2s, off)


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (input formatting only)."""
    return (np.asarray(u, np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even narrowing of float32 to bf16 bit patterns (no NaN inputs)."""
    u = np.ascontiguousarray(f, np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)
