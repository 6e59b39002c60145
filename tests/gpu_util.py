"""Helpers shared by the GPU parity tests: host<->device marshalling and the error metrics."""
import numpy as np

import oracle

# Output tolerance for floating-point results (the layer's stated bar):
#   max|gpu - oracle| / max|oracle| <= 2e-2  and  mean|gpu - oracle| / mean|oracle| <= 5e-3
TOL_MAX = 2e-2
TOL_MEAN = 5e-3


def torch():
    import torch as _t
    return _t


def dev_bf16(u16: np.ndarray):
    t = torch()
    return t.from_numpy(np.ascontiguousarray(u16).view(np.int16)).cuda().view(t.bfloat16)


def dev(a: np.ndarray):
    return torch().from_numpy(np.ascontiguousarray(a)).cuda()


def host_bf16_f64(t) -> np.ndarray:
    tt = torch()
    return oracle.bf16_to_f64(t.detach().contiguous().view(tt.int16).cpu().numpy().view(np.uint16))


def host(t) -> np.ndarray:
    return t.detach().cpu().numpy()


def rel_errors(gpu: np.ndarray, ref: np.ndarray):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    d = np.abs(gpu - ref)
    return float(d.max() / max(np.abs(ref).max(), 1e-300)), float(d.mean() / max(np.abs(ref).mean(), 1e-300))


def assert_close(gpu, ref, what="", tol_max=TOL_MAX, tol_mean=TOL_MEAN):
    mx, mean = rel_errors(gpu, ref)
    assert mx <= tol_max and mean <= tol_mean, f"{what}: max-rel {mx:.3e} (<= {tol_max}), mean-rel {mean:.3e} (<= {tol_mean})"
    return mx, mean


def assert_bf16_rounding_close(gpu, ref, what=""):
    """Single rounding of an fp32-accumulated value to bf16: elementwise within 2^-8 relative
    plus an absolute slack of 2e-3 * max|ref| for fp32 summation-order effects near zero."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    bound = 2.0 ** -8 * np.abs(ref) + 2e-3 * np.abs(ref).max()
    bad = np.abs(gpu - ref) > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements outside the bf16 rounding bound, e.g. {np.argwhere(bad)[:3]}"
