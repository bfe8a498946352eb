"""Shared test helpers: tolerances and device transfer (no method arithmetic)."""
import numpy as np

# Tolerances the workload definition states: per-tensor max relative error
# (max_i |a_i - b_i| / max_i |b_i|) <= 1e-2 for TF32 GEMM outputs and
# gradients, <= 1e-6 for the fp32 update; loss within 1e-3 relative.
TOL_TF32 = 1e-2
TOL_UPDATE = 1e-6
TOL_LOSS = 1e-3
# exact-fp32 elementwise kernels (softmax, CUDA-core GEMM/conv paths): fp32
# rounding of sums of up to a few thousand terms
TOL_FP32 = 1e-5


def rel_inf(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = np.max(np.abs(b)) if b.size else 0.0
    num = np.max(np.abs(a - b)) if b.size else 0.0
    if den == 0.0:
        return float(num)
    return float(num / den)


def dev(x, dtype=None):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        t = t.to(dtype)
    return t.cuda()


def host(t):
    import torch
    torch.cuda.synchronize()
    return t.detach().cpu().numpy()
