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


# ---- sampled outputs of full-size tensors (data movement only)

def sample_pixels(seed, N, H, W, count=384):
    """Sampled output pixels: the four corners of the first and last image, the
    middle of each edge, and uniform draws."""
    g = np.random.default_rng(seed)
    fixed = [(0, 0, 0), (0, 0, W - 1), (0, H - 1, 0), (N - 1, H - 1, W - 1), (N - 1, 0, W // 2),
             (N - 1, H // 2, 0), (0, H // 2, W - 1), (N // 2, H - 1, W // 2)]
    n = np.concatenate([[p[0] for p in fixed], g.integers(0, N, count)])
    h = np.concatenate([[p[1] for p in fixed], g.integers(0, H, count)])
    w = np.concatenate([[p[2] for p in fixed], g.integers(0, W, count)])
    return n, h, w


def crops3x3(t, n, h, w):
    """Host float64 [S][3][3][C]: the 3x3 neighbourhoods (zero outside the image)
    of the sampled pixels of a device NHWC tensor."""
    import torch
    tp = torch.nn.functional.pad(t, (0, 0, 1, 1, 1, 1))
    d = torch.arange(3, device=t.device)
    ni = torch.as_tensor(n, device=t.device)[:, None, None]
    hi = torch.as_tensor(h, device=t.device)[:, None, None] + d[None, :, None]
    wi = torch.as_tensor(w, device=t.device)[:, None, None] + d[None, None, :]
    return tp[ni, hi, wi].double().cpu().numpy()


def at_pixels(t, n, h, w):
    import torch
    return t[torch.as_tensor(n, device=t.device), torch.as_tensor(h, device=t.device),
             torch.as_tensor(w, device=t.device)].double().cpu().numpy()
