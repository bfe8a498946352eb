"""The SPRINT report's GPU cost model, refitted to this library's kernels.

IPSJ SIG Technical Report Vol.2016-HPC-155 No.8 ("SPRINT"), Sec. 3.3-3.6:
  * Eq. (4): a replica's ComputeGradient time is the sum over layers of the
    time of its CUDA kernels and SGEMMs;
  * Eq. (6): one SGEMM role of (m, n, k) costs
        a_mnk*m*n*k + a_mn*m*n + a_mk*m*k + a_nk*n*k + a_m*m + a_n*n + a_k*k + b,
    with the coefficients fitted per role from measurements;
  * the role table of Sec. 3.3 gives (m, n, k) of every layer's GEMMs:
        convolution  m = x_l^2 N, n = m_l,      k = c^2 m_{l-1}
        fc           m = N,       n = m_l,      k = x_{l-1}^2 m_{l-1}
        dedw         m = c^2 m_{l-1} (conv) or the fc fan-in, n = m_l, k = x_l^2 N
        dedb         m = 1,       n = m_l,      k = x_l^2 N
        dedx fc      m = N,       n = fan-in,   k = m_l
        dedx conv    m = x_l^2 N, n = c^2 m_{l-1}, k = m_l     (not for layer 1)
    (c = 3, the filter size; x_l the output side of layer l, N = N_Subbatch);
  * Eq. (9): the average number of samples behind one update,
        N_Minibatch_avg = N_Node * N_GPU * N_Subbatch * T_Update / T_GPU;
  * Eq. (10): one epoch over N_File images takes
        T_Epoch = N_File * T_Update / N_Minibatch_avg.
Here a "role" is what one library call (or the difference of two) does: the
implicit-GEMM convolutions have no separate im2col (Eq. (5)'s term is 0), and
dedb comes out of the dedw GEMM, so dedw and dedb are one fitted role.
This module is host arithmetic only (numpy least squares)."""
from __future__ import annotations

import numpy as np

from .model import LayerShape

ROLES = ("convolution", "fc", "dedw", "dedx_fc", "dedx_conv")
N_COEF = 8


def sgemm_features(m, n, k) -> np.ndarray:
    """The eight terms of Eq. (6) for one (m, n, k)."""
    m, n, k = float(m), float(n), float(k)
    return np.array([m * n * k, m * n, m * k, n * k, m, n, k, 1.0])


def role_dims(L: LayerShape, N: int, first: bool) -> dict:
    """(m, n, k) of each GEMM role of layer L at N_Subbatch = N (Sec. 3.3 table),
    for the roles this layer has (no input gradient for the first layer)."""
    if L.kind == "conv":
        px = L.h * L.w * N          # output pixels (stride 1, same padding)
        kk = 9 * L.cin
        out = {"convolution": (px, L.cout, kk), "dedw": (kk, L.cout, px)}
        if not first:
            out["dedx_conv"] = (px, kk, L.cout)
    else:
        out = {"fc": (N, L.cout, L.cin), "dedw": (L.cin, L.cout, N)}
        if not first:
            out["dedx_fc"] = (N, L.cin, L.cout)
    return out


def fit_role(samples) -> np.ndarray:
    """Least-squares coefficients of Eq. (6) from [(m, n, k, seconds), ...].
    Columns are scaled to unit norm before solving (the terms span ~10 orders of
    magnitude); terms the samples cannot tell apart get the minimum-norm share."""
    X = np.array([sgemm_features(m, n, k) for m, n, k, _ in samples])
    y = np.array([t for *_, t in samples], dtype=np.float64)
    scale = np.linalg.norm(X, axis=0)
    scale[scale == 0] = 1.0
    coef, *_ = np.linalg.lstsq(X / scale, y, rcond=None)
    return coef / scale


def predict(coef: np.ndarray, m, n, k) -> float:
    return float(sgemm_features(m, n, k) @ coef)


def predict_t_gpu(shapes: list[LayerShape], N: int, coefs: dict) -> float:
    """Eq. (4) with Eq. (6) per role: a replica's forward + backward GEMM time."""
    total = 0.0
    for i, L in enumerate(shapes):
        for role, (m, n, k) in role_dims(L, N, i == 0).items():
            total += predict(coefs[role], m, n, k)
    return total


def n_minibatch_avg(n_node: int, n_gpu: int, n_subbatch: int, t_update: float, t_gpu: float) -> float:
    """Eq. (9): samples behind one update on average."""
    return n_node * n_gpu * n_subbatch * t_update / t_gpu


def t_epoch(n_file: int, t_update: float, n_mb_avg: float) -> float:
    """Eq. (10): seconds for one pass over n_file images."""
    return n_file * t_update / n_mb_avg
