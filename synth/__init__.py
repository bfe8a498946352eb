"""Seeded synthetic inputs shared by the FP64 oracle and the CUDA path.

This module draws random numbers and nothing else: it holds none of the
training method's arithmetic (no convolution, no gradient, no update rule).
Both sides of every parity test take their inputs from here, so that they see
bit-identical fp32 tensors.

Recipe (stand-ins for CIFAR-10 / ILSVRC 2012 images, which are not available):
  * images: i.i.d. N(0, 1) fp32, drawn in logical NCHW order and stored NHWC;
  * labels: uniform integers in [0, classes);
  * weights: N(0, std^2) with the std the caller passes (He-normal
    sqrt(2 / fan_in) for the networks), biases zero;
  * parameter-server buffers: N(0, std^2) flat vectors;
  * dyadic values k * 2**-12 (small integer k) for order-invariance tests,
    whose sums are exact in fp32 and fp64.

Every draw is keyed by (seed, tag) through numpy's PCG64 + SeedSequence, so a
tensor does not depend on which other tensors were drawn before it.
"""
from __future__ import annotations

import zlib

import numpy as np

__all__ = [
    "rng",
    "normal",
    "labels",
    "images_nhwc",
    "dyadic",
    "batch_pool",
    "device_normal",
]


def rng(seed: int, tag: str) -> np.random.Generator:
    """Independent generator for one named tensor."""
    key = zlib.crc32(tag.encode("utf-8"))
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed) & 0xFFFFFFFF, int(seed) >> 32, key])))


def normal(seed: int, tag: str, shape, std: float = 1.0, dtype=np.float32) -> np.ndarray:
    """N(0, std^2) samples of the given shape (drawn in double, then cast)."""
    g = rng(seed, tag)
    out = g.standard_normal(size=shape, dtype=np.float64)
    if std != 1.0:
        out *= std
    return out.astype(dtype, copy=False)


def labels(seed: int, tag: str, n: int, classes: int) -> np.ndarray:
    """Class labels uniform in [0, classes), int32."""
    return rng(seed, tag).integers(0, classes, size=n, dtype=np.int64).astype(np.int32)


def images_nhwc(seed: int, tag: str, n: int, c: int, h: int, w: int) -> np.ndarray:
    """N(0,1) images drawn in logical NCHW order, returned as contiguous NHWC fp32."""
    x = normal(seed, tag, (n, c, h, w))
    return np.ascontiguousarray(x.transpose(0, 2, 3, 1))


def dyadic(seed: int, tag: str, shape, kmax: int = 64, exp: int = 12) -> np.ndarray:
    """Values k * 2**-exp with k uniform in [-kmax, kmax]; small sums of them are exact."""
    k = rng(seed, tag).integers(-kmax, kmax + 1, size=shape, dtype=np.int64)
    return (k.astype(np.float64) * 2.0 ** (-exp)).astype(np.float32)


def batch_pool(seed: int, count: int, n: int, c: int, h: int, w: int, classes: int, flat: bool = False):
    """`count` pre-generated (images, labels) batches.

    Batch j is drawn under tags ``x/j`` and ``y/j``; with ``flat`` the images
    are returned as [n][c*h*w] rows in (h, w, c) order (the MLP input).
    """
    out = []
    for j in range(count):
        x = images_nhwc(seed, f"x/{j}", n, c, h, w)
        if flat:
            x = x.reshape(n, -1)
        out.append((x, labels(seed, f"y/{j}", n, classes)))
    return out


def device_normal(seed: int, tag: str, shape, std: float = 1.0, device="cuda"):
    """N(0, std^2) fp32 samples drawn on a GPU by a torch generator keyed by
    (seed, tag): the large full-size tensors (hundreds of MB) of the parity
    tests, which both sides then read from the same device buffer."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1000003 + zlib.crc32(tag.encode("utf-8"))) & 0x7FFFFFFFFFFFFFFF)
    t = torch.randn(tuple(shape), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t
