"""Network shapes and the device parameter layout of the worker step.

The networks are the ones the pages and the workload definitions name:
  * the CNN class of the SPRINT report (IPSJ SIG Technical Report
    Vol.2016-HPC-155 No.8, Sec. 3.2, Eq. (2)-(3)): L_c 3x3 'same' conv layers,
    each followed by ReLU and optionally a 2x2 max-pool (p_l = 2), then FC
    layers; softmax output;
  * SMLPs (Qiita "Chainer multi-GPU", Sec. 4): two 3-layer MLPs with a ReLU
    between them, 3072 -> 5000 x 5 -> 10;
  * VGG-16-style stacks, CIFAR- and ILSVRC-shaped.

Device parameter layout: one flat fp32 vector per weight version holding,
layer by layer, W then b. Every tensor starts on a 4-element (16-byte)
boundary (TMA and 128-bit vector access need it); the gap elements are zero
and stay zero under every update rule (their gradient is zero). ``pack`` /
``unpack`` convert to and from the dense order (no gaps).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

_VGG = [(64, False), (64, True), (128, False), (128, True), (256, False), (256, False), (256, True),
        (512, False), (512, False), (512, True), (512, False), (512, False), (512, True)]

# ("conv", out_channels, pool_after) | ("fc", out_features, relu)
NETWORKS = {
    "tiny": dict(input=(3, 32, 32), classes=10, layers=[("conv", 16, True), ("conv", 32, True), ("fc", 10, False)]),
    "smlps": dict(input=(3072, 1, 1), classes=10, layers=[("fc", 5000, True)] * 5 + [("fc", 10, False)]),
    "vgg_c": dict(input=(3, 32, 32), classes=10,
                  layers=[("conv", c, p) for c, p in _VGG] + [("fc", 512, True), ("fc", 512, True), ("fc", 10, False)]),
    "vgg_i": dict(input=(3, 224, 224), classes=1000,
                  layers=[("conv", c, p) for c, p in _VGG] + [("fc", 4096, True), ("fc", 4096, True),
                                                               ("fc", 1000, False)]),
}

# Pipeline stage of each layer for the 4-stage VGG-C pipeline: stage 0 = block 1,
# 1 = block 2, 2 = block 3, 3 = blocks 4-5 and the classifier (registers early).
VGG_C_STAGES = [0, 0, 1, 1, 2, 2, 2, 3, 3, 3, 3, 3, 3, 3, 3, 3]


@dataclass(frozen=True)
class LayerShape:
    kind: str           # "conv" | "fc"
    cin: int
    cout: int
    h: int              # conv: input (= output) height; fc: 1
    w: int
    pool: bool
    relu: bool
    w_off: int          # offset of W in the padded flat vector
    b_off: int          # offset of b
    w_numel: int
    fan_in: int

    @property
    def out_hw(self):
        return (self.h // 2, self.w // 2) if self.pool else (self.h, self.w)


def _pad4(n: int) -> int:
    return (n + 3) & ~3


def layer_shapes(net) -> list[LayerShape]:
    """Shapes of every layer (Eq. (2): x_l = x_{l-1}/p_l for conv, 1 for FC)."""
    c, h, w = net["input"]
    flat = None
    off = 0
    out = []
    for kind, cout, flag in net["layers"]:
        if kind == "conv":
            if flat is not None:
                raise ValueError("conv layer after an FC layer")
            numel = cout * 9 * c
            w_off = off
            b_off = _pad4(w_off + numel)
            off = _pad4(b_off + cout)
            out.append(LayerShape("conv", c, cout, h, w, bool(flag), True, w_off, b_off, numel, 9 * c))
            c = cout
            if flag:
                h, w = h // 2, w // 2
        else:
            fin = c * h * w if flat is None else flat
            numel = cout * fin
            w_off = off
            b_off = _pad4(w_off + numel)
            off = _pad4(b_off + cout)
            out.append(LayerShape("fc", fin, cout, 1, 1, False, bool(flag), w_off, b_off, numel, fin))
            flat = cout
    return out


def padded_size(shapes: list[LayerShape]) -> int:
    last = shapes[-1]
    return _pad4(last.b_off + last.cout)


def dense_size(shapes: list[LayerShape]) -> int:
    return sum(L.w_numel + L.cout for L in shapes)


def param_count(net) -> int:
    """N_Param of Eq. (3): the number of weights and biases."""
    return dense_size(layer_shapes(net))


def pack(shapes, dense: np.ndarray) -> np.ndarray:
    """Dense [W0 b0 W1 b1 ...] -> padded device layout (gaps zero)."""
    out = np.zeros(padded_size(shapes), dense.dtype)
    o = 0
    for L in shapes:
        out[L.w_off:L.w_off + L.w_numel] = dense[o:o + L.w_numel]
        o += L.w_numel
        out[L.b_off:L.b_off + L.cout] = dense[o:o + L.cout]
        o += L.cout
    return out


def unpack(shapes, padded: np.ndarray) -> np.ndarray:
    """Padded device layout -> dense [W0 b0 W1 b1 ...]."""
    parts = []
    for L in shapes:
        parts.append(padded[L.w_off:L.w_off + L.w_numel])
        parts.append(padded[L.b_off:L.b_off + L.cout])
    return np.concatenate(parts)


def train_flops_per_image(net) -> float:
    """GEMM FLOPs per image for one training step: forward, dW and dX
    (2 per multiply-add), no dX for the first layer."""
    f = 0.0
    for i, L in enumerate(layer_shapes(net)):
        macs = L.h * L.w * L.cout * 9 * L.cin if L.kind == "conv" else L.cout * L.cin
        f += 2.0 * macs * (2 if i == 0 else 3)
    return f


def staleness_degrees(stage_delays) -> list[int]:
    """Degree of staleness of each pipeline stage pair: the number of steps its
    weights lag ("Pipelined training of deep CNNs with stale weights", Sec. 4.1)."""
    return [int(s) for s in stage_delays]


def stale_weight_percent(shapes: list[LayerShape], stage_of_layer, stage_delays) -> float:
    """Percentage of the parameters (weights and biases) that sit in stages
    computing on stale weights (delay > 0), same section: every layer before
    the last pipeline-register pair trains on old weights."""
    counts = [L.w_numel + L.cout for L in shapes]
    stale = sum(n for n, k in zip(counts, stage_of_layer) if stage_delays[k] > 0)
    return 100.0 * stale / sum(counts)
