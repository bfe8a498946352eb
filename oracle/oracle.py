"""FP64 CPU oracle for the stale-weight SGD worker step and the parameter-server update.

TEST INFRASTRUCTURE. Only tests/, ``__graft_entry__.smoke()`` and bench.py's
``cpu_baseline`` leg / reference arm may import this module. The product path
(the ``stale_weight_sgd_gb300`` package and its CUDA library) never imports it
and shares no code with it; the two meet only through the seeded inputs of
the ``synth`` module.

Everything is computed in float64 from the (float32) inputs. It is written to be
read against the pages, not to be fast: plain numpy, one step of the definition
per line, a library matmul where the definition has an inner sum.

Pages this follows (by title, section / equation):
  [S]  IPSJ SIG Technical Report Vol.2016-HPC-155 No.8, "SPRINT" ASGD CNN
       framework (Oyama et al.): Eq. (1) minibatch SGD, Eq. (2) spatial sizes,
       Eq. (3) N_Param, Sec. 3.3 SGEMM role table (convolution / fc / dedw /
       dedb / dedx), Algorithm 1 (GPU thread: ComputeGradient,
       ComputeUpdateVal, UpdateGradient into GradBuf), Algorithm 2 (update
       thread: SumGradient, momentum through DeltaWeights, UpdateWeights).
  [PB] "Pipelined training of deep CNNs with stale weights" (Zhang &
       Abdelrahman), Sec. 4.1: a forward/backward stage pair uses the same,
       stale, weights.
  [Q]  Qiita "Chainer multi-GPU: model-parallel vs data-parallel", Sec. 4
       (SMLPs model), Sec. 6 (addgrads + halved learning rate == one batch).
  [DB] "Google DistBelief Paper: Large Scale Distributed Deep Networks"
       (blog summary): replicas fetch w, push dw, the server applies
       w' := w - eta*dw; gradients commute and add; per-parameter Adagrad.

Readings taken where the pages are silent or garbled (each one is listed with
its reason in the design notes):
  R1 loss = mean over the replica batch (dz = (p - onehot)/N); Eq. (1)'s sum is
     absorbed into eta. ``reduction="sum"`` keeps the literal form.
  R2 across replicas gradients are summed: W' = W - eta * sum_r g_r.
  R4 GradBuf stores raw gradients (alpha = 1); eta is applied once at update.
  R5 momentum: v' = nu*v - eta*S, W' = W + v' (v0 = 0).
  R6 Adagrad: G' = G + S*S, W' = W - eta*S/(sqrt(G') + eps).
  R7 staleness: replica r at step t uses W(max(0, t - s[t,r])), where W(t) is
     the version before step t's update; delays from SplitMix64.
  R8 pipeline stage k (forward and backward) uses W_k(max(0, t - s_k)).
  R11 Nesterov momentum (the pipelined-training page's appendices train with
     "SGD with Nesterov momentum" but print no formula): in R5's units,
     v' = nu*v - eta*S, W' = W + nu*v' - eta*S.
  R12 weight decay (same appendices, a coefficient only): L2 on the summed
     gradient at the parameter server, S <- S + lambda*W, before any rule.
  R13 hybrid pipelined/non-pipelined training ([PB] Sec. 4.2): the stage
     delays s_k hold for steps t < N_p and are 0 from t = N_p on. Degree of
     staleness of stage pair k = s_k (steps its weights lag); percentage of
     stale weights = the parameters (W and b) of layers in stages with s_k > 0
     over all parameters ([PB] Sec. 4.1).
  R14 DistBelief n_fetch / n_push ([DB]): every replica refreshes a local copy
     of the parameters from the server at steps t with t % n_fetch == 0 and
     computes its gradients on that copy; it accumulates them in its GradBuf
     (assigned at t % n_push == 0, added otherwise) and pushes at steps with
     (t + 1) % n_push == 0, where the server applies the sum of the R pushed
     buffers (replica order) once. All replicas run in phase.
  R10 max-pool argmax = first window offset in row-major order under strict >.
  R11 ReLU derivative at 0 is 0.

Layouts (a convention both sides follow; the pages fix none):
  activations NHWC [N][H][W][C]; conv weights [Cout][3][3][Cin]; FC weights
  [out][in]; the FC input flattens NHWC in (h, w, c) order; the flat parameter
  vector holds, layer by layer, the weight then the bias.

Parity status: every function here is pinned by tests/test_oracle_*.py
(brute force, adjoint identities, finite differences, closed forms,
published SplitMix64 vectors); see each docstring for its pin.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

F64 = np.float64
_M64 = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15

# ---------------------------------------------------------------------------
# Networks (written from the pages; the product keeps its own copy)
# ---------------------------------------------------------------------------
# conv entry: ("conv", out_channels, pool_after); every conv is 3x3, stride 1,
# pad 1 and is followed by ReLU ([S] Sec. 3.2).  fc entry: ("fc", out, relu).

_VGG_CONV = [(64, False), (64, True), (128, False), (128, True),
             (256, False), (256, False), (256, True),
             (512, False), (512, False), (512, True),
             (512, False), (512, False), (512, True)]

ARCHS = {
    # tiny CNN: conv 3->16 ReLU pool, conv 16->32 ReLU pool, FC 2048->10
    "tiny": dict(input=(3, 32, 32), layers=[("conv", 16, True), ("conv", 32, True), ("fc", 10, False)]),
    # [Q] Sec. 4: mlp1 = (3072->u, ReLU, u->u, ReLU, u->u), ReLU, mlp2 = (u->u, ReLU, u->u, ReLU, u->10)
    "smlps": dict(input=(3072, 1, 1), layers=[("fc", 5000, True)] * 5 + [("fc", 10, False)]),
    # VGG-16 conv stack [S] ref. [11], CIFAR-shaped with FC 512-512-512-10
    "vgg_c": dict(input=(3, 32, 32),
                  layers=[("conv", c, p) for c, p in _VGG_CONV] + [("fc", 512, True), ("fc", 512, True), ("fc", 10, False)]),
    # VGG-16, ILSVRC-shaped, FC 25088-4096-4096-1000
    "vgg_i": dict(input=(3, 224, 224),
                  layers=[("conv", c, p) for c, p in _VGG_CONV] + [("fc", 4096, True), ("fc", 4096, True), ("fc", 1000, False)]),
}


@dataclass
class Layer:
    kind: str        # "conv" or "fc"
    cin: int         # input channels (conv) / input features (fc)
    cout: int
    h: int           # input spatial size (conv only)
    w: int
    pool: bool       # conv: 2x2 max-pool after ReLU
    relu: bool       # fc: ReLU after the affine map (conv: always)
    w_shape: tuple
    fan_in: int


def build_layers(arch) -> list[Layer]:
    """Layer shapes from an architecture description, following Eq. (2) of [S]:
    a conv layer keeps the spatial size (c x c kernel, 'same' padding) and a
    pooled layer divides it by p_l = 2; an FC layer sees the flattened input."""
    c, h, w = arch["input"]
    out = []
    flat = None
    for kind, cout, flag in arch["layers"]:
        if kind == "conv":
            assert flat is None, "conv after fc"
            out.append(Layer("conv", c, cout, h, w, bool(flag), True, (cout, 3, 3, c), 9 * c))
            c = cout
            if flag:
                h, w = h // 2, w // 2
        else:
            fin = c * h * w if flat is None else flat
            out.append(Layer("fc", fin, cout, 1, 1, False, bool(flag), (cout, fin), fin))
            flat = cout
    return out


def spatial_sizes_eq2(arch) -> list[int]:
    """x_l of Eq. (2) in [S]: x_l = x_{l-1}/p_l for conv layers, 1 for FC layers
    (x_0 = input size)."""
    c, h, w = arch["input"]
    xs = [h]
    for kind, _, flag in arch["layers"]:
        if kind == "conv":
            xs.append(xs[-1] // (2 if flag else 1))
        else:
            xs.append(1)
    return xs


def param_count_eq3(arch) -> int:
    """N_Param of Eq. (3) in [S]:
    sum_{l<=Lc} m_l (c^2 m_{l-1} + 1) + sum_{l>Lc} m_l (x_{l-1}^2 m_{l-1} + 1), c = 3."""
    xs = spatial_sizes_eq2(arch)
    m_prev = arch["input"][0]
    total = 0
    for l, (kind, m_l, _) in enumerate(arch["layers"], start=1):
        if kind == "conv":
            total += m_l * (3 * 3 * m_prev + 1)
        else:
            total += m_l * (xs[l - 1] * xs[l - 1] * m_prev + 1)
        m_prev = m_l
    return total


def param_offsets(layers: list[Layer]):
    """(weight offset, bias offset) of each layer in the flat parameter vector."""
    offs, o = [], 0
    for L in layers:
        nw = int(np.prod(L.w_shape))
        offs.append((o, o + nw))
        o += nw + L.cout
    return offs, o


def unflatten(layers, flat):
    offs, n = param_offsets(layers)
    assert flat.size == n
    return [(flat[a:b].reshape(L.w_shape), flat[b:b + L.cout]) for L, (a, b) in zip(layers, offs)]


def flatten(params) -> np.ndarray:
    return np.concatenate([np.concatenate([w.ravel(), b.ravel()]) for w, b in params])


# ---------------------------------------------------------------------------
# Convolution (3x3, stride 1) — [S] Sec. 3.3 "convolution", "dedx conv", "dedw", "dedb"
# ---------------------------------------------------------------------------

def _pad_hw(x, pad):
    return np.pad(x, ((0, 0), (pad, pad), (pad, pad), (0, 0)))


def conv3x3_fwd(x, w, b, pad=1):
    """y[n,oh,ow,co] = b[co] + sum_{kh,kw,ci} x[n, oh+kh-pad, ow+kw-pad, ci] * w[co,kh,kw,ci],
    zero outside the image (cross-correlation, as every CNN framework defines it).
    The sum over the 9 taps is written out; the inner sum over ci is a matmul.
    Pinned by: pure-Python 7-loop brute force, the im2col route, the centre-tap
    (1x1) special case and the impulse-input special case."""
    x = np.asarray(x, F64)
    w = np.asarray(w, F64)
    n, h, wd, ci = x.shape
    ho, wo = h + 2 * pad - 2, wd + 2 * pad - 2
    xp = _pad_hw(x, pad)
    y = np.zeros((n, ho, wo, w.shape[0]), F64)
    for kh in range(3):
        for kw in range(3):
            y += xp[:, kh:kh + ho, kw:kw + wo, :] @ w[:, kh, kw, :].T
    if b is not None:
        y += np.asarray(b, F64)
    return y


def conv3x3_dx(dy, w, h, wd, pad=1):
    """dE/dx of conv3x3_fwd: the adjoint map.
    dx[n,i,j,ci] = sum_{kh,kw,co} dy[n, i-kh+pad, j-kw+pad, co] * w[co,kh,kw,ci]
    (terms with an output index outside the output are absent).
    Pinned by the adjoint identity <conv(x), y> = <x, conv_dx(y)> and by
    finite differences."""
    dy = np.asarray(dy, F64)
    w = np.asarray(w, F64)
    n, ho, wo, co = dy.shape
    dxp = np.zeros((n, h + 2 * pad, wd + 2 * pad, w.shape[3]), F64)
    for kh in range(3):
        for kw in range(3):
            dxp[:, kh:kh + ho, kw:kw + wo, :] += dy @ w[:, kh, kw, :]
    return dxp[:, pad:pad + h, pad:pad + wd, :]


def conv3x3_dw(x, dy, pad=1):
    """dE/dw and dE/db of conv3x3_fwd ([S] 'dedw' and 'dedb' roles):
    dw[co,kh,kw,ci] = sum_{n,oh,ow} dy[n,oh,ow,co] * x[n, oh+kh-pad, ow+kw-pad, ci]
    db[co]          = sum_{n,oh,ow} dy[n,oh,ow,co].
    Pinned by the adjoint identity <dw(x,y), w> = <conv(x; w, no bias), y> and
    by finite differences."""
    x = np.asarray(x, F64)
    dy = np.asarray(dy, F64)
    n, ho, wo, co = dy.shape
    xp = _pad_hw(x, pad)
    dw = np.zeros((co, 3, 3, x.shape[3]), F64)
    for kh in range(3):
        for kw in range(3):
            dw[:, kh, kw, :] = np.tensordot(dy, xp[:, kh:kh + ho, kw:kw + wo, :], axes=([0, 1, 2], [0, 1, 2]))
    return dw, dy.sum(axis=(0, 1, 2))


def im2col(x, pad=1):
    """The im2col unrolling of [S] Sec. 3.3 / Eq. (5): one row per output pixel
    (n, oh, ow) in NHWC order, one column per (kh, kw, ci) (K index
    (kh*3+kw)*C + ci). Returns (col, src_index) where src_index is the flat
    NHWC index of the source element in x, or -1 for zero padding.
    Pinned by brute-force enumeration and by conv3x3_fwd == col @ w^T."""
    n, h, wd, c = x.shape
    ho, wo = h + 2 * pad - 2, wd + 2 * pad - 2
    src = np.full((n, ho, wo, 3, 3, c), -1, np.int64)
    nn, oh, ow, kh, kw, ci = np.meshgrid(np.arange(n), np.arange(ho), np.arange(wo), np.arange(3), np.arange(3),
                                         np.arange(c), indexing="ij")
    ih, iw = oh + kh - pad, ow + kw - pad
    ok = (ih >= 0) & (ih < h) & (iw >= 0) & (iw < wd)
    src[ok] = ((nn[ok] * h + ih[ok]) * wd + iw[ok]) * c + ci[ok]
    src = src.reshape(n * ho * wo, 9 * c)
    flat = np.asarray(x).reshape(-1)
    col = np.where(src >= 0, flat[np.maximum(src, 0)], 0).astype(np.asarray(x).dtype)
    return col, src.astype(np.int32)


# ---------------------------------------------------------------------------
# ReLU and 2x2 max-pool — [S] Sec. 3.2 (conv, ReLU, optional pooling p_l)
# ---------------------------------------------------------------------------

def relu(x):
    return np.maximum(np.asarray(x, F64), 0.0)


def relu_mask(y):
    """Derivative of ReLU read off its output: 1 where y > 0, else 0 (R11)."""
    return (np.asarray(y) > 0).astype(F64)


def maxpool2x2_fwd(x):
    """2x2, stride-2 max-pool. Argmax codes 0..3 = 2*dy + dx of the first window
    element, in row-major order, that is strictly greater than all before it
    (R10). Odd trailing rows/columns are dropped. Pinned by brute force."""
    x = np.asarray(x)
    n, h, w, c = x.shape
    ho, wo = h // 2, w // 2
    best = x[:, 0:2 * ho:2, 0:2 * wo:2, :].astype(F64)
    arg = np.zeros((n, ho, wo, c), np.uint8)
    for code in (1, 2, 3):
        dy, dx = divmod(code, 2)
        v = x[:, dy:2 * ho:2, dx:2 * wo:2, :].astype(F64)
        gt = v > best
        best = np.where(gt, v, best)
        arg[gt] = code
    return best, arg


def maxpool2x2_bwd(dy, arg, h, w):
    """Routes each output gradient to the window element the forward pass picked."""
    dy = np.asarray(dy, F64)
    n, ho, wo, c = dy.shape
    dx = np.zeros((n, h, w, c), F64)
    for code in range(4):
        oy, ox = divmod(code, 2)
        sel = (arg == code)
        dx[:, oy:2 * ho:2, ox:2 * wo:2, :] += np.where(sel, dy, 0.0)
    return dx


# ---------------------------------------------------------------------------
# Fully connected layer — [S] Sec. 3.3 'fc', 'dedx fc', 'dedw', 'dedb'
# ---------------------------------------------------------------------------

def fc_fwd(x, w, b):
    """y = x W^T + b, x [N][in], W [out][in]."""
    return np.asarray(x, F64) @ np.asarray(w, F64).T + np.asarray(b, F64)


def fc_bwd(x, w, dy):
    """dx = dy W, dW = dy^T x, db = sum_n dy[n]."""
    x, w, dy = (np.asarray(a, F64) for a in (x, w, dy))
    return dy @ w, dy.T @ x, dy.sum(axis=0)


# ---------------------------------------------------------------------------
# Softmax cross-entropy — the softmax output layer of [S] Sec. 3.2; [Q] Sec. 6
# uses the batch-mean softmax_cross_entropy (R1)
# ---------------------------------------------------------------------------

def softmax_xent(z, labels, reduction="mean"):
    """loss = mean_i [logsumexp(z_i) - z_i[y_i]], dz = (softmax(z) - onehot(y)) / N.
    Pinned by: uniform logits give ln C exactly, dz rows sum to 0, finite
    differences."""
    z = np.asarray(z, F64)
    n = z.shape[0]
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    s = e.sum(axis=1, keepdims=True)
    lse = (m + np.log(s))[:, 0]
    picked = z[np.arange(n), labels]
    p = e / s
    onehot = np.zeros_like(z)
    onehot[np.arange(n), labels] = 1.0
    if reduction == "mean":
        return float(np.mean(lse - picked)), (p - onehot) / n
    return float(np.sum(lse - picked)), (p - onehot)


# ---------------------------------------------------------------------------
# Worker step: forward, loss, backward (Algorithm 1 'ComputeGradient' of [S])
# ---------------------------------------------------------------------------

def forward(layers: list[Layer], params, x):
    """Forward pass; returns (logits, saved) with saved[i] = (input of layer i,
    its output after ReLU (before pooling), pool argmax or None).

    ``params`` is a list of (W, b) per layer; each layer may come from a
    different weight version (pipeline stages, R8). Conv layers: y = ReLU(conv + b),
    then optional 2x2 max-pool. FC layers: y = xW^T + b, ReLU unless the layer
    says otherwise. The input of the first FC layer is the NHWC activation
    flattened in (h, w, c) order."""
    a = np.asarray(x, F64)
    n = a.shape[0]
    if layers[0].kind == "fc":
        a = a.reshape(n, -1)
    saved = []
    for L, (w, b) in zip(layers, params):
        if L.kind == "conv":
            y = relu(conv3x3_fwd(a, w, b))
            if L.pool:
                p, arg = maxpool2x2_fwd(y)
                saved.append((a, y, arg))
                a = p
            else:
                saved.append((a, y, None))
                a = y
        else:
            if a.ndim == 4:
                a = a.reshape(n, -1)
            z = fc_fwd(a, w, b)
            y = relu(z) if L.relu else z
            saved.append((a, y, None))
            a = y
    return a, saved


def backward(layers: list[Layer], params, saved, g):
    """Backward pass by hand, layer by layer, from dE/dlogits ``g``; returns
    the per-layer (dW, db). Every decision it takes (ReLU derivative = 1 where
    the saved output is > 0, R11; the pool argmax, R10) is read from ``saved``,
    so it can be replayed on another implementation's saved activations."""
    grads = [None] * len(layers)
    g = np.asarray(g, F64)
    for i in range(len(layers) - 1, -1, -1):
        L = layers[i]
        w, _ = params[i]
        xin, y, arg = saved[i]
        xin = np.asarray(xin, F64)
        if L.kind == "fc":
            if L.relu:
                g = g * relu_mask(y)
            dx, dw, db = fc_bwd(xin, w, g)
            grads[i] = (dw, db)
            g = dx
            if i > 0 and layers[i - 1].kind == "conv":
                g = g.reshape(xin.shape[0], *_out_hw(layers[i - 1]), layers[i - 1].cout)
        else:
            if L.pool:
                g = maxpool2x2_bwd(g, arg, y.shape[1], y.shape[2])
            g = g * relu_mask(y)
            dw, db = conv3x3_dw(xin, g)
            grads[i] = (dw, db)
            if i > 0:
                g = conv3x3_dx(g, w, xin.shape[1], xin.shape[2])
    return grads


def forward_backward(layers: list[Layer], params, x, labels, reduction="mean"):
    """Loss and per-layer (dW, db) for one batch (forward, softmax
    cross-entropy, backward). Pinned by central finite differences."""
    logits, saved = forward(layers, params, x)
    loss, g = softmax_xent(logits, labels, reduction)
    return loss, backward(layers, params, saved, g)


def _out_hw(L: Layer):
    return (L.h // 2, L.w // 2) if L.pool else (L.h, L.w)


def gradient(layers, flat_params, x, labels, reduction="mean"):
    """Flat gradient of the loss at one weight version."""
    loss, grads = forward_backward(layers, unflatten(layers, np.asarray(flat_params, F64)), x, labels, reduction)
    return loss, flatten(grads)


# ---------------------------------------------------------------------------
# GradBuf and parameter-server update — Algorithm 1 (UpdateGradient) and
# Algorithm 2 (SumGradient, momentum, UpdateWeights) of [S]; [DB] w' := w - eta dw
# ---------------------------------------------------------------------------

def gradbuf_accumulate(buf, grad, alpha=1.0, first=False):
    """GradBuf <- alpha*grad if the buffer is empty, else GradBuf + alpha*grad
    (Algorithm 1 of [S]: assign when empty, add otherwise)."""
    g = alpha * np.asarray(grad, F64)
    return g if first else np.asarray(buf, F64) + g


def sum_buffers(bufs):
    """SendBuf = sum_t GradBuf_t, in buffer order (Algorithm 2 of [S])."""
    s = np.zeros(np.asarray(bufs[0]).shape, F64)
    for b in bufs:
        s = s + np.asarray(b, F64)
    return s


def decayed_sum(w, bufs, weight_decay=0.0):
    """S = sum of the buffers, plus lambda*W when weight decay is on (R12)."""
    s = sum_buffers(bufs)
    if weight_decay:
        s = s + weight_decay * np.asarray(w, F64)
    return s


def update_sgd(w, bufs, eta, weight_decay=0.0):
    """W' = W - eta * S   (Eq. (1) of [S] with S the summed gradient; [DB])."""
    return np.asarray(w, F64) - eta * decayed_sum(w, bufs, weight_decay)


def update_momentum(w, v, bufs, eta, nu, weight_decay=0.0):
    """v' = nu*v - eta*S, W' = W + v'  (Algorithm 2 of [S] with DeltaWeights = v, R5)."""
    v_new = nu * np.asarray(v, F64) - eta * decayed_sum(w, bufs, weight_decay)
    return np.asarray(w, F64) + v_new, v_new


def update_nesterov(w, v, bufs, eta, nu, weight_decay=0.0):
    """v' = nu*v - eta*S, W' = W + nu*v' - eta*S  (Nesterov momentum, R11)."""
    s = decayed_sum(w, bufs, weight_decay)
    v_new = nu * np.asarray(v, F64) - eta * s
    return np.asarray(w, F64) + nu * v_new - eta * s, v_new


def update_adagrad(w, g2, bufs, eta, eps, weight_decay=0.0):
    """G' = G + S*S, W' = W - eta*S/(sqrt(G') + eps)  (per-parameter rate of [DB], R6)."""
    s = decayed_sum(w, bufs, weight_decay)
    g_new = np.asarray(g2, F64) + s * s
    return np.asarray(w, F64) - eta * s / (np.sqrt(g_new) + eps), g_new


# ---------------------------------------------------------------------------
# Staleness schedule — SplitMix64 (Steele, Lea & Flood, OOPSLA 2014), R7
# ---------------------------------------------------------------------------

def splitmix64_mix(z: int) -> int:
    """The SplitMix64 output function (the variant of Stafford's Mix13)."""
    z &= _M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _M64
    return z ^ (z >> 31)


def splitmix64_at(seed: int, i: int) -> int:
    """The i-th output (i = 0, 1, ...) of a SplitMix64 generator seeded with
    ``seed``: the state advances by the golden gamma before each output."""
    return splitmix64_mix((seed + (i + 1) * _GAMMA) & _M64)


def staleness_schedule(seed: int, steps: int, replicas: int, max_delay: int) -> np.ndarray:
    """Delay s[t, r] in {0..max_delay} for replica r at step t: the
    (t*replicas + r)-th SplitMix64 output z, reduced by (hi32(z) * (S+1)) >> 32."""
    out = np.zeros((steps, replicas), np.int32)
    for t in range(steps):
        for r in range(replicas):
            z = splitmix64_at(seed, t * replicas + r)
            out[t, r] = ((z >> 32) * (max_delay + 1)) >> 32
    return out


def version_used(t: int, s: int) -> int:
    """Weights 's steps old' at step t are W(max(0, t - s)) (R7)."""
    return max(0, t - s)


# ---------------------------------------------------------------------------
# Stale-weight training driver (ASGD replicas [S] Fig. 1 / [DB]; pipeline [PB] 4.1)
# ---------------------------------------------------------------------------

def stage_delay(stage_delays, k, t, hybrid_switch=None):
    """Delay of pipeline stage k at step t: s_k, or 0 from step N_p on in
    hybrid training (R13)."""
    if hybrid_switch is not None and t >= hybrid_switch:
        return 0
    return int(stage_delays[k])


def staleness_degrees(stage_delays):
    """Degree of staleness of each stage pair: the steps its weights lag (R13)."""
    return [int(s) for s in stage_delays]


def stale_weight_percent(layers, stage_of_layer, stage_delays):
    """Percentage of the parameters (W and b) held by layers whose stage uses
    stale weights (s_k > 0), R13 / [PB] Sec. 4.1."""
    stale = total = 0
    for li, L in enumerate(layers):
        n = int(np.prod(L.w_shape)) + L.cout
        total += n
        if stage_delays[stage_of_layer[li]] > 0:
            stale += n
    return 100.0 * stale / total


def replica_params(layers, hist, t, r, *, schedule=None, stage_delays=None, stage_of_layer=None, hybrid_switch=None):
    """Per-layer (W, b) that replica r uses at step t: W(max(0, t - s[t, r]))
    for asynchronous replicas (R7), or W_l(max(0, t - s_k)) for the layers of
    pipeline stage k (R8; s_k = 0 from step N_p on in hybrid training, R13)."""
    offs, _ = param_offsets(layers)
    params = []
    for li, L in enumerate(layers):
        if stage_delays is not None:
            ver = version_used(t, stage_delay(stage_delays, stage_of_layer[li], t, hybrid_switch))
        else:
            ver = version_used(t, 0 if schedule is None else int(schedule[t, r]))
        a, b = offs[li]
        params.append((hist[ver][a:b].reshape(L.w_shape), hist[ver][b:b + L.cout]))
    return params


def step_gradients(layers, hist, t, batches, *, replicas=1, schedule=None, stage_delays=None, stage_of_layer=None,
                   reduction="mean", hybrid_switch=None):
    """Per-replica (loss, flat gradient) of global step t, given the weight
    history hist[0..t] (hist[v] = W(v)).

    Replica r draws batch (t*R + r) mod len(batches) and computes its gradient
    at W(max(0, t - s[t, r])) (``schedule``), or, for a pipeline, every layer l
    of stage k at W_l(max(0, t - s_k)) (``stage_delays``, ``stage_of_layer``)."""
    losses, grads = [], []
    for r in range(replicas):
        x, y = batches[(t * replicas + r) % len(batches)]
        params = replica_params(layers, hist, t, r, schedule=schedule, stage_delays=stage_delays,
                                stage_of_layer=stage_of_layer, hybrid_switch=hybrid_switch)
        loss, gl = forward_backward(layers, params, x, y, reduction)
        losses.append(loss)
        grads.append(flatten(gl))
    return losses, grads


def apply_update(w, grads, optimizer="sgd", eta=0.01, nu=0.9, eps=1e-8, state=None, weight_decay=0.0):
    """The parameter-server apply of the summed gradients; returns (W', state')."""
    if optimizer == "sgd":
        return update_sgd(w, grads, eta, weight_decay), state
    if optimizer == "momentum":
        return update_momentum(w, state, grads, eta, nu, weight_decay)
    if optimizer == "nesterov":
        return update_nesterov(w, state, grads, eta, nu, weight_decay)
    if optimizer == "adagrad":
        return update_adagrad(w, state, grads, eta, eps, weight_decay)
    raise ValueError(optimizer)


def train_step(layers, hist, t, batches, *, replicas=1, schedule=None, stage_delays=None, stage_of_layer=None,
               optimizer="sgd", eta=0.01, nu=0.9, eps=1e-8, state=None, reduction="mean", hybrid_switch=None,
               weight_decay=0.0):
    """One global step: the R replica gradients (step_gradients), summed in
    replica order and applied once (apply_update) with the optimizer state
    before the step (momentum / Nesterov v or Adagrad G; ignored for SGD).
    Returns (mean loss over replicas, W(t+1), new state)."""
    losses, grads = step_gradients(layers, hist, t, batches, replicas=replicas, schedule=schedule,
                                   stage_delays=stage_delays, stage_of_layer=stage_of_layer, reduction=reduction,
                                   hybrid_switch=hybrid_switch)
    w_new, state = apply_update(hist[t], grads, optimizer, eta, nu, eps, state, weight_decay)
    return sum(losses) / replicas, w_new, state


def initial_state(optimizer, n, g0=0.1):
    """v0 = 0 for momentum and Nesterov, G0 = g0 for Adagrad, none for SGD."""
    if optimizer in ("momentum", "nesterov"):
        return np.zeros(n, F64)
    if optimizer == "adagrad":
        return np.full(n, g0, F64)
    return None


def train(arch, w0, batches, steps, *, replicas=1, schedule=None, stage_delays=None, stage_of_layer=None,
          optimizer="sgd", eta=0.01, nu=0.9, eps=1e-8, g0=0.1, reduction="mean", hybrid_switch=None,
          weight_decay=0.0):
    """Simulated asynchronous training from W(0) = w0; returns (per-step mean
    loss, final W, history). The full history of W is kept, which is the plain
    brute-force way to look up old versions."""
    layers = build_layers(arch)
    _, n = param_offsets(layers)
    hist = [np.asarray(w0, F64).copy()]
    state = initial_state(optimizer, n, g0)
    losses = []
    for t in range(steps):
        loss, w_new, state = train_step(layers, hist, t, batches, replicas=replicas, schedule=schedule,
                                        stage_delays=stage_delays, stage_of_layer=stage_of_layer, optimizer=optimizer,
                                        eta=eta, nu=nu, eps=eps, state=state, reduction=reduction,
                                        hybrid_switch=hybrid_switch, weight_decay=weight_decay)
        losses.append(loss)
        hist.append(w_new)
    return losses, hist[-1], hist


def train_fetch_push(arch, w0, batches, steps, *, replicas=1, n_fetch=1, n_push=1, optimizer="sgd", eta=0.01,
                     nu=0.9, eps=1e-8, g0=0.1, reduction="mean", weight_decay=0.0):
    """DistBelief-style training with n_fetch / n_push (R14), step by step as
    the rule reads: refresh the local copies, compute and accumulate every
    replica's gradient, and at a push step apply the R buffers. Returns
    (per-step mean loss, final server W, the server W after each update)."""
    layers = build_layers(arch)
    _, n = param_offsets(layers)
    w = np.asarray(w0, F64).copy()
    state = initial_state(optimizer, n, g0)
    local = [None] * replicas
    bufs = [None] * replicas
    losses, versions = [], [w]
    for t in range(steps):
        if t % n_fetch == 0:
            local = [w.copy() for _ in range(replicas)]
        step_losses = []
        for r in range(replicas):
            x, y = batches[(t * replicas + r) % len(batches)]
            loss, gl = forward_backward(layers, unflatten(layers, local[r]), x, y, reduction)
            step_losses.append(loss)
            bufs[r] = gradbuf_accumulate(bufs[r], flatten(gl), 1.0, first=(t % n_push == 0))
        losses.append(sum(step_losses) / replicas)
        if (t + 1) % n_push == 0:
            w, state = apply_update(w, bufs, optimizer, eta, nu, eps, state, weight_decay)
            versions.append(w)
    return losses, w, versions


def flops_per_image(arch) -> float:
    """Training FLOPs per image: forward + dW + dX GEMM work (2 per MAC), no dX
    for the first layer; the count the throughput figures use."""
    layers = build_layers(arch)
    f = 0.0
    for i, L in enumerate(layers):
        macs = (L.h * L.w * L.cout * 9 * L.cin) if L.kind == "conv" else L.cout * L.cin
        f += 2 * macs * (2 if i == 0 else 3)
    return f


def he_std(L: Layer) -> float:
    return math.sqrt(2.0 / L.fan_in)
