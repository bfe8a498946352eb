"""Pins of the FP64 oracle against what the pages and the mathematics fix.

None of these re-types the oracle's own formula: each compares it with an
independent route (brute force, an adjoint identity, finite differences, a
closed form, a published vector, a special case)."""
import math
import os

import numpy as np
import pytest

import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# small architectures for exhaustive / finite-difference checks
SMALL_CNN = dict(input=(3, 8, 8), layers=[("conv", 4, True), ("conv", 5, False), ("conv", 4, True), ("fc", 6, True), ("fc", 5, False)])
SMALL_MLP = dict(input=(12, 1, 1), layers=[("fc", 9, True), ("fc", 7, True), ("fc", 4, False)])


def _brute_conv(x, w, b, pad):
    n, h, wd, ci = x.shape
    co = w.shape[0]
    ho, wo = h + 2 * pad - 2, wd + 2 * pad - 2
    y = np.zeros((n, ho, wo, co))
    for a in range(n):
        for oh in range(ho):
            for ow in range(wo):
                for o in range(co):
                    s = float(b[o])
                    for kh in range(3):
                        for kw in range(3):
                            ih, iw = oh + kh - pad, ow + kw - pad
                            if 0 <= ih < h and 0 <= iw < wd:
                                for c in range(ci):
                                    s += float(x[a, ih, iw, c]) * float(w[o, kh, kw, c])
                    y[a, oh, ow, o] = s
    return y


# ---------------------------------------------------------------- SplitMix64

def test_splitmix64_published_vectors():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "splitmix64.txt")) if l.strip() and not l.startswith("#")]
    assert len(rows) == 9
    for seed, i, hexv in rows:
        assert O.splitmix64_at(int(seed), int(i)) == int(hexv, 16)


def test_schedule_range_and_uniformity():
    S = 7
    s = O.staleness_schedule(1234, 500, 8, S)
    assert s.dtype == np.int32 and s.shape == (500, 8)
    assert s.min() == 0 and s.max() == S
    counts = np.bincount(s.ravel(), minlength=S + 1)
    exp = s.size / (S + 1)
    chi2 = float(((counts - exp) ** 2 / exp).sum())
    assert chi2 < 30.0  # 7 dof; p ~ 1e-4 threshold
    assert (O.staleness_schedule(5, 10, 3, 0) == 0).all()


def test_schedule_is_counter_based():
    # entry (t, r) depends only on (seed, t*R + r): a longer schedule extends a shorter one
    a = O.staleness_schedule(99, 4, 3, 5)
    b = O.staleness_schedule(99, 9, 3, 5)
    assert (a == b[:4]).all()


# ---------------------------------------------------------------- Eq. (2), (3)

def test_param_count_eq3_matches_tensor_sizes():
    for name, arch in O.ARCHS.items():
        layers = O.build_layers(arch)
        assert O.param_count_eq3(arch) == O.param_offsets(layers)[1], name
    # tiny: 16*(27+1) + 32*(144+1) + 10*(2048+1); VGG-16 ILSVRC: the widely quoted 138,357,544
    assert O.param_count_eq3(O.ARCHS["tiny"]) == 16 * 28 + 32 * 145 + 10 * 2049 == 25578
    assert O.param_count_eq3(O.ARCHS["smlps"]) == 3072 * 5000 + 5000 + 4 * (5000 * 5000 + 5000) + 5000 * 10 + 10
    assert O.param_count_eq3(O.ARCHS["vgg_i"]) == 138357544
    assert O.param_count_eq3(O.ARCHS["vgg_c"]) == 15245130


def test_spatial_sizes_eq2_fc_inputs():
    # the FC input sizes the configurations name: 2048 (tiny), 512 (VGG-C), 25088 (VGG-I)
    for name, fin in (("tiny", 2048), ("vgg_c", 512), ("vgg_i", 25088)):
        layers = O.build_layers(O.ARCHS[name])
        first_fc = next(L for L in layers if L.kind == "fc")
        assert first_fc.cin == fin, name
    assert O.spatial_sizes_eq2(O.ARCHS["vgg_i"])[:14] == [224, 224, 112, 112, 56, 56, 56, 28, 28, 28, 14, 14, 14, 7]


# ---------------------------------------------------------------- convolution

@pytest.mark.parametrize("pad", [1, 0])
def test_conv_fwd_brute_force(pad):
    x = synth.normal(1, "x", (2, 5, 4, 3)).astype(np.float64)
    w = synth.normal(1, "w", (2, 3, 3, 3)).astype(np.float64)
    b = synth.normal(1, "b", (2,)).astype(np.float64)
    np.testing.assert_allclose(O.conv3x3_fwd(x, w, b, pad), _brute_conv(x, w, b, pad), rtol=0, atol=1e-12)


def test_conv_fwd_im2col_route():
    x = synth.normal(2, "x", (3, 6, 7, 5)).astype(np.float64)
    w = synth.normal(2, "w", (4, 3, 3, 5)).astype(np.float64)
    b = synth.normal(2, "b", (4,)).astype(np.float64)
    col, _ = O.im2col(x)
    y2 = (col @ w.reshape(4, -1).T + b).reshape(3, 6, 7, 4)
    np.testing.assert_allclose(O.conv3x3_fwd(x, w, b), y2, rtol=0, atol=1e-12)


def test_conv_centre_tap_is_pointwise_matmul():
    x = synth.normal(3, "x", (2, 4, 4, 3)).astype(np.float64)
    w = np.zeros((5, 3, 3, 3))
    w[:, 1, 1, :] = synth.normal(3, "wc", (5, 3))
    b = synth.normal(3, "b", (5,)).astype(np.float64)
    np.testing.assert_allclose(O.conv3x3_fwd(x, w, b), x @ w[:, 1, 1, :].T + b, rtol=0, atol=1e-12)


def test_conv_impulse_reads_back_weights():
    x = np.zeros((1, 5, 5, 2))
    x[0, 2, 3, 1] = 1.0
    w = synth.normal(4, "w", (3, 3, 3, 2)).astype(np.float64)
    y = O.conv3x3_fwd(x, w, None)
    for kh in range(3):
        for kw in range(3):
            np.testing.assert_array_equal(y[0, 2 - kh + 1, 3 - kw + 1, :], w[:, kh, kw, 1])


def test_conv_adjoint_identities():
    x = synth.normal(5, "x", (2, 6, 5, 3)).astype(np.float64)
    w = synth.normal(5, "w", (4, 3, 3, 3)).astype(np.float64)
    y = synth.normal(5, "y", (2, 6, 5, 4)).astype(np.float64)
    lhs = np.vdot(O.conv3x3_fwd(x, w, None), y)
    assert abs(lhs - np.vdot(x, O.conv3x3_dx(y, w, 6, 5))) < 1e-12 * abs(lhs) + 1e-12
    dw, db = O.conv3x3_dw(x, y)
    assert abs(np.vdot(dw, w) - lhs) < 1e-12 * abs(lhs) + 1e-12
    np.testing.assert_allclose(db, y.sum(axis=(0, 1, 2)), rtol=1e-14)


@pytest.mark.parametrize("pad", [0, 1])
def test_conv_dw_brute_force(pad):
    """dedw / dedb of [S] Sec. 3.3 by explicit loops over every output pixel and
    tap, skipping taps that fall outside the image (the few-channel shapes of
    the RGB layer, both paddings)."""
    x = synth.normal(21, "x", (2, 5, 7, 3)).astype(np.float64)
    n, h, wd, ci = x.shape
    ho, wo = h + 2 * pad - 2, wd + 2 * pad - 2
    dy = synth.normal(21, "dy", (n, ho, wo, 4)).astype(np.float64)
    dw_ref = np.zeros((4, 3, 3, ci))
    db_ref = np.zeros(4)
    for a in range(n):
        for oh in range(ho):
            for ow in range(wo):
                for co in range(4):
                    g = dy[a, oh, ow, co]
                    db_ref[co] += g
                    for kh in range(3):
                        for kw in range(3):
                            ih, iw = oh + kh - pad, ow + kw - pad
                            if 0 <= ih < h and 0 <= iw < wd:
                                for c in range(ci):
                                    dw_ref[co, kh, kw, c] += g * x[a, ih, iw, c]
    dw, db = O.conv3x3_dw(x, dy, pad=pad)
    np.testing.assert_allclose(dw, dw_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(db, db_ref, rtol=0, atol=1e-12)


def test_conv_adjoint_identities_pad0():
    x = synth.normal(22, "x", (2, 6, 5, 2)).astype(np.float64)
    w = synth.normal(22, "w", (3, 3, 3, 2)).astype(np.float64)
    y = synth.normal(22, "y", (2, 4, 3, 3)).astype(np.float64)
    lhs = np.vdot(O.conv3x3_fwd(x, w, None, pad=0), y)
    assert abs(lhs - np.vdot(x, O.conv3x3_dx(y, w, 6, 5, pad=0))) < 1e-12 * abs(lhs) + 1e-12
    dw, _ = O.conv3x3_dw(x, y, pad=0)
    assert abs(np.vdot(dw, w) - lhs) < 1e-12 * abs(lhs) + 1e-12


def test_im2col_brute_force_index_map():
    x = synth.normal(6, "x", (2, 3, 4, 2))
    col, src = O.im2col(x)
    n, h, w, c = x.shape
    r = 0
    for a in range(n):
        for oh in range(h):
            for ow in range(w):
                k = 0
                for kh in range(3):
                    for kw in range(3):
                        for ci in range(c):
                            ih, iw = oh + kh - 1, ow + kw - 1
                            if 0 <= ih < h and 0 <= iw < w:
                                assert src[r, k] == ((a * h + ih) * w + iw) * c + ci
                                assert col[r, k] == x[a, ih, iw, ci]
                            else:
                                assert src[r, k] == -1 and col[r, k] == 0
                            k += 1
                r += 1


# ---------------------------------------------------------------- pool / relu

def test_pool_brute_force_with_ties():
    x = synth.normal(7, "x", (2, 6, 4, 3))
    x[0, 0:2, 0:2, 0] = 0.0          # all-zero window -> argmax 0
    x[1, 2:4, 2:4, 1] = 0.5          # all-equal window
    x[0, 2, 1, 2] = x[0, 3, 0, 2] = 9.0  # tie between codes 1 and 2 -> first (1)
    y, arg = O.maxpool2x2_fwd(x)
    for a in range(2):
        for i in range(3):
            for j in range(2):
                for c in range(3):
                    win = [x[a, 2 * i + dy, 2 * j + dx, c] for dy in range(2) for dx in range(2)]
                    best = 0
                    for k in range(1, 4):
                        if win[k] > win[best]:
                            best = k
                    assert arg[a, i, j, c] == best and y[a, i, j, c] == win[best]
    assert arg[0, 0, 0, 0] == 0 and arg[1, 1, 1, 1] == 0 and arg[0, 1, 0, 2] == 1


def test_pool_bwd_routes_to_argmax():
    x = synth.normal(8, "x", (1, 4, 6, 2))
    y, arg = O.maxpool2x2_fwd(x)
    dy = synth.normal(8, "dy", y.shape).astype(np.float64)
    dx = O.maxpool2x2_bwd(dy, arg, 4, 6)
    # adjoint of the linear map "pick the argmax element"
    assert abs(np.vdot(dx, x) - np.vdot(dy, y)) < 1e-12
    assert np.count_nonzero(dx) == dy.size


# ---------------------------------------------------------------- softmax

def test_softmax_uniform_logits_give_ln_c():
    for c in (10, 1000):
        z = np.full((4, c), 3.25)
        loss, dz = O.softmax_xent(z, np.arange(4) % c)
        assert loss == pytest.approx(math.log(c), rel=0, abs=1e-14)
        np.testing.assert_allclose(dz.sum(axis=1), 0, atol=1e-15)


def test_softmax_fd_and_stability():
    z = synth.normal(9, "z", (5, 7)).astype(np.float64) * 3
    y = synth.labels(9, "y", 5, 7)
    loss, dz = O.softmax_xent(z, y)
    h = 1e-6
    for (i, j) in [(0, 0), (1, 3), (4, 6), (2, int(y[2]))]:
        zp, zm = z.copy(), z.copy()
        zp[i, j] += h
        zm[i, j] -= h
        fd = (O.softmax_xent(zp, y)[0] - O.softmax_xent(zm, y)[0]) / (2 * h)
        assert fd == pytest.approx(dz[i, j], abs=1e-8)
    big = z + 1e4   # shift invariance, no overflow
    assert O.softmax_xent(big, y)[0] == pytest.approx(loss, abs=1e-9)


# ---------------------------------------------------------------- whole network

@pytest.mark.parametrize("arch", [SMALL_CNN, SMALL_MLP], ids=["cnn", "mlp"])
def test_network_gradient_finite_differences(arch):
    layers = O.build_layers(arch)
    _, n = O.param_offsets(layers)
    w = np.concatenate([np.concatenate([synth.normal(10, f"w{i}", L.w_shape, O.he_std(L)).ravel(),
                                        synth.normal(10, f"b{i}", (L.cout,), 0.1)]) for i, L in enumerate(layers)]).astype(np.float64)
    c, h, wd = arch["input"]
    x = synth.images_nhwc(10, "x", 3, c, h, wd)
    if layers[0].kind == "fc":
        x = x.reshape(3, -1)
    y = synth.labels(10, "y", 3, layers[-1].cout)
    loss, g = O.gradient(layers, w, x, y)
    idx = synth.rng(10, "idx").choice(n, size=40, replace=False)
    hstep = 1e-6
    for i in idx:
        wp, wm = w.copy(), w.copy()
        wp[i] += hstep
        wm[i] -= hstep
        fd = (O.gradient(layers, wp, x, y)[0] - O.gradient(layers, wm, x, y)[0]) / (2 * hstep)
        assert fd == pytest.approx(g[i], abs=2e-7 + 1e-5 * abs(g[i])), i


def test_fc_first_layer_input_gradient_fd():
    # dX of the FC layer (dedx fc) pinned through a two-layer net's input gradient
    w1 = synth.normal(11, "w1", (4, 6)).astype(np.float64)
    w2 = synth.normal(11, "w2", (3, 4)).astype(np.float64)
    x = synth.normal(11, "x", (2, 6)).astype(np.float64)
    y = np.array([0, 2])

    def f(xx):
        h = O.relu(O.fc_fwd(xx, w1, np.zeros(4)))
        return O.softmax_xent(O.fc_fwd(h, w2, np.zeros(3)), y)[0]
    h = O.relu(O.fc_fwd(x, w1, np.zeros(4)))
    _, dz = O.softmax_xent(O.fc_fwd(h, w2, np.zeros(3)), y)
    dh = O.fc_bwd(h, w2, dz)[0] * O.relu_mask(h)
    dx = O.fc_bwd(x, w1, dh)[0]
    for i in range(2):
        for j in range(6):
            xp, xm = x.copy(), x.copy()
            xp[i, j] += 1e-6
            xm[i, j] -= 1e-6
            assert (f(xp) - f(xm)) / 2e-6 == pytest.approx(dx[i, j], abs=1e-8)


# ---------------------------------------------------------------- updates

def test_sgd_single_step_exact_dyadic():
    w = synth.dyadic(12, "w", 64).astype(np.float64)
    bufs = [synth.dyadic(12, f"g{j}", 64).astype(np.float64) for j in range(3)]
    eta = 2.0 ** -4
    out = O.update_sgd(w, bufs, eta)
    for i in range(64):
        assert out[i] == w[i] - eta * (bufs[0][i] + bufs[1][i] + bufs[2][i])


def test_momentum_constant_gradient_closed_form():
    w0, g, eta, nu, T = 0.7, 0.3, 0.01, 0.9, 25
    w, v = np.array([w0]), np.array([0.0])
    for _ in range(T):
        w, v = O.update_momentum(w, v, [np.array([g])], eta, nu)
    closed = w0 - eta * g * sum((1 - nu ** t) / (1 - nu) for t in range(1, T + 1))
    assert w[0] == pytest.approx(closed, rel=1e-13)
    # nu = 0 reduces to plain SGD
    w1, _ = O.update_momentum(np.array([w0]), np.array([5.0]), [np.array([g])], eta, 0.0)
    assert w1[0] == pytest.approx(w0 - eta * g, rel=1e-15)


def test_adagrad_constant_gradient_closed_form():
    w0, g, eta, eps, g0, T = -0.2, 0.05, 0.01, 1e-8, 0.1, 30
    w, G = np.array([w0]), np.array([g0])
    for _ in range(T):
        w, G = O.update_adagrad(w, G, [np.array([g / 2]), np.array([g / 2])], eta, eps)
    closed = w0 - eta * g * sum(1.0 / (math.sqrt(g0 + t * g * g) + eps) for t in range(1, T + 1))
    assert w[0] == pytest.approx(closed, rel=1e-13)
    assert G[0] == pytest.approx(g0 + T * g * g, rel=1e-14)


def test_gradbuf_assign_then_add():
    g1, g2 = np.array([1.0, -2.0]), np.array([0.5, 0.25])
    b = O.gradbuf_accumulate(np.array([99.0, 99.0]), g1, 1.0, first=True)
    assert (b == g1).all()
    b = O.gradbuf_accumulate(b, g2, -0.5, first=False)
    assert (b == g1 - 0.5 * g2).all()


def test_order_invariance_dyadic_exact():
    bufs = [synth.dyadic(13, f"g{j}", 1000).astype(np.float64) for j in range(16)]
    w = synth.dyadic(13, "w", 1000).astype(np.float64)
    a = O.update_sgd(w, bufs, 2.0 ** -3)
    perm = synth.rng(13, "perm").permutation(16)
    b = O.update_sgd(w, [bufs[i] for i in perm], 2.0 ** -3)
    assert (a == b).all()


# ---------------------------------------------------------------- replicas / staleness

def _init(arch, seed=20):
    layers = O.build_layers(arch)
    return np.concatenate([np.concatenate([synth.normal(seed, f"w{i}", L.w_shape, O.he_std(L)).ravel(),
                                           np.zeros(L.cout)]) for i, L in enumerate(layers)]).astype(np.float64)


def _batches(arch, count, n, seed=21):
    c, h, w = arch["input"]
    out = synth.batch_pool(seed, count, n, c, h, w, O.build_layers(arch)[-1].cout, flat=arch["layers"][0][0] == "fc")
    return out


def test_replica_sum_equals_one_big_batch():
    # Chainer addgrads with a halved rate (Qiita Sec. 6): R shards at eta with summed
    # per-shard mean gradients == one R*N batch (mean loss) at eta*R
    arch = SMALL_MLP
    layers = O.build_layers(arch)
    w = _init(arch)
    R, n = 4, 5
    shards = _batches(arch, R, n)
    g_sum = sum(O.gradient(layers, w, x, y)[1] for x, y in shards)
    xb = np.concatenate([x for x, _ in shards])
    yb = np.concatenate([y for _, y in shards])
    g_big = O.gradient(layers, w, xb, yb)[1]
    eta = 0.01
    np.testing.assert_allclose(w - eta * g_sum, w - eta * R * g_big, rtol=0, atol=1e-12)


def test_zero_delays_equal_plain_sgd():
    arch = SMALL_CNN
    w0 = _init(arch)
    b = _batches(arch, 6, 3)
    l1, w1, _ = O.train(arch, w0, b, 3, replicas=2, schedule=np.zeros((3, 2), np.int32))
    l2, w2, _ = O.train(arch, w0, b, 3, replicas=2, schedule=None)
    assert l1 == l2 and (w1 == w2).all()
    l3, w3, _ = O.train(arch, w0, b, 3, replicas=2, stage_delays=[0, 0], stage_of_layer=[0, 0, 1, 1, 1])
    assert l3 == l2 and (w3 == w2).all()


def test_constant_delay_matches_explicit_loop():
    # delay 1 for every replica: W(t+1) = W(t) - eta * sum_r g(W(t-1)), W(-1) := W(0)
    arch = SMALL_MLP
    layers = O.build_layers(arch)
    w0 = _init(arch)
    b = _batches(arch, 8, 4)
    T, R, eta = 4, 2, 0.05
    _, wT, _ = O.train(arch, w0, b, T, replicas=R, schedule=np.ones((T, R), np.int32), eta=eta)
    prev, cur = w0.copy(), w0.copy()
    for t in range(T):
        s = sum(O.gradient(layers, prev, *b[(t * R + r) % len(b)])[1] for r in range(R))
        prev, cur = cur, cur - eta * s
    np.testing.assert_array_equal(wT, cur)


def test_pipeline_stage_delays_use_per_stage_versions():
    # two stages: layers 0-1 at delay 1, layer 2 at delay 0 ([PB] Sec. 4.1)
    arch = SMALL_MLP
    layers = O.build_layers(arch)
    offs, _ = O.param_offsets(layers)
    w0 = _init(arch)
    b = _batches(arch, 5, 3)
    T, eta = 3, 0.05
    _, wT, hist = O.train(arch, w0, b, T, stage_delays=[1, 0], stage_of_layer=[0, 0, 1], eta=eta)
    W = [w0.copy()]
    for t in range(T):
        old, new = W[max(0, t - 1)], W[t]
        mixed = np.concatenate([old[:offs[2][0]], new[offs[2][0]:]])
        W.append(W[t] - eta * O.gradient(layers, mixed, *b[t % len(b)])[1])
    np.testing.assert_array_equal(wT, W[-1])


# ---- Nesterov momentum, weight decay (pipelined-training page, Appendices A/B)

def test_nesterov_constant_gradient_closed_form():
    # v_t = -eta*g*(1 - nu^t)/(1 - nu); W_T = W_0 + sum_t (nu*v_t - eta*g)
    w0, g, eta, nu, T = 0.4, -0.25, 0.02, 0.9, 30
    w, v = np.array([w0]), np.array([0.0])
    for _ in range(T):
        w, v = O.update_nesterov(w, v, [np.array([g])], eta, nu)
    closed = w0 - eta * g * sum(nu * (1 - nu ** t) / (1 - nu) + 1.0 for t in range(1, T + 1))
    assert w[0] == pytest.approx(closed, rel=1e-13)
    assert v[0] == pytest.approx(-eta * g * (1 - nu ** T) / (1 - nu), rel=1e-13)
    # nu = 0 reduces to plain SGD
    w1, _ = O.update_nesterov(np.array([w0]), np.array([3.0]), [np.array([g])], eta, 0.0)
    assert w1[0] == pytest.approx(w0 - eta * g, rel=1e-15)


def test_weight_decay_alone_is_geometric_shrink():
    # zero gradient: S = lambda*W, so SGD gives W_T = W_0 * (1 - eta*lambda)^T
    w0, eta, lam, T = np.array([1.5, -0.75, 0.0]), 0.05, 0.004, 40
    w = w0.copy()
    for _ in range(T):
        w = O.update_sgd(w, [np.zeros(3)], eta, weight_decay=lam)
    np.testing.assert_allclose(w, w0 * (1 - eta * lam) ** T, rtol=1e-13, atol=0)
    # Adagrad, one step from G0: G' = G0 + (lambda*W)^2, W' = W - eta*lambda*W/(sqrt(G') + eps)
    G0, eps = 0.1, 1e-8
    w1, G1 = O.update_adagrad(np.array([2.0]), np.array([G0]), [np.array([0.0])], eta, eps, weight_decay=lam)
    g = lam * 2.0
    assert G1[0] == pytest.approx(G0 + g * g, rel=1e-15)
    assert w1[0] == pytest.approx(2.0 - eta * g / (math.sqrt(G0 + g * g) + eps), rel=1e-15)


def test_weight_decay_is_one_more_pushed_buffer():
    # the decay term enters like an extra GradBuf holding lambda*W, for every rule
    rng = np.random.default_rng(5)
    w, v, b = rng.standard_normal(7), rng.standard_normal(7), [rng.standard_normal(7) for _ in range(3)]
    lam = 0.01
    extra = b + [lam * w]
    np.testing.assert_allclose(O.update_sgd(w, b, 0.1, lam), O.update_sgd(w, extra, 0.1), rtol=0, atol=1e-15)
    for fn in (O.update_momentum, O.update_nesterov):
        a = fn(w, v, b, 0.1, 0.9, lam)
        c = fn(w, v, extra, 0.1, 0.9)
        np.testing.assert_allclose(a[0], c[0], rtol=0, atol=1e-15)
        np.testing.assert_allclose(a[1], c[1], rtol=0, atol=1e-15)


# ---- hybrid pipelined / non-pipelined training and stale-weight metrics (pipelined-training page, Sec. 4)

# VGG-16 stage cut of the pipeline reading: block 1 | block 2 | block 3 | blocks 4-5 + FC
VGG_STAGE_CUT = [0, 0, 1, 1, 2, 2, 2] + [3] * 9


def test_stale_weight_percent_vgg_by_hand():
    layers = O.build_layers(O.ARCHS["vgg_c"])
    # stages 0-2 (delays 3, 2, 1) hold conv1_1 .. conv3_3: 9*Cin*Cout + Cout each
    convs = [(3, 64), (64, 64), (64, 128), (128, 128), (128, 256), (256, 256), (256, 256)]
    stale = sum(9 * ci * co + co for ci, co in convs)
    assert stale == 1735488
    total = O.param_count_eq3(O.ARCHS["vgg_c"])
    assert O.stale_weight_percent(layers, VGG_STAGE_CUT, [3, 2, 1, 0]) == pytest.approx(100.0 * stale / total,
                                                                                         rel=1e-15)
    assert O.stale_weight_percent(layers, VGG_STAGE_CUT, [0, 0, 0, 0]) == 0.0
    assert O.stale_weight_percent(layers, VGG_STAGE_CUT, [1, 1, 1, 1]) == 100.0
    assert O.staleness_degrees([3, 2, 1, 0]) == [3, 2, 1, 0]


def test_hybrid_switch_endpoints_and_prefix():
    arch = SMALL_CNN
    stages, delays = [0, 0, 1, 1, 1], [2, 0]
    w0 = _init(arch)
    b = _batches(arch, 5, 3)
    T = 4
    base = O.train(arch, w0, b, T, stage_delays=delays, stage_of_layer=stages)
    plain = O.train(arch, w0, b, T, stage_delays=[0, 0], stage_of_layer=stages)
    # switching at step 0 is plain SGD; never switching is the pipeline
    h0 = O.train(arch, w0, b, T, stage_delays=delays, stage_of_layer=stages, hybrid_switch=0)
    hT = O.train(arch, w0, b, T, stage_delays=delays, stage_of_layer=stages, hybrid_switch=T)
    assert h0[0] == plain[0] and all((x == y).all() for x, y in zip(h0[2], plain[2]))
    assert hT[0] == base[0] and all((x == y).all() for x, y in zip(hT[2], base[2]))
    # switching at N_p = 2: the first two steps are the pipeline's, and from there every
    # step uses the current weights (a brute-force loop over the same history)
    h2 = O.train(arch, w0, b, T, stage_delays=delays, stage_of_layer=stages, hybrid_switch=2)
    assert h2[0][:2] == base[0][:2] and all((x == y).all() for x, y in zip(h2[2][:3], base[2][:3]))
    layers = O.build_layers(arch)
    hist = list(h2[2][:3])
    for t in range(2, T):
        x, y = b[t % len(b)]
        g = O.gradient(layers, hist[t], x, y)[1]
        hist.append(hist[t] - 0.01 * g)
    np.testing.assert_allclose(h2[2][T], hist[T], rtol=0, atol=1e-13)


# ---- DistBelief n_fetch / n_push

def test_fetch_push_every_step_is_synchronous_sgd():
    arch = SMALL_MLP
    w0 = _init(arch)
    b = _batches(arch, 6, 4)
    a = O.train(arch, w0, b, 5, replicas=3)
    f = O.train_fetch_push(arch, w0, b, 5, replicas=3, n_fetch=1, n_push=1)
    assert a[0] == f[0] and (a[1] == f[1]).all()


@pytest.mark.parametrize("m", [2, 3])
def test_fetch_push_windows_equal_a_bigger_synchronous_step(m):
    # n_fetch = n_push = m: the m steps of a window use one copy of W and push their
    # gradient sum once, i.e. one synchronous step with m*R replicas (same batches)
    arch = SMALL_MLP
    R = 2
    w0 = _init(arch)
    b = _batches(arch, 12, 3)
    f = O.train_fetch_push(arch, w0, b, 2 * m, replicas=R, n_fetch=m, n_push=m, optimizer="momentum")
    s = O.train(arch, w0, b, 2, replicas=m * R, optimizer="momentum")
    np.testing.assert_allclose(f[1], s[1], rtol=0, atol=1e-12)
    assert len(f[2]) == 3


def test_fetch_slower_than_push_uses_stale_local_copies():
    # n_fetch = 2, n_push = 1, one replica: step 2j+1 computes on W before step 2j's update
    arch = SMALL_MLP
    layers = O.build_layers(arch)
    w0 = _init(arch)
    b = _batches(arch, 4, 3)
    f = O.train_fetch_push(arch, w0, b, 4, replicas=1, n_fetch=2, n_push=1)
    w = w0.copy()
    for t in range(4):
        local = w if t % 2 == 0 else local
        g = O.gradient(layers, local, *b[t % len(b)])[1]
        w = w - 0.01 * g
    np.testing.assert_allclose(f[1], w, rtol=0, atol=1e-13)


# ---------------------------------------------------------------- training FLOPs per image

def _flops_by_sgemm_roles(arch):
    """2*m*n*k summed over the SGEMM roles of the SPRINT report's Sec. 3.3 table
    for one image (N = 1): convolution / fc, dedw (+ dedb as the k-sum, not a
    GEMM), dedx (none for the first layer)."""
    total = 0
    for i, L in enumerate(O.build_layers(arch)):
        if L.kind == "conv":
            x2 = L.h * L.w
            roles = [(x2, L.cout, 9 * L.cin),           # convolution
                     (9 * L.cin, L.cout, x2)]           # dedw
            if i > 0:
                roles.append((x2, 9 * L.cin, L.cout))   # dedx conv (col2im of dY . W)
        else:
            roles = [(1, L.cout, L.cin), (L.cin, L.cout, 1)]
            if i > 0:
                roles.append((1, L.cin, L.cout))
        total += sum(2 * m * n * k for m, n, k in roles)
    return total


def test_flops_per_image_pinned():
    # tiny CNN by hand: conv1 32*32*16*27 MACs, conv2 16*16*32*144, fc 2048*10; the first layer has no dX
    assert O.flops_per_image(O.ARCHS["tiny"]) == 2 * (2 * 442368 + 3 * 1179648 + 3 * 20480) == 8970240
    # the per-image figures the workload table states (8.97 MFLOP, 0.662 / 1.879 / 92.65 GFLOP)
    for name, stated in (("tiny", 8.97e6), ("smlps", 0.662e9), ("vgg_c", 1.879e9), ("vgg_i", 92.65e9)):
        f = O.flops_per_image(O.ARCHS[name])
        assert abs(f - stated) <= 1e-3 * stated, (name, f)
        assert f == _flops_by_sgemm_roles(O.ARCHS[name]), name


def test_product_flops_count_equals_oracle():
    """The bench's achieved-FLOP/s denominators (product host code) count what the oracle counts."""
    from stale_weight_sgd_gb300 import model
    for name in ("tiny", "smlps", "vgg_c", "vgg_i"):
        assert model.train_flops_per_image(model.NETWORKS[name]) == O.flops_per_image(O.ARCHS[name]), name
