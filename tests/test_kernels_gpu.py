"""Kernel-by-kernel parity of the CUDA path (through the C ABI) against the FP64 oracle."""
import numpy as np
import pytest

import oracle as O
import synth
from helpers import TOL_FP32, TOL_TF32, TOL_UPDATE, dev, host, rel_inf

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def S():
    from stale_weight_sgd_gb300 import sprint
    sprint.lib()
    return sprint


def _f32(seed, tag, shape, std=1.0):
    return synth.normal(seed, tag, shape, std)


def _status_clean(S):
    assert S.sprint_device_status(reset=True) == 0


# ---------------------------------------------------------------- parameter-server update

@pytest.mark.parametrize("k", [1, 3, 4, 16])
@pytest.mark.parametrize("n", [0, 1, 7, 1000, 65537])
@pytest.mark.parametrize("opt", ["sgd", "momentum", "adagrad"])
def test_update(S, k, n, opt):
    w = _f32(1, f"w{n}", n, 0.01)
    bufs = [_f32(1, f"g{j}/{n}", n, 1e-3) for j in range(k)]
    eta, nu, eps = 0.01, 0.9, 1e-8
    dw = dev(w)
    dout = torch.empty_like(dw)
    dbufs = [dev(b) for b in bufs]
    if opt == "sgd":
        S.sprint_apply_update_sgd(dw, dout, dbufs, n, eta)
        ref = O.update_sgd(w, bufs, eta)
    elif opt == "momentum":
        v = _f32(1, f"v{n}", n, 1e-4)
        dv = dev(v)
        S.sprint_apply_update_momentum(dw, dout, dv, dbufs, n, eta, nu)
        ref, vref = O.update_momentum(w, v, bufs, eta, nu)
        assert rel_inf(host(dv), vref) <= TOL_UPDATE
    else:
        G = np.full(n, 0.1, np.float32)
        dG = dev(G)
        S.sprint_apply_update_adagrad(dw, dout, dG, dbufs, n, eta, eps)
        ref, Gref = O.update_adagrad(w, G, bufs, eta, eps)
        assert rel_inf(host(dG), Gref) <= TOL_UPDATE
    assert rel_inf(host(dout), ref) <= TOL_UPDATE


@pytest.mark.parametrize("rows,cols,tail", [(300, 136, 303), (37, 27, 0), (64, 4096, 64), (129, 260, 1)])
@pytest.mark.parametrize("k", [1, 4, 16])
@pytest.mark.parametrize("opt", ["sgd", "momentum", "adagrad"])
def test_update_transposed(S, rows, cols, tail, k, opt):
    """sprint_apply_update_t over a matrix plus `tail` elements after it (a bias and padding):
    W', state bit for bit the flat update's; W'^T the exact transpose of the matrix part;
    W' against the oracle's update."""
    n = rows * cols + tail
    w = _f32(4, f"w{n}", n, 0.01)
    bufs = [_f32(4, f"g{j}/{n}", n, 1e-3) for j in range(k)]
    st0 = np.abs(_f32(4, f"s{n}", n, 1e-2)) + (0.1 if opt == "adagrad" else 0.0)
    eta, hp = 0.01, (1e-8 if opt == "adagrad" else 0.9)
    dbufs = [dev(b) for b in bufs]
    dw = dev(w)
    out_t, out_f = torch.empty_like(dw), torch.empty_like(dw)
    wT = torch.empty(rows * cols, dtype=torch.float32, device="cuda")
    st_t, st_f = (dev(st0), dev(st0)) if opt != "sgd" else (None, None)
    S.sprint_apply_update_t(opt, dw, out_t, wT, st_t, dbufs, rows, cols, eta, hp, n_total=n)
    if opt == "sgd":
        S.sprint_apply_update_sgd(dw, out_f, dbufs, n, eta)
        ref = O.update_sgd(w, bufs, eta)
    elif opt == "momentum":
        S.sprint_apply_update_momentum(dw, out_f, st_f, dbufs, n, eta, hp)
        ref, _ = O.update_momentum(w, st0, bufs, eta, hp)
    else:
        S.sprint_apply_update_adagrad(dw, out_f, st_f, dbufs, n, eta, hp)
        ref, _ = O.update_adagrad(w, st0, bufs, eta, hp)
    a = host(out_t)
    assert np.array_equal(a, host(out_f))
    assert np.array_equal(host(wT).reshape(cols, rows), a[:rows * cols].reshape(rows, cols).T)
    if opt != "sgd":
        assert np.array_equal(host(st_t), host(st_f))
    assert rel_inf(a, ref) <= TOL_UPDATE


@pytest.mark.parametrize("opt", ["sgd", "momentum", "nesterov", "adagrad"])
@pytest.mark.parametrize("wd", [0.0, 0.004])
@pytest.mark.parametrize("k", [1, 3])
def test_update_rules_with_weight_decay(S, opt, wd, k):
    """sprint_apply_update by rule, with weight decay, against the oracle; with
    weight decay 0 bit for bit the rule-specific entry points."""
    n = 10007
    w = _f32(6, "w", n, 0.05)
    bufs = [_f32(6, f"g{j}", n, 1e-3) for j in range(k)]
    st0 = np.abs(_f32(6, "s", n, 1e-2)) + (0.1 if opt == "adagrad" else 0.0)
    eta, hp = 0.01, (1e-8 if opt == "adagrad" else 0.9)
    dbufs = [dev(b) for b in bufs]
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    st = dev(st0) if opt != "sgd" else None
    S.sprint_apply_update(opt, dev(w), out, st, dbufs, n, eta, hp, wd)
    ref, st_ref = O.apply_update(w, bufs, opt, eta, nu=hp, eps=hp, state=st0.astype(np.float64), weight_decay=wd)
    assert rel_inf(host(out), ref) <= TOL_UPDATE
    if opt != "sgd":
        assert rel_inf(host(st), st_ref) <= TOL_UPDATE
    if wd == 0.0 and opt != "nesterov":
        out2 = torch.empty_like(out)
        st2 = dev(st0) if opt != "sgd" else None
        if opt == "sgd":
            S.sprint_apply_update_sgd(dev(w), out2, dbufs, n, eta)
        elif opt == "momentum":
            S.sprint_apply_update_momentum(dev(w), out2, st2, dbufs, n, eta, hp)
        else:
            S.sprint_apply_update_adagrad(dev(w), out2, st2, dbufs, n, eta, hp)
        assert np.array_equal(host(out), host(out2))
    # the transposing form over a matrix (plus a bias tail): bit for bit the flat one
    rows, cols = 97, 100
    out_t = torch.empty(n, dtype=torch.float32, device="cuda")
    wT = torch.empty(rows * cols, dtype=torch.float32, device="cuda")
    st_t = dev(st0) if opt != "sgd" else None
    S.sprint_apply_update_t(opt, dev(w), out_t, wT, st_t, dbufs, rows, cols, eta, hp, n_total=n, weight_decay=wd)
    assert np.array_equal(host(out_t), host(out))
    assert np.array_equal(host(wT).reshape(cols, rows), host(out)[:rows * cols].reshape(rows, cols).T)
    if opt != "sgd":
        assert np.array_equal(host(st_t), host(st))


def test_update_in_place_and_order_invariance_exact(S):
    n, k = 4099, 8
    w = synth.dyadic(2, "w", n)
    bufs = [synth.dyadic(2, f"g{j}", n) for j in range(k)]
    dw = dev(w)
    S.sprint_apply_update_sgd(dw, dw, [dev(b) for b in bufs], n, 2.0 ** -3)
    perm = synth.rng(2, "perm").permutation(k)
    dw2 = dev(w)
    S.sprint_apply_update_sgd(dw2, dw2, [dev(bufs[i]) for i in perm], n, 2.0 ** -3)
    a, b = host(dw), host(dw2)
    assert (a == b).all()
    assert (a.astype(np.float64) == O.update_sgd(w, bufs, 2.0 ** -3)).all()


@pytest.mark.parametrize("first", [0, 1])
def test_gradbuf_accumulate(S, first):
    n = 10003
    buf = _f32(3, "buf", n)
    g = _f32(3, "g", n)
    d = dev(buf)
    S.sprint_gradbuf_accumulate(d, dev(g), n, -0.01, first)
    assert rel_inf(host(d), O.gradbuf_accumulate(buf, g, -0.01, bool(first))) <= TOL_UPDATE


# ---------------------------------------------------------------- pool / softmax / im2col

@pytest.mark.parametrize("shape", [(2, 8, 6, 8), (3, 7, 5, 3), (1, 4, 4, 16), (2, 2, 2, 5)])
def test_pool_fwd_bwd_bit_exact(S, shape):
    N, H, W, C = shape
    x = _f32(4, f"x{shape}", shape)
    x[0, 0:2, 0:2, 0] = 0.0       # tie: all-zero window
    x = np.maximum(x, 0.0)        # pool sees ReLU outputs: many exact zero ties
    y_ref, a_ref = O.maxpool2x2_fwd(x)
    dx_ = dev(x)
    y = torch.empty((N, H // 2, W // 2, C), dtype=torch.float32, device="cuda")
    a = torch.empty(y.shape, dtype=torch.uint8, device="cuda")
    S.sprint_pool_fwd(dx_, y, a, N, H, W, C)
    assert (host(a) == a_ref).all()
    assert (host(y) == y_ref.astype(np.float32)).all()
    dy = _f32(4, f"dy{shape}", y.shape)
    out = torch.full((N, H, W, C), 7.0, dtype=torch.float32, device="cuda")
    S.sprint_pool_bwd(dev(dy), a, y, out, N, H, W, C)
    ref = O.maxpool2x2_bwd(dy * (y_ref > 0), a_ref, H, W)
    assert (host(out) == ref.astype(np.float32)).all()


@pytest.mark.parametrize("N,C", [(8, 10), (512, 10), (64, 1000), (33, 7), (1500, 10), (20, 32), (20, 33)])
def test_softmax_xent(S, N, C):
    z = _f32(5, f"z{N}", (N, C), 3.0)
    y = synth.labels(5, f"y{N}", N, C)
    loss_ref, dz_ref = O.softmax_xent(z, y)
    dz = torch.empty((N, C), dtype=torch.float32, device="cuda")
    loss = torch.zeros(4, dtype=torch.float32, device="cuda")
    S.sprint_softmax_xent(dev(z), dev(y), N, C, loss, dz)
    assert abs(host(loss)[0] - loss_ref) <= 1e-6 * abs(loss_ref)
    assert rel_inf(host(dz), dz_ref) <= TOL_FP32


def test_softmax_uniform_is_ln_c(S):
    z = np.full((16, 1000), 2.5, np.float32)
    loss = torch.zeros(4, dtype=torch.float32, device="cuda")
    dz = torch.empty((16, 1000), dtype=torch.float32, device="cuda")
    S.sprint_softmax_xent(dev(z), dev(np.arange(16, dtype=np.int32)), 16, 1000, loss, dz)
    assert abs(host(loss)[0] - np.log(1000.0)) < 1e-5


@pytest.mark.parametrize("shape,pad", [((2, 5, 4, 3), 1), ((1, 6, 6, 8), 1), ((2, 4, 5, 4), 0)])
def test_im2col_bit_exact(S, shape, pad):
    N, H, W, C = shape
    x = _f32(6, f"x{shape}", shape)
    col_ref, src_ref = O.im2col(x, pad)
    rows = N * (H + 2 * pad - 2) * (W + 2 * pad - 2)
    col = torch.empty((rows, 9 * C), dtype=torch.float32, device="cuda")
    src = torch.empty((rows, 9 * C), dtype=torch.int32, device="cuda")
    S.sprint_im2col(dev(x), N, H, W, C, pad, col, src)
    assert (host(src) == src_ref).all()
    assert (host(col) == col_ref).all()


# ---------------------------------------------------------------- FC (tcgen05 TF32 and CUDA-core paths)

FC_CASES = [
    (300, 200, 136),    # tensor cores: ragged M, N and K tiles
    (512, 320, 384),    # several full tiles, N-tile 128/256
    (64, 256, 512),     # M below one tile
    (37, 50, 10),       # CUDA-core path (widths not multiples of 4)
    (512, 5000, 10),    # classifier of SMLPs
    (64, 48, 10),       # 10 outputs: tensor-core dW with a partial M tile, short-reduction dX
    (16, 40, 33),       # 33 outputs: tensor-core dW, CUDA-core dX
    (41, 64, 3),        # 3 outputs: float4 skinny forward (4-wide accumulators), ragged row block
    (24, 96, 13),       # 13 outputs: float4 skinny forward (16-wide accumulators)
    (20, 64, 30),       # 30 outputs: short-reduction dX with 32 registers of dy, CUDA-core forward
]


@pytest.mark.parametrize("N,fin,fout", FC_CASES)
@pytest.mark.parametrize("relu", [0, 1])
def test_fc_fwd(S, N, fin, fout, relu):
    x = _f32(7, f"x{N}{fin}", (N, fin))
    w = _f32(7, f"w{fin}{fout}", (fout, fin), np.sqrt(2.0 / fin))
    b = _f32(7, f"b{fout}", fout, 0.1)
    ref = O.fc_fwd(x, w, b)
    if relu:
        ref = O.relu(ref)
    y = torch.empty((N, fout), dtype=torch.float32, device="cuda")
    S.sprint_fc_fwd(dev(x), dev(w), dev(b), y, N, fin, fout, relu)
    assert rel_inf(host(y), ref) <= TOL_TF32
    _status_clean(S)


@pytest.mark.parametrize("N,fin,fout", FC_CASES)
@pytest.mark.parametrize("accumulate", [0, 1])
@pytest.mark.parametrize("with_wT", [0, 1])
def test_fc_bwd(S, N, fin, fout, accumulate, with_wT):
    x = np.maximum(_f32(8, f"x{N}{fin}", (N, fin)), 0)   # a ReLU output: mask source
    w = _f32(8, f"w{fin}{fout}", (fout, fin), np.sqrt(2.0 / fin))
    dy = _f32(8, f"dy{N}{fout}", (N, fout))
    dw0 = _f32(8, "dw0", (fout, fin))
    db0 = _f32(8, "db0", fout)
    dx_ref, dw_ref, db_ref = O.fc_bwd(x, w, dy)
    dx_ref = dx_ref * O.relu_mask(x)
    alpha = 0.5
    dw_ref = O.gradbuf_accumulate(dw0, dw_ref, alpha, not accumulate)
    db_ref = O.gradbuf_accumulate(db0, db_ref, alpha, not accumulate)
    dx = torch.empty((N, fin), dtype=torch.float32, device="cuda")
    dw = dev(dw0)
    db = dev(db0)
    xd = dev(x)
    wT = dev(np.ascontiguousarray(w.T)) if with_wT else None
    nb = S.sprint_fc_workspace_size(N, fin, fout, with_wT)
    ws = torch.empty(nb // 4 + 64, dtype=torch.float32, device="cuda")
    S.sprint_fc_bwd(xd, dev(w), wT, dev(dy), xd, dx, dw, db, alpha, accumulate, N, fin, fout, ws, nb)
    assert rel_inf(host(dx), dx_ref) <= TOL_TF32
    assert rel_inf(host(dw), dw_ref) <= TOL_TF32
    assert rel_inf(host(db), db_ref) <= TOL_FP32
    _status_clean(S)


# ---------------------------------------------------------------- FC batched over replicas (grouped launches)

FC_BATCHED_CASES = [
    (3, 300, 200, 136),    # grouped tensor-core launch, ragged tiles
    (2, 512, 320, 384),    # grouped pair tiles
    (17, 64, 96, 64),      # more problems than one launch takes
    (3, 37, 50, 10),       # CUDA-core paths, looped per problem
    (2, 64, 48, 10),       # grouped tensor-core dW, short-reduction dX
    (5, 42, 128, 7),       # grouped float4 skinny forward (8-wide accumulators), ragged row block
    (4, 96, 512, 10),      # narrow output, long k: grouped tensor cores + k-split last round (with workspace)
    (3, 64, 300, 13),      # the same with a ragged k tile and 13 outputs
]


def _fc_problem(seed, g, N, fin, fout):
    x = np.maximum(_f32(seed, f"bx{g}", (N, fin)), 0)
    w = _f32(seed, f"bw{g}", (fout, fin), np.sqrt(2.0 / fin))
    b = _f32(seed, f"bb{g}", fout, 0.1)
    dy = _f32(seed, f"bdy{g}", (N, fout))
    return x, w, b, dy


@pytest.mark.parametrize("G,N,fin,fout", FC_BATCHED_CASES + [(4, 512, 3072, 5000)])
@pytest.mark.parametrize("relu", [0, 1])
@pytest.mark.parametrize("tail", [0, 1])
def test_fc_fwd_batched(S, G, N, fin, fout, relu, tail):
    probs = [_fc_problem(11, g, N, fin, fout) for g in range(G)]
    xs = [dev(p[0]) for p in probs]
    ws = [dev(p[1]) for p in probs]
    bs = [dev(p[2]) if g % 3 != 1 else None for g, p in enumerate(probs)]   # some problems without bias
    ys = [torch.empty((N, fout), dtype=torch.float32, device="cuda") for _ in range(G)]
    # with the workspace the last round's tiles may be split along k (partials added afterwards)
    nb = S.sprint_fc_fwd_batched_workspace_size() if tail else 0
    wsb = torch.empty(nb // 4 + 64, dtype=torch.float32, device="cuda") if tail else None
    S.sprint_fc_fwd_batched(xs, ws, bs, ys, N, fin, fout, relu, wsb, nb)
    for g, (x, w, b, _) in enumerate(probs):
        ref = O.fc_fwd(x, w, b if g % 3 != 1 else np.zeros_like(b))
        if relu:
            ref = O.relu(ref)
        assert rel_inf(host(ys[g]), ref) <= TOL_TF32, g
    _status_clean(S)


@pytest.mark.parametrize("G,N,fin,fout", FC_BATCHED_CASES)
@pytest.mark.parametrize("with_wT,with_dx", [(0, 1), (1, 1), (1, 0)])
@pytest.mark.parametrize("accumulate,tail", [(0, 1), (1, 1), (1, 0)])
def test_fc_bwd_batched(S, G, N, fin, fout, with_wT, with_dx, accumulate, tail):
    probs = [_fc_problem(12, g, N, fin, fout) for g in range(G)]
    alpha = 0.5
    xs = [dev(p[0]) for p in probs]
    ws = [dev(p[1]) for p in probs]
    wTs = [dev(np.ascontiguousarray(p[1].T)) for p in probs] if with_wT else None
    dys = [dev(p[3]) for p in probs]
    masks = [xs[g] if g % 2 == 0 else None for g in range(G)]      # odd problems: no ReLU mask
    dxs = [torch.empty((N, fin), dtype=torch.float32, device="cuda") for _ in range(G)] if with_dx else None
    dw0 = [_f32(12, f"dw0{g}", (fout, fin)) for g in range(G)]
    db0 = [_f32(12, f"db0{g}", fout) for g in range(G)]
    dws = [dev(a) for a in dw0]
    dbs = [dev(a) for a in db0]
    nb = S.sprint_fc_batched_workspace_size(G, N, fin, fout, with_wT or not with_dx)
    if not tail:   # only the per-problem slices: no k split of the last round
        nb -= S.sprint_fc_fwd_batched_workspace_size()
    wsb = torch.empty(nb // 4 + 64, dtype=torch.float32, device="cuda")
    S.sprint_fc_bwd_batched(xs, ws, wTs, dys, masks, dxs, dws, dbs, alpha, accumulate, N, fin, fout, wsb, nb)
    for g, (x, w, _, dy) in enumerate(probs):
        dx_ref, dw_ref, db_ref = O.fc_bwd(x, w, dy)
        if g % 2 == 0:
            dx_ref = dx_ref * O.relu_mask(x)
        dw_ref = O.gradbuf_accumulate(dw0[g], dw_ref, alpha, not accumulate)
        db_ref = O.gradbuf_accumulate(db0[g], db_ref, alpha, not accumulate)
        if with_dx:
            assert rel_inf(host(dxs[g]), dx_ref) <= TOL_TF32, g
        assert rel_inf(host(dws[g]), dw_ref) <= TOL_TF32, g
        assert rel_inf(host(dbs[g]), db_ref) <= TOL_FP32, g
    _status_clean(S)


@pytest.mark.parametrize("G,N,fin,fout", FC_BATCHED_CASES + [(4, 512, 3072, 5000)])
@pytest.mark.parametrize("tail", [0, 1])
def test_fc_fwd_batched_transposed_copy(S, G, N, fin, fout, tail):
    """yT: the same outputs as the plain call, bit for bit, and their exact transpose."""
    probs = [_fc_problem(14, g, N, fin, fout) for g in range(G)]
    xs = [dev(p[0]) for p in probs]
    ws = [dev(p[1]) for p in probs]
    bs = [dev(p[2]) for p in probs]
    nb = S.sprint_fc_fwd_batched_workspace_size() if tail else 0
    wsb = torch.empty(nb // 4 + 64, dtype=torch.float32, device="cuda") if tail else None
    ys = [torch.empty((N, fout), dtype=torch.float32, device="cuda") for _ in range(G)]
    ys2 = [torch.empty((N, fout), dtype=torch.float32, device="cuda") for _ in range(G)]
    yTs = [torch.full((fout + 1, N), 7.0, dtype=torch.float32, device="cuda") for _ in range(G)]
    S.sprint_fc_fwd_batched(xs, ws, bs, ys, N, fin, fout, 1, wsb, nb)
    S.sprint_fc_fwd_batched(xs, ws, bs, ys2, N, fin, fout, 1, wsb, nb, yT=yTs)
    for g, (x, w, b, _) in enumerate(probs):
        y, y2, yT = host(ys[g]), host(ys2[g]), host(yTs[g])
        assert np.array_equal(y, y2), g
        assert np.array_equal(yT[:fout], y.T), g
        assert np.all(yT[fout] == 7.0), g          # the row past the output is not written
        assert rel_inf(y, O.relu(O.fc_fwd(x, w, b))) <= TOL_TF32, g
    _status_clean(S)


@pytest.mark.parametrize("G,N,fin,fout", FC_BATCHED_CASES + [(4, 512, 5000, 5000)])
@pytest.mark.parametrize("accumulate,tail", [(0, 1), (1, 1), (1, 0)])
def test_fc_bwd_batched_transposed_operands(S, G, N, fin, fout, accumulate, tail):
    """xT1 / dyT / dxT: x^T with a row of ones (dedb inside the dedw GEMM), dy^T read
    as given, dx^T written next to dx; results as the oracle's, dxT the exact transpose."""
    probs = [_fc_problem(15, g, N, fin, fout) for g in range(G)]
    alpha = 0.5
    xs = [dev(p[0]) for p in probs]
    xT1 = [dev(np.concatenate([p[0].T, np.ones((1, N), np.float32)])) for p in probs]
    ws = [dev(p[1]) for p in probs]
    wTs = [dev(np.ascontiguousarray(p[1].T)) for p in probs]
    dys = [dev(p[3]) for p in probs]
    dyT = [dev(np.ascontiguousarray(p[3].T)) for p in probs]
    masks = [xs[g] if g % 2 == 0 else None for g in range(G)]
    dxs = [torch.empty((N, fin), dtype=torch.float32, device="cuda") for _ in range(G)]
    dxT = [torch.empty((fin, N), dtype=torch.float32, device="cuda") for _ in range(G)]
    dw0 = [_f32(15, f"dw0{g}", (fout, fin)) for g in range(G)]
    db0 = [_f32(15, f"db0{g}", fout) for g in range(G)]
    dws = [dev(a) for a in dw0]
    dbs = [dev(a) for a in db0]
    nb = S.sprint_fc_batched_workspace_size(G, N, fin, fout, 1)
    if not tail:
        nb -= S.sprint_fc_fwd_batched_workspace_size()
    wsb = torch.empty(nb // 4 + 64, dtype=torch.float32, device="cuda")
    S.sprint_fc_bwd_batched(xs, ws, wTs, dys, masks, dxs, dws, dbs, alpha, accumulate, N, fin, fout, wsb, nb,
                            xT1=xT1, dyT=dyT, dxT=dxT)
    for g, (x, w, _, dy) in enumerate(probs):
        dx_ref, dw_ref, db_ref = O.fc_bwd(x, w, dy)
        if g % 2 == 0:
            dx_ref = dx_ref * O.relu_mask(x)
        dw_ref = O.gradbuf_accumulate(dw0[g], dw_ref, alpha, not accumulate)
        db_ref = O.gradbuf_accumulate(db0[g], db_ref, alpha, not accumulate)
        dx = host(dxs[g])
        assert rel_inf(dx, dx_ref) <= TOL_TF32, g
        assert np.array_equal(host(dxT[g]), dx.T), g
        assert rel_inf(host(dws[g]), dw_ref) <= TOL_TF32, g
        # db: a column of the TF32 dedw GEMM when that runs on the tensor cores
        assert rel_inf(host(dbs[g]), db_ref) <= TOL_TF32, g
    _status_clean(S)


@pytest.mark.parametrize("G,N,fin,fout", [c for c in FC_BATCHED_CASES if c[0] <= 16] + [(4, 512, 1000, 768), (1, 64, 256, 128)])
@pytest.mark.parametrize("opt", ["sgd", "momentum", "adagrad"])
@pytest.mark.parametrize("with_xT1", [0, 1])
def test_fc_bwd_update_batched(S, G, N, fin, fout, opt, with_xT1):
    """Backward + the parameter-server apply of the layer over the G GradBufs: GradBufs as
    the oracle's; W', b' and the optimizer state bit for bit what the standalone update
    computes from those GradBufs; W'^T the exact transpose of W'."""
    probs = [_fc_problem(16, g, N, fin, fout) for g in range(G)]
    xs = [dev(p[0]) for p in probs]
    ws = [dev(p[1]) for p in probs]
    wTs = [dev(np.ascontiguousarray(p[1].T)) for p in probs]
    dys = [dev(p[3]) for p in probs]
    xT1 = [dev(np.concatenate([p[0].T, np.ones((1, N), np.float32)])) for p in probs] if with_xT1 else None
    dxs = [torch.empty((N, fin), dtype=torch.float32, device="cuda") for _ in range(G)]
    dws = [torch.empty((fout, fin), dtype=torch.float32, device="cuda") for _ in range(G)]
    dbs = [torch.empty(fout, dtype=torch.float32, device="cuda") for _ in range(G)]
    w_in = dev(_f32(16, "win", (fout, fin), 0.05))
    b_in = dev(_f32(16, "bin", fout, 0.05))
    if opt == "adagrad":
        st0 = np.abs(_f32(16, "st", fout * fin + fout)) + 0.1
    else:
        st0 = _f32(16, "st", fout * fin + fout, 0.01)
    w_st, b_st = dev(st0[:fout * fin].reshape(fout, fin)), dev(st0[fout * fin:])
    w_out = torch.full((fout, fin), 5.0, dtype=torch.float32, device="cuda")
    b_out = torch.full((fout,), 5.0, dtype=torch.float32, device="cuda")
    wT_out = torch.empty((fin, fout), dtype=torch.float32, device="cuda")
    eta, hp = 0.05, (1e-6 if opt == "adagrad" else 0.9)
    nb = S.sprint_fc_batched_workspace_size(G, N, fin, fout, 1)
    wsb = torch.empty(nb // 4 + 64, dtype=torch.float32, device="cuda")
    S.sprint_fc_bwd_update_batched(xs, ws, wTs, dys, None, dxs, dws, dbs, 1.0, 0, N, fin, fout, opt, w_in, b_in, w_out,
                                   b_out, wT_out, w_st if opt != "sgd" else None, b_st if opt != "sgd" else None, eta,
                                   hp, wsb, nb, xT1=xT1)
    for g, (x, w, _, dy) in enumerate(probs):
        dx_ref, dw_ref, db_ref = O.fc_bwd(x, w, dy)
        assert rel_inf(host(dxs[g]), dx_ref) <= TOL_TF32, g
        assert rel_inf(host(dws[g]), dw_ref) <= TOL_TF32, g
        assert rel_inf(host(dbs[g]), db_ref) <= TOL_TF32, g
    # the standalone update on the GradBufs just written, from the same starting state
    w_ref = torch.empty_like(w_out)
    b_ref = torch.empty_like(b_out)
    w_st2, b_st2 = dev(st0[:fout * fin].reshape(fout, fin)), dev(st0[fout * fin:])
    if opt == "sgd":
        S.sprint_apply_update_sgd(w_in, w_ref, dws, fout * fin, eta)
        S.sprint_apply_update_sgd(b_in, b_ref, dbs, fout, eta)
    elif opt == "momentum":
        S.sprint_apply_update_momentum(w_in, w_ref, w_st2, dws, fout * fin, eta, hp)
        S.sprint_apply_update_momentum(b_in, b_ref, b_st2, dbs, fout, eta, hp)
    else:
        S.sprint_apply_update_adagrad(w_in, w_ref, w_st2, dws, fout * fin, eta, hp)
        S.sprint_apply_update_adagrad(b_in, b_ref, b_st2, dbs, fout, eta, hp)
    assert np.array_equal(host(w_out), host(w_ref))
    assert np.array_equal(host(b_out), host(b_ref))
    assert np.array_equal(host(wT_out), host(w_out).T)
    if opt != "sgd":
        assert np.array_equal(host(w_st), host(w_st2))
        assert np.array_equal(host(b_st), host(b_st2))
    _status_clean(S)


@pytest.mark.parametrize("G,N,C", [(4, 512, 10), (3, 64, 1000), (17, 33, 7)])
def test_softmax_xent_batched(S, G, N, C):
    zs = [_f32(13, f"z{g}", (N, C), 3.0) for g in range(G)]
    ys = [synth.labels(13, f"y{g}", N, C) for g in range(G)]
    loss = torch.zeros((G, 4), dtype=torch.float32, device="cuda")
    dz = [torch.empty((N, C), dtype=torch.float32, device="cuda") for _ in range(G)]
    S.sprint_softmax_xent_batched([dev(z) for z in zs], [dev(y) for y in ys], [loss[g] for g in range(G)], dz, N, C)
    lh = host(loss)
    for g in range(G):
        loss_ref, dz_ref = O.softmax_xent(zs[g], ys[g])
        assert abs(lh[g, 0] - loss_ref) <= 1e-6 * abs(loss_ref), g
        assert rel_inf(host(dz[g]), dz_ref) <= TOL_FP32, g


# ---------------------------------------------------------------- convolution

CONV_CASES = [
    (2, 8, 8, 32, 64),      # tensor cores, one pixel tile per image pair
    (3, 10, 6, 64, 32),     # ragged pixel tiles (boxes overhang the image)
    (2, 16, 16, 32, 128),   # several pixel tiles, N-tile 128
    (2, 4, 4, 64, 256),     # small spatial, wide channels
    (2, 6, 5, 3, 16),       # RGB input layer: CUDA-core path
    (1, 8, 8, 16, 32),      # Cin not a multiple of 32: CUDA-core path
    (8, 16, 16, 16, 32),    # batch % 4 == 0: tensor-core weight gradient (the tiny CNN's conv2)
    (4, 8, 8, 32, 64),      # tensor-core weight gradient, W*N = 32 per row
    (12, 7, 5, 64, 32),     # ragged rows (W*N = 60), Cout < 128
    (32, 4, 4, 128, 256),   # wide channels, split-K
    (4, 12, 12, 3, 64),     # RGB layer 3 -> 64: im2col rows in shared memory (tensor cores), tensor-core dW
    (3, 7, 9, 3, 64),       # the same with a ragged last pixel tile (189 pixels)
    (2, 37, 35, 3, 64),     # the same across image rows and images (2590 pixels)
    (8, 9, 7, 3, 16),       # RGB layer, ragged spatial size
    (3, 7, 6, 1, 16),       # one input channel: direct CUDA-core forward, zero-filled tap boxes in dW
    (4, 8, 5, 4, 32),       # four input channels: direct forward (4-wide patch), CUDA-core dX
    (2, 37, 35, 3, 48),     # RGB dW: ragged 16-pixel row segments, two channels per lane with idle lanes
    (3, 20, 40, 2, 64),     # RGB dW: two input channels, full warp of channel pairs
    (2, 11, 9, 4, 64),      # RGB dW: the widest patch (4 channels) with channel pairs
    (1, 6, 17, 1, 40),      # RGB dW: one input channel, Cout between 32 and 64
    (2, 7, 9, 3, 18),       # RGB dW with Cout % 4 != 0 (4-byte dy copies); CUDA-core forward and dX
    # batch % 32 == 0: the weight gradient's blocked [H][W*N/32][C][32] copies
    (32, 6, 5, 64, 64),     # Cin = Cout = 64: factored over kernel rows x columns on a CTA pair, w-shift one block
    (64, 9, 20, 64, 64),    # factored, w-shift = two blocks, several k-tiles per split
    (64, 3, 3, 32, 48),     # w-shift = two blocks, Cout % 32 != 0
    (32, 5, 7, 256, 128),   # one tap per tile, split-K
    (32, 4, 6, 6, 32),      # Cin < 8: tap boxes of 8 channel rows, rows past Cin zero-filled
    (32, 3, 4, 128, 256),   # CTA pairs over Cout, packed taps of 128 rows
    # 64 output channels on rows of >= 96 pixels: forward / input gradient factored over the kernel columns
    (2, 4, 100, 64, 64),    # forward and input gradient factored; one 126-pixel tile per row
    (2, 5, 130, 32, 64),    # forward factored, two tiles per row (the second holds 4 pixels)
    (1, 3, 253, 64, 96),    # input gradient factored (k = 3 x 96), three tiles per row, odd tile count
    # 64 or 128 output channels: halo-staged tiles of whole output rows
    (2, 6, 112, 64, 128),   # forward BN 128, input gradient BN 64; one 112-pixel row per tile
    (2, 8, 56, 128, 64),    # two rows of 56 pixels per tile, four input chunks (forward)
    (2, 8, 56, 128, 256),   # input gradient with 128 outputs and 8 chunks: flipped, four 56-pixel rows per tile
    (1, 2, 452, 32, 128),   # rows too wide to flip: forward on pair tiles of 113 pixels, N = 128
    (1, 4, 224, 64, 64),    # two tiles per row (the VGG conv1_2 width)
    (1, 6, 56, 64, 64),     # odd tile count: the last pair's second CTA has no tile
    (2, 15, 28, 64, 128),   # four rows per tile, the last tile row holds three
    (1, 3, 221, 64, 64),    # two tiles per row, the second one pixel short
]



def _conv_inputs(seed, N, H, W, Cin, Cout):
    x = np.maximum(_f32(seed, f"x{N}{H}{W}{Cin}", (N, H, W, Cin)), 0)
    w = _f32(seed, f"w{Cin}{Cout}", (Cout, 3, 3, Cin), np.sqrt(2.0 / (9 * Cin)))
    b = _f32(seed, f"b{Cout}", Cout, 0.1)
    return x, w, b


def _ws(S, op, *shape):
    n = S.sprint_conv_workspace_size(op, *shape, 1)
    return (torch.empty(max(n // 4, 1) + 64, dtype=torch.float32, device="cuda"), n)


def test_conv_plans_of_the_cases(S):
    """The small cases reach every forward / input-gradient tiling of the 64- and 128-channel
    outputs (whole-tensor parity below covers every tile edge): halo-staged pairs factored to
    192 columns (one-row tiles with TMA epilogue boxes, and multi-row tiles), the flipped
    128-channel tiles (forward and input gradient), pair tiles of N = 128, and the factored
    tap windows."""
    seen = set()
    for case in CONV_CASES:
        N, H, W, Cin, Cout = case
        for op in (S.SPRINT_CONV_FWD, S.SPRINT_CONV_DX):
            pl = S.sprint_conv_plan(op, N, H, W, Cin, Cout, 1, True)
            nout = Cout if op == S.SPRINT_CONV_FWD else Cin
            if pl["conv_halo"]:
                assert nout in (64, 128) and pl["path"] == "tc", (case, op, pl)
                if nout == 64:
                    assert pl["pair"] == 1 and pl["bn"] == 192 and not pl["conv_hflip"]
                    seen.add(("fact192", pl["box_h"] == 1))
                elif pl["conv_hflip"]:
                    assert pl["pair"] == 0 and pl["bn"] == 128 and (pl["box_w"] + 2) * pl["box_h"] <= 256
                    seen.add(("flip", op))
                else:
                    assert pl["pair"] == 1 and pl["bn"] == 128 and op == S.SPRINT_CONV_FWD
                    seen.add(("pair128", op))
            if pl["conv_fact"]:
                seen.add(("fact", op))
    want = {("fact192", True), ("fact192", False), ("flip", S.SPRINT_CONV_FWD), ("flip", S.SPRINT_CONV_DX),
            ("pair128", S.SPRINT_CONV_FWD), ("fact", S.SPRINT_CONV_FWD), ("fact", S.SPRINT_CONV_DX)}
    assert want <= seen, want - seen


@pytest.mark.parametrize("N,H,W,Cin,Cout", CONV_CASES)
def test_conv_fwd(S, N, H, W, Cin, Cout):
    x, w, b = _conv_inputs(9, N, H, W, Cin, Cout)
    ref = O.relu(O.conv3x3_fwd(x, w, b))
    y = torch.empty((N, H, W, Cout), dtype=torch.float32, device="cuda")
    ws, nb = _ws(S, S.SPRINT_CONV_FWD, N, H, W, Cin, Cout)
    S.sprint_conv_fwd(dev(x), dev(w), dev(b), y, N, H, W, Cin, Cout, 1, 1, ws, nb)
    assert rel_inf(host(y), ref) <= TOL_TF32
    _status_clean(S)


@pytest.mark.parametrize("N,H,W,Cin,Cout", CONV_CASES)
def test_conv_dx(S, N, H, W, Cin, Cout):
    x, w, _ = _conv_inputs(10, N, H, W, Cin, Cout)
    dy = _f32(10, "dy", (N, H, W, Cout))
    ref = O.conv3x3_dx(dy, w, H, W) * O.relu_mask(x)
    dx = torch.full((N, H, W, Cin), 3.0, dtype=torch.float32, device="cuda")
    ws, nb = _ws(S, S.SPRINT_CONV_DX, N, H, W, Cin, Cout)
    xd = dev(x)
    S.sprint_conv_dX(dev(dy), dev(w), None, xd, dx, N, H, W, Cin, Cout, 1, ws, nb)
    assert rel_inf(host(dx), ref) <= TOL_TF32
    # with a caller-provided w^T ([3][3][Cin][Cout])
    wT = np.ascontiguousarray(w.reshape(Cout, 9 * Cin).T)
    dx.fill_(5.0)
    S.sprint_conv_dX(dev(dy), dev(w), dev(wT), xd, dx, N, H, W, Cin, Cout, 1, ws, nb)
    assert rel_inf(host(dx), ref) <= TOL_TF32
    _status_clean(S)


@pytest.mark.parametrize("N,H,W,Cin,Cout", CONV_CASES)
@pytest.mark.parametrize("accumulate", [0, 1])
def test_conv_dw(S, N, H, W, Cin, Cout, accumulate):
    x, _, _ = _conv_inputs(11, N, H, W, Cin, Cout)
    dy = _f32(11, "dy", (N, H, W, Cout))
    dw0 = _f32(11, "dw0", (Cout, 3, 3, Cin))
    db0 = _f32(11, "db0", Cout)
    dw_ref, db_ref = O.conv3x3_dw(x, dy)
    dw_ref = O.gradbuf_accumulate(dw0, dw_ref, 1.0, not accumulate)
    db_ref = O.gradbuf_accumulate(db0, db_ref, 1.0, not accumulate)
    dw, db = dev(dw0), dev(db0)
    ws, nb = _ws(S, S.SPRINT_CONV_DW, N, H, W, Cin, Cout)
    S.sprint_conv_dW(dev(x), dev(dy), dw, db, 1.0, accumulate, N, H, W, Cin, Cout, 1, ws, nb)
    assert rel_inf(host(dw), dw_ref) <= TOL_TF32
    assert rel_inf(host(db), db_ref) <= TOL_FP32
    _status_clean(S)


@pytest.mark.parametrize("Cin,Cout", [(3, 64), (1, 16), (4, 32)])
def test_conv_dw_rgb_pad0(S, Cin, Cout):
    N, H, W = 3, 9, 21
    x, _, _ = _conv_inputs(15, N, H, W, Cin, Cout)
    dy = _f32(15, "dy", (N, H - 2, W - 2, Cout))
    dw_ref, db_ref = O.conv3x3_dw(x, dy, pad=0)
    dw = torch.full((Cout, 3, 3, Cin), 7.0, dtype=torch.float32, device="cuda")
    n = S.sprint_conv_workspace_size(S.SPRINT_CONV_DW, N, H, W, Cin, Cout, 0)
    ws = torch.empty(max(n // 4, 1) + 64, dtype=torch.float32, device="cuda")
    S.sprint_conv_dW(dev(x), dev(dy), dw, None, 0.5, 0, N, H, W, Cin, Cout, 0, ws, n)
    assert rel_inf(host(dw), 0.5 * dw_ref) <= TOL_FP32
    _status_clean(S)


def test_conv_dw_vgg_conv1_1(S):
    """The ILSVRC-shaped VGG first layer (224 x 224 x 3 -> 64) at batch 2:
    every output against the oracle, and the same bits on a second call."""
    N, H, W, Cin, Cout = 2, 224, 224, 3, 64
    x, _, _ = _conv_inputs(16, N, H, W, Cin, Cout)
    dy = _f32(16, "dy", (N, H, W, Cout))
    dw_ref, db_ref = O.conv3x3_dw(x, dy)
    dw = torch.empty((Cout, 3, 3, Cin), dtype=torch.float32, device="cuda")
    db = torch.empty(Cout, dtype=torch.float32, device="cuda")
    ws, nb = _ws(S, S.SPRINT_CONV_DW, N, H, W, Cin, Cout)
    xd, dyd = dev(x), dev(dy)
    S.sprint_conv_dW(xd, dyd, dw, db, 1.0, 0, N, H, W, Cin, Cout, 1, ws, nb)
    assert rel_inf(host(dw), dw_ref) <= TOL_FP32
    assert rel_inf(host(db), db_ref) <= TOL_FP32
    dw1, db1 = dw.clone(), db.clone()
    S.sprint_conv_dW(xd, dyd, dw, db, 1.0, 0, N, H, W, Cin, Cout, 1, ws, nb)
    assert torch.equal(dw, dw1) and torch.equal(db, db1)
    _status_clean(S)


def test_transpose(S):
    a = _f32(13, "a", (70, 45))
    out = torch.empty((45, 70), dtype=torch.float32, device="cuda")
    S.sprint_transpose(dev(a), out, 70, 45)
    assert (host(out) == a.T).all()


def test_conv_rgb_pad0(S):
    N, H, W, Cin, Cout = 2, 9, 10, 3, 32
    x, w, b = _conv_inputs(14, N, H, W, Cin, Cout)
    ref = O.relu(O.conv3x3_fwd(x, w, b, pad=0))
    y = torch.empty((N, H - 2, W - 2, Cout), dtype=torch.float32, device="cuda")
    S.sprint_conv_fwd(dev(x), dev(w), dev(b), y, N, H, W, Cin, Cout, 0, 1, None, 0)
    assert rel_inf(host(y), ref) <= TOL_TF32
    _status_clean(S)


def test_conv_pad0(S):
    N, H, W, Cin, Cout = 2, 9, 10, 32, 32
    x, w, b = _conv_inputs(12, N, H, W, Cin, Cout)
    ref = O.conv3x3_fwd(x, w, b, pad=0)
    y = torch.empty((N, H - 2, W - 2, Cout), dtype=torch.float32, device="cuda")
    S.sprint_conv_fwd(dev(x), dev(w), dev(b), y, N, H, W, Cin, Cout, 0, 0, None, 0)
    assert rel_inf(host(y), ref) <= TOL_TF32


@pytest.mark.parametrize("N,H,W,Cin,Cout", [(32, 6, 5, 64, 64), (64, 3, 3, 32, 48), (32, 5, 7, 256, 128),
                                            (32, 3, 4, 128, 256), (32, 4, 6, 6, 32)])
def test_conv_dw_with_precomputed_xT(S, N, H, W, Cin, Cout):
    """sprint_conv_xT + sprint_conv_dW_xT: the copy made ahead of time is the one
    the weight gradient would make, so dW and db equal sprint_conv_dW bit for bit."""
    x, _, _ = _conv_inputs(12, N, H, W, Cin, Cout)
    dy = _f32(12, "dy", (N, H, W, Cout))
    n = S.sprint_conv_xT_size(N, H, W, Cin, Cout, 1)
    assert n == 4 * N * H * W * Cin
    xT = torch.empty(n // 4, dtype=torch.float32, device="cuda")
    xd, dyd = dev(x), dev(dy)
    S.sprint_conv_xT(xd, xT, N, H, W, Cin, Cout, 1)
    ws, nb = _ws(S, S.SPRINT_CONV_DW, N, H, W, Cin, Cout)
    out = []
    for use_xT in (False, True):
        dw = torch.full((Cout, 3, 3, Cin), 7.0, dtype=torch.float32, device="cuda")
        db = torch.full((Cout,), 7.0, dtype=torch.float32, device="cuda")
        if use_xT:
            S.sprint_conv_dW_xT(xd, xT, dyd, dw, db, 1.0, 0, N, H, W, Cin, Cout, 1, ws, nb)
        else:
            S.sprint_conv_dW(xd, dyd, dw, db, 1.0, 0, N, H, W, Cin, Cout, 1, ws, nb)
        out.append((host(dw), host(db)))
    assert np.array_equal(out[0][0], out[1][0]) and np.array_equal(out[0][1], out[1][1])
    dw_ref, _ = O.conv3x3_dw(x, dy)
    assert rel_inf(out[1][0], dw_ref) <= TOL_TF32
    _status_clean(S)


def test_conv_xT_needs_blocked_copies(S):
    """No blocked copy when the batch is not a multiple of 32: size 0, and the calls refuse."""
    assert S.sprint_conv_xT_size(16, 8, 8, 64, 64, 1) == 0
    x = torch.zeros(16 * 8 * 8 * 64, dtype=torch.float32, device="cuda")
    with pytest.raises(S.SprintError):
        S.sprint_conv_xT(x, x, 16, 8, 8, 64, 64, 1)


@pytest.mark.parametrize("C", [10, 1000])
def test_softmax_xent_label_out_of_range(S, C):
    """A label outside [0, C) is not read through: the row adds nothing to the
    loss, its gradient row is zero, the other rows are as usual, and the device
    status word reports it (flag 16)."""
    N = 6
    z = _f32(15, f"zb{C}", (N, C), 2.0)
    y = synth.labels(15, f"yb{C}", N, C)
    bad = y.copy()
    bad[2], bad[4] = C, -1
    loss = torch.zeros(4, dtype=torch.float32, device="cuda")
    dz = torch.empty((N, C), dtype=torch.float32, device="cuda")
    S.sprint_device_status(reset=True)
    S.sprint_softmax_xent(dev(z), dev(bad), N, C, loss, dz)
    assert S.sprint_device_status(reset=True) == 16
    good = [0, 1, 3, 5]
    loss_ref, dz_ref = O.softmax_xent(z[good], y[good])
    assert abs(host(loss)[0] - loss_ref * len(good) / N) <= 1e-5 * abs(loss_ref)
    assert rel_inf(host(dz)[good], dz_ref * len(good) / N) <= TOL_FP32
    assert not host(dz)[[2, 4]].any()
