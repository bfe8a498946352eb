"""Parity at the configured sizes: every 3x3 convolution of the ILSVRC-shaped
VGG-16 at batch 64 and of the CIFAR-shaped VGG-16 at batch 128 (the shapes the
training steps and the bench run), forward, input gradient and weight/bias
gradient through the C ABI, each with the plan the library chose for it
(tile width, CTA pair, split-K, tail split, packed taps), against the FP64
oracle on outputs it can compute one by one:
  * forward / input gradient: a sample of output pixels (the corners and edges
    included), every channel, each from the 3x3 neighbourhood the oracle's own
    convolution (pad 0) sees;
  * weight / bias gradient: a subset of output and input channels over every
    pixel of the batch (each entry of dW sums over all pixels but only one
    channel of x and one of dy, so a channel subset is exact).
Tolerances as everywhere: 1e-2 (TF32 GEMMs), 1e-5 (fp32 sums)."""
import math

import numpy as np
import pytest

import oracle as O
import synth
from helpers import TOL_FP32, TOL_TF32, at_pixels as _at, crops3x3 as _crops, host, rel_inf, sample_pixels as _pixels

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def S():
    from stale_weight_sgd_gb300 import sprint
    sprint.lib()
    return sprint


def _conv_layers(net, N):
    from stale_weight_sgd_gb300 import model
    return [(net, li, N, L.h, L.w, L.cin, L.cout) for li, L in enumerate(model.layer_shapes(model.NETWORKS[net]))
            if L.kind == "conv"]


CASES = _conv_layers("vgg_i", 64) + _conv_layers("vgg_c", 128)
PLANS = {}   # (net, li, op) -> plan, for the coverage check at the end


@pytest.mark.parametrize("net,li,N,H,W,Cin,Cout", CASES,
                         ids=[f"{c[0]}-conv{c[1]}-{c[3]}x{c[4]}x{c[5]}to{c[6]}-N{c[2]}" for c in CASES])
def test_conv_at_configured_size(S, net, li, N, H, W, Cin, Cout):
    seed = 100 + li + (0 if net == "vgg_i" else 50)
    x = synth.device_normal(seed, "x", (N, H, W, Cin)).relu_()      # a post-ReLU layer input
    w = synth.device_normal(seed, "w", (Cout, 3, 3, Cin), math.sqrt(2.0 / (9 * Cin)))
    b = synth.device_normal(seed, "b", (Cout,), 0.1)
    dy = synth.device_normal(seed, "dy", (N, H, W, Cout))
    wT = w.reshape(Cout, 9 * Cin).t().contiguous()
    nb = max(S.sprint_conv_workspace_size(op, N, H, W, Cin, Cout, 1)
             for op in (S.SPRINT_CONV_FWD, S.SPRINT_CONV_DX, S.SPRINT_CONV_DW))
    ws = torch.empty(nb // 4 + 64, dtype=torch.float32, device="cuda")
    for op in (S.SPRINT_CONV_FWD, S.SPRINT_CONV_DX, S.SPRINT_CONV_DW):
        PLANS[(net, li, op)] = S.sprint_conv_plan(op, N, H, W, Cin, Cout, 1, True)
    # the plans the training step gets: the tensor cores for every layer (the RGB layer's forward
    # with its im2col rows built in shared memory) but the RGB layer's weight gradient
    assert PLANS[(net, li, S.SPRINT_CONV_FWD)]["path"] == "tc"
    assert PLANS[(net, li, S.SPRINT_CONV_FWD)]["conv_rgb"] == (Cin == 3)
    assert PLANS[(net, li, S.SPRINT_CONV_DW)]["path"] == ("smallc" if Cin <= 4 else "tc")

    y = torch.empty((N, H, W, Cout), dtype=torch.float32, device="cuda")
    S.sprint_conv_fwd(x, w, b, y, N, H, W, Cin, Cout, 1, 1, ws, nb)
    n, h, ww = _pixels(seed, N, H, W)
    ref = O.relu(O.conv3x3_fwd(_crops(x, n, h, ww), host(w), host(b), pad=0))[:, 0, 0, :]
    e = rel_inf(_at(y, n, h, ww), ref)
    assert e <= TOL_TF32, ("forward", e)

    if li > 0:   # the first layer has no input gradient in the step
        dx = torch.empty((N, H, W, Cin), dtype=torch.float32, device="cuda")
        S.sprint_conv_dX(dy, w, wT, x, dx, N, H, W, Cin, Cout, 1, ws, nb)
        crop = _crops(dy, n, h, ww)
        ref = O.conv3x3_dx(crop, host(w), 5, 5, pad=0)[:, 2, 2, :] * O.relu_mask(_at(x, n, h, ww))
        e = rel_inf(_at(dx, n, h, ww), ref)
        assert e <= TOL_TF32, ("input gradient", e)
        del dx

    dw = torch.empty((Cout, 3, 3, Cin), dtype=torch.float32, device="cuda")
    db = torch.empty(Cout, dtype=torch.float32, device="cuda")
    S.sprint_conv_dW(x, dy, dw, db, 1.0, 0, N, H, W, Cin, Cout, 1, ws, nb)
    g = np.random.default_rng(seed + 7)
    co = np.sort(g.choice(Cout, min(Cout, 8), replace=False))
    ci = np.sort(g.choice(Cin, min(Cin, 16), replace=False))
    xs = x[..., torch.as_tensor(ci, device="cuda")].double().cpu().numpy()
    dys = dy[..., torch.as_tensor(co, device="cuda")].double().cpu().numpy()
    dw_ref, db_ref = O.conv3x3_dw(xs, dys)
    dw_got = host(dw)[co][:, :, :, ci]
    e = rel_inf(dw_got, dw_ref)
    assert e <= TOL_TF32, ("weight gradient", e)
    assert rel_inf(host(db)[co], db_ref) <= TOL_FP32
    assert S.sprint_device_status(reset=True) == 0


def test_plans_cover_every_kernel_path(S):
    """Across the configured shapes the tests above ran (this test needs them in
    the same session) every way the library tiles a convolution occurs: CTA
    pairs and single CTAs, the tail split of the last round, split-K and packed
    taps of the weight gradient, and the direct CUDA-core RGB layer."""
    if len(PLANS) < 3 * len(CASES):
        pytest.skip("run with the configured-size convolution tests")
    fwd_dx = [p for (_, _, op), p in PLANS.items() if op != S.SPRINT_CONV_DW and p["path"] == "tc"]
    dw = [p for (_, _, op), p in PLANS.items() if op == S.SPRINT_CONV_DW and p["path"] == "tc"]
    print("forward / input-gradient plans:", sorted({(p["bn"], p["pair"], p["tail_splits"]) for p in fwd_dx}))
    print("weight-gradient plans:", sorted({(p["bn"], p["pair"], p["splits"], p["wg_tpt"], p["wg_fact"]) for p in dw}))
    assert any(p["pair"] for p in fwd_dx + dw) and any(not p["pair"] for p in fwd_dx + dw)
    assert any(p["tail_splits"] > 1 for p in fwd_dx) and any(p["tail_splits"] == 1 for p in fwd_dx)
    assert any(p["splits"] > 1 for p in dw)
    assert any(p["wg_tpt"] > 0 for p in dw) and any(p["wg_tpt"] == 0 and not p["wg_fact"] for p in dw)
    assert any(p["wg_fact"] for p in dw)          # the Cout = 64 layers: factored on CTA pairs
    # the 64- and 128-channel outputs of the wide VGG-I layers: halo-staged tiles
    assert any(p["conv_halo"] for p in fwd_dx) and any(not p["conv_halo"] for p in fwd_dx)
    assert all(p["wg_blocked"] for p in dw)       # batch 64 and 128: blocked operand copies
    assert any(p["path"] == "smallc" for (_, _, op), p in PLANS.items())
