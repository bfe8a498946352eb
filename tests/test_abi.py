"""C-ABI checks that need no GPU: the library builds, loads, exports every
function include/sprint.h declares, and its host-side validation returns the
documented status codes before touching the device."""
import ctypes

import numpy as np
import pytest

import oracle as O


@pytest.fixture(scope="module")
def S():
    from stale_weight_sgd_gb300 import build, sprint
    build.build()
    sprint.lib()
    return sprint


def test_exports_every_declared_function(S):
    names = S.header_functions()
    assert len(names) >= 20
    L = S.lib()
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    # and the binding wraps each one under the same name
    assert not [n for n in names if not hasattr(S, n)]


def test_version(S):
    assert S.sprint_version() == 100


@pytest.mark.parametrize("seed,steps,R,Smax", [(0, 7, 1, 0), (1234, 50, 8, 7), (2 ** 63 + 5, 13, 4, 3)])
def test_schedule_matches_oracle_bit_exact(S, seed, steps, R, Smax):
    # two independent implementations of the same published generator
    assert (S.sprint_staleness_schedule(seed, steps, R, Smax) == O.staleness_schedule(seed, steps, R, Smax)).all()


P = ctypes.c_void_p


def test_update_rejects_bad_arguments(S):
    L = S.lib()
    arr = (P * 17)(*([16] * 17))
    assert L.sprint_apply_update_sgd(16, 16, arr, 17, 100, ctypes.c_float(0.1), None) == 4   # k > 16
    assert L.sprint_apply_update_sgd(16, 16, arr, 0, 100, ctypes.c_float(0.1), None) == 2    # k < 1
    assert L.sprint_apply_update_sgd(None, 16, arr, 2, 100, ctypes.c_float(0.1), None) == 1  # NULL w_in
    assert L.sprint_apply_update_sgd(20, 16, arr, 2, 100, ctypes.c_float(0.1), None) == 3    # misaligned
    assert L.sprint_apply_update_sgd(16, 16, arr, 2, 0, ctypes.c_float(0.1), None) == 0      # n == 0: no-op
    assert "aligned" in S.sprint_last_error()   # the message of the last failed call
    bad = (P * 2)(16, 24)
    assert L.sprint_apply_update_momentum(16, 16, 16, bad, 2, 10, ctypes.c_float(0.1), ctypes.c_float(0.9), None) == 3
    assert L.sprint_apply_update_adagrad(16, 16, None, arr, 2, 10, ctypes.c_float(0.1), ctypes.c_float(1e-8), None) == 1
    f = ctypes.c_float
    n = ctypes.c_size_t
    assert L.sprint_apply_update_t(0, 16, 16, 16, None, arr, 2, 0, 8, n(0), f(0.1), f(0), f(0), None) == 2     # no rows
    assert L.sprint_apply_update_t(0, 16, 16, 16, None, arr, 2, 4, 8, n(31), f(0.1), f(0), f(0), None) == 2    # n < 4*8
    assert L.sprint_apply_update_t(0, 16, 16, None, None, arr, 2, 4, 8, n(32), f(0.1), f(0), f(0), None) == 1  # NULL wT
    assert L.sprint_apply_update_t(1, 16, 16, 16, None, arr, 2, 4, 8, n(32), f(0.1), f(0.9), f(0), None) == 1  # NULL v
    assert L.sprint_apply_update_t(0, 16, 16, 16, None, arr, 17, 4, 8, n(32), f(0.1), f(0), f(0), None) == 4   # k > 16
    assert L.sprint_apply_update_t(5, 16, 16, 16, None, arr, 2, 4, 8, n(32), f(0.1), f(0), f(0), None) == 1    # rule
    assert L.sprint_apply_update(3, 16, 16, None, arr, 2, n(8), f(0.1), f(0.9), f(0), None) == 1   # Nesterov, NULL v
    assert L.sprint_apply_update(4, 16, 16, 16, arr, 2, n(8), f(0.1), f(0.9), f(0), None) == 1     # unknown rule


def test_shape_and_workspace_errors(S):
    L = S.lib()
    assert L.sprint_fc_fwd(16, 16, None, 16, 0, 8, 8, 0, None) == 2
    assert L.sprint_pool_fwd(16, 16, 16, 1, 1, 4, 4, None) == 2
    assert L.sprint_softmax_xent(16, 16, 0, 10, 16, 16, 0, None) == 2
    assert L.sprint_im2col(16, 1, 4, 4, 3, 2, 16, None, None) == 2          # pad 2
    assert L.sprint_conv_fwd(16, 16, None, 16, 1, 4, 4, 3, 8, 5, 1, None, 0, None) == 2
    need = S.sprint_fc_workspace_size(64, 256, 512, 0)
    assert need > 0
    rc = L.sprint_fc_bwd(16, 16, None, 16, None, 16, 16, None, ctypes.c_float(1), 0, 64, 256, 512, 16, need - 16, None)
    assert rc == 7 and "workspace" in S.sprint_last_error()
    assert S.sprint_fc_workspace_size(64, 256, 512, 1) < need       # wT supplied: no transposed copy needed
    assert S.sprint_conv_workspace_size(2, 8, 16, 16, 64, 64, 1) > 0  # dedw: transposed copies
    assert S.sprint_conv_workspace_size(9, 8, 16, 16, 64, 64, 1) == 0
    # the RGB layer's dedw: block partials of Cout * (9 * Cin + 1) floats, far
    # below the transposed copies (x^T 9.6 MB + dy^T 205.5 MB at 16 x 224 x 224)
    rgb = S.sprint_conv_workspace_size(2, 16, 224, 224, 3, 64, 1)
    per_block = 64 * (9 * 3 + 1) * 4
    assert rgb % per_block < 256 and 1 <= rgb // per_block <= 4 * 1024
    assert rgb < 16 * 224 * 224 * (3 + 64) * 4 // 50
    assert S.sprint_conv_workspace_size(2, 16, 224, 224, 3, 96, 1) > 16 * 224 * 224 * 96 * 4   # Cout > 64: copies
    assert L.sprint_transpose(16, 16, 4, 4, None) == 1               # aliasing


def test_halo_tile_plans(S):
    """Host-side tile choice of the halo-staged forward / input gradient: 64 outputs on CTA
    pairs, factored to 192 columns, tiles of whole output rows filling >= 80% of the 128 MMA
    rows; 128 outputs flipped (weights as the 128-row operand, 256 tile positions as N, one
    CTA per tile) when such tiles fill >= 80% of the positions; the halo buffer within its stage."""
    def plan(op, N, H, W, Cin, Cout):
        return S.sprint_conv_plan(op, N, H, W, Cin, Cout, 1, True)
    for N, H, W, Cin, Cout, bw, bh in [(64, 224, 224, 64, 64, 112, 1), (1, 3, 221, 64, 64, 111, 1)]:
        p = plan(0, N, H, W, Cin, Cout)
        assert p["conv_halo"] == 1 and p["conv_hflip"] == 0 and p["pair"] == 1 and p["bn"] == 192, p
        assert (p["box_w"], p["box_h"], p["box_img"]) == (bw, bh, 1)
        assert p["num_kt"] == 9 * Cin // 32
        assert (bw + 2) * bh <= 128 and 2 * (bw + 2) + 130 <= 360   # the last tap's window inside the buffer
    for op, N, H, W, Cin, Cout, bw, bh in [(0, 64, 112, 112, 64, 128, 112, 2), (0, 64, 112, 112, 128, 128, 112, 2),
                                           (1, 64, 56, 56, 128, 256, 56, 4), (0, 2, 15, 28, 64, 128, 28, 8)]:
        p = plan(op, N, H, W, Cin, Cout)
        assert p["conv_halo"] == 1 and p["conv_hflip"] == 1 and p["pair"] == 0 and p["bn"] == 128, p
        assert (p["box_w"], p["box_h"]) == (bw, bh)
        assert (bw + 2) * bh <= 256 and max((bh + 2) * (bw + 2), 2 * (bw + 2) + 258) <= 488
    assert plan(1, 64, 112, 112, 64, 128)["conv_halo"] == 1           # dX of conv2_1: 64 outputs, factored
    assert plan(1, 64, 112, 112, 128, 128)["conv_halo"] == 0          # dX, 128 outputs, 4 chunks: tap by tap
    p = plan(0, 1, 2, 452, 32, 128)                                   # rows too wide to flip: pair tiles
    assert p["conv_halo"] == 1 and p["conv_hflip"] == 0 and p["pair"] == 1 and p["bn"] == 128
    assert plan(0, 64, 56, 56, 128, 256)["conv_halo"] == 0            # 256 output channels: tap by tap
    assert plan(0, 64, 14, 14, 64, 64)["conv_halo"] == 0              # 196 of 256 rows: tap by tap
    assert plan(0, 128, 16, 16, 128, 128)["conv_halo"] == 0           # 256 of 512 positions: tap by tap
    assert plan(0, 2, 4, 100, 64, 64)["conv_fact"] == 1               # 100 of 128 rows: factored
    assert plan(0, 2, 8, 8, 48, 64)["conv_halo"] == 0                 # input channels % 32 != 0


def test_rgb_layer_plans(S):
    """The RGB layer's forward (3 -> 64 channels, pad 1) takes the tensor cores with its
    im2col rows built in shared memory; other few-channel forwards stay on the CUDA cores."""
    for shape in [(64, 224, 224, 3, 64), (128, 32, 32, 3, 64), (3, 7, 9, 3, 64)]:
        p = S.sprint_conv_plan(0, *shape, 1, True)
        assert p["path"] == "tc" and p["conv_rgb"] == 1 and p["bn"] == 64 and p["num_kt"] == 1
        assert S.sprint_conv_workspace_size(0, *shape, 1) == 64 * 32 * 4   # the padded weights
    for shape in [(8, 32, 32, 3, 16), (2, 11, 9, 4, 64), (2, 37, 35, 3, 48)]:
        p = S.sprint_conv_plan(0, *shape, 1, True)
        assert p["conv_rgb"] == 0 and p["path"] == "smallc"


def test_batched_entry_points_validate(S):
    L = S.lib()
    f1 = ctypes.c_float(1)
    ok = (P * 3)(16, 32, 48)
    mis = (P * 3)(16, 36, 48)
    nul = (P * 3)(16, None, 48)
    # batch 0 is a no-op; shapes checked first
    assert L.sprint_fc_fwd_batched(None, None, None, None, None, 0, 8, 8, 8, 0, None, 0, None) == 0
    assert L.sprint_fc_fwd_batched(ok, ok, None, ok, None, 3, 0, 8, 8, 0,None, 0, None) == 2
    assert L.sprint_fc_fwd_batched(None, ok, None, ok, None, 3, 8, 8, 8, 0,None, 0, None) == 1      # NULL array
    assert L.sprint_fc_fwd_batched(ok, nul, None, ok, None, 3, 8, 8, 8, 0,None, 0, None) == 1       # NULL entry
    assert L.sprint_fc_fwd_batched(ok, ok, mis, ok, None, 3, 8, 8, 8, 0,None, 0, None) == 3         # misaligned bias entry
    assert "b[1]" in S.sprint_last_error()
    need = S.sprint_fc_batched_workspace_size(3, 64, 256, 512, 0)
    tail = S.sprint_fc_fwd_batched_workspace_size()
    assert tail > 0 and need >= 3 * S.sprint_fc_workspace_size(64, 256, 512, 0) + tail
    need -= tail   # the per-problem slices alone are accepted
    assert S.sprint_fc_batched_workspace_size(0, 64, 256, 512, 0) == 0
    # (x, xT1, w, wT, dy, dyT, relu_src, dx, dxT, dw, db, ...)
    rc = L.sprint_fc_bwd_batched(ok, None, ok, None, ok, None, None, ok, None, ok, None, f1, 0, 3, 64, 256, 512, 16,
                                 need - 16, None)
    assert rc == 7 and "workspace" in S.sprint_last_error()
    assert L.sprint_fc_bwd_batched(ok, None, ok, None, ok, None, None, ok, None, None, None, f1, 0, 3, 64, 256, 512,
                                   16, need, None) == 1   # dw array is required
    assert L.sprint_fc_bwd_batched(ok, mis, ok, None, ok, None, None, ok, None, ok, None, f1, 0, 3, 64, 256, 512,
                                   16, need, None) == 3   # misaligned xT1 entry
    assert "xT1[1]" in S.sprint_last_error()
    assert L.sprint_fc_bwd_batched(ok, None, ok, None, ok, None, None, None, ok, ok, None, f1, 0, 3, 64, 256, 512,
                                   16, need, None) == 1   # dxT without dx
    assert L.sprint_fc_fwd_batched(ok, ok, None, ok, nul, 3, 8, 8, 8, 0, None, 0, None) == 1   # NULL yT entry
    assert L.sprint_softmax_xent_batched(ok, ok, ok, nul, 3, 8, 10, 0, None) == 1
    assert L.sprint_softmax_xent_batched(ok, ok, mis, ok, 3, 8, 10, 0, None) == 3
    assert L.sprint_softmax_xent_batched(None, None, None, None, 0, 8, 10, 0, None) == 0


def test_binding_raises_with_message(S):
    with pytest.raises(S.SprintError) as e:
        S.sprint_apply_update_sgd(16, 16, [16] * 17, 10, 0.1, stream=0)
    assert "SPRINT_ERR_UNSUPPORTED" in str(e.value)


def test_no_cpu_fallback_in_product_path():
    import os
    import re
    root = os.path.join(os.path.dirname(os.path.dirname(__file__)), "stale_weight_sgd_gb300")
    for dirpath, _, files in os.walk(root):
        for f in files:
            if f.endswith(".py"):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle", src, re.M), f
                assert not re.search(r"^\s*(import|from)\s+synth", src, re.M), f


def test_stale_weight_metrics_match_the_oracle():
    # host logic of the pipeline metrics against the oracle's own count (VGG-16, CIFAR shape)
    import oracle as O
    from stale_weight_sgd_gb300 import model
    shapes = model.layer_shapes(model.NETWORKS["vgg_c"])
    layers = O.build_layers(O.ARCHS["vgg_c"])
    for delays in ([3, 2, 1, 0], [0, 0, 0, 0], [1, 0, 2, 0], [5, 5, 5, 5]):
        assert model.stale_weight_percent(shapes, model.VGG_C_STAGES, delays) == pytest.approx(
            O.stale_weight_percent(layers, model.VGG_C_STAGES, delays), rel=1e-15)
        assert model.staleness_degrees(delays) == O.staleness_degrees(delays)
