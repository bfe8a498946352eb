"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin fails.

Each mutant replaces one oracle function with a wrong version (a flipped index,
a dropped term, a wrong sign, a transposed operand) and re-runs the pin that
should catch it."""
import numpy as np
import pytest

import oracle as O
import oracle.oracle as OM
import test_oracle_pins as P

_ORIG = {k: getattr(OM, k) for k in ("conv3x3_dx", "conv3x3_fwd", "conv3x3_dw", "softmax_xent", "fc_bwd")}


def _flipped_dx(dy, w, h, wd, pad=1):
    return _ORIG["conv3x3_dx"](dy, w[:, ::-1, ::-1, :], h, wd, pad)


def _no_bias_fwd(x, w, b, pad=1):
    return _ORIG["conv3x3_fwd"](x, w, None, pad)


def _swapped_taps_fwd(x, w, b, pad=1):
    return _ORIG["conv3x3_fwd"](x, np.swapaxes(w, 1, 2), b, pad)


def _dw_taps_transposed(x, dy, pad=1):
    dw, db = _ORIG["conv3x3_dw"](x, dy, pad)
    return np.swapaxes(dw, 1, 2), db


def _dw_pad_ignored(x, dy, pad=1):
    return _ORIG["conv3x3_dw"](x, dy, 1)


def _db_first_image_only(x, dy, pad=1):
    dw, _ = _ORIG["conv3x3_dw"](x, dy, pad)
    return dw, np.asarray(dy, float)[0].sum(axis=(0, 1))


def _softmax_sum(z, labels, reduction="mean"):
    loss, dz = _ORIG["softmax_xent"](z, labels, reduction)
    return loss, dz * z.shape[0]


def _momentum_sign(w, v, bufs, eta, nu):
    v_new = nu * np.asarray(v, float) + eta * OM.sum_buffers(bufs)
    return np.asarray(w, float) + v_new, v_new


def _adagrad_no_square(w, g2, bufs, eta, eps):
    s = OM.sum_buffers(bufs)
    g_new = np.asarray(g2, float) + np.abs(s)
    return np.asarray(w, float) - eta * s / (np.sqrt(g_new) + eps), g_new


def _pool_last_max(x):
    x = np.asarray(x)
    n, h, w, c = x.shape
    best = x[:, 0:h:2, 0:w:2, :].astype(float)
    arg = np.zeros(best.shape, np.uint8)
    for code in (1, 2, 3):
        dy, dx = divmod(code, 2)
        v = x[:, dy:h:2, dx:w:2, :].astype(float)
        ge = v >= best
        best = np.where(ge, v, best)
        arg[ge] = code
    return best, arg


def _stale_off_by_one(t, s):
    return max(0, t - s + 1)


def _fc_bwd_half_db(x, w, dy):
    dx, dw, db = _ORIG["fc_bwd"](x, w, dy)
    return dx, dw, db * 0.5


def _nesterov_old_velocity(w, v, bufs, eta, nu, weight_decay=0.0):
    s = OM.decayed_sum(w, bufs, weight_decay)
    v_new = nu * np.asarray(v, float) - eta * s
    return np.asarray(w, float) + nu * np.asarray(v, float) - eta * s, v_new


def _decay_sign(w, bufs, weight_decay=0.0):
    return OM.sum_buffers(bufs) - weight_decay * np.asarray(w, float)


def _never_switch(stage_delays, k, t, hybrid_switch=None):
    return int(stage_delays[k])


def _stale_weights_only(layers, stage_of_layer, stage_delays):
    stale = total = 0
    for li, L in enumerate(layers):
        n = int(np.prod(L.w_shape))
        total += n + L.cout
        if stage_delays[stage_of_layer[li]] > 0:
            stale += n
    return 100.0 * stale / total


MUTANTS = [
    ("conv3x3_dx", _flipped_dx, P.test_conv_adjoint_identities, ()),
    ("conv3x3_fwd", _no_bias_fwd, P.test_conv_fwd_brute_force, (1,)),
    ("conv3x3_fwd", _swapped_taps_fwd, P.test_conv_fwd_im2col_route, ()),
    ("conv3x3_dw", _dw_taps_transposed, P.test_conv_dw_brute_force, (1,)),
    ("conv3x3_dw", _dw_pad_ignored, P.test_conv_dw_brute_force, (0,)),
    ("conv3x3_dw", _db_first_image_only, P.test_conv_dw_brute_force, (1,)),
    ("softmax_xent", _softmax_sum, P.test_softmax_fd_and_stability, ()),
    ("update_momentum", _momentum_sign, P.test_momentum_constant_gradient_closed_form, ()),
    ("update_adagrad", _adagrad_no_square, P.test_adagrad_constant_gradient_closed_form, ()),
    ("maxpool2x2_fwd", _pool_last_max, P.test_pool_brute_force_with_ties, ()),
    ("version_used", _stale_off_by_one, P.test_constant_delay_matches_explicit_loop, ()),
    ("fc_bwd", _fc_bwd_half_db, P.test_network_gradient_finite_differences, (P.SMALL_MLP,)),
    ("update_nesterov", _nesterov_old_velocity, P.test_nesterov_constant_gradient_closed_form, ()),
    ("decayed_sum", _decay_sign, P.test_weight_decay_alone_is_geometric_shrink, ()),
    ("stage_delay", _never_switch, P.test_hybrid_switch_endpoints_and_prefix, ()),
    ("stale_weight_percent", _stale_weights_only, P.test_stale_weight_percent_vgg_by_hand, ()),
]


@pytest.mark.parametrize("name,mutant,pin,args", MUTANTS, ids=[m[0] + ":" + m[1].__name__ for m in MUTANTS])
def test_pin_catches_planted_mistake(monkeypatch, name, mutant, pin, args):
    monkeypatch.setattr(OM, name, mutant)
    monkeypatch.setattr(O, name, mutant, raising=False)
    with pytest.raises(AssertionError):
        pin(*args)
