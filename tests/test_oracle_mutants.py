"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin fails.

Each mutant replaces one oracle function with a wrong version (a flipped index,
a dropped term, a wrong sign, a transposed operand) and re-runs the pin that
should catch it."""
import numpy as np
import pytest

import oracle as O
import oracle.oracle as OM
import test_oracle_pins as P

_ORIG = {k: getattr(OM, k) for k in ("conv3x3_dx", "conv3x3_fwd", "softmax_xent", "fc_bwd")}


def _flipped_dx(dy, w, h, wd, pad=1):
    return _ORIG["conv3x3_dx"](dy, w[:, ::-1, ::-1, :], h, wd, pad)


def _no_bias_fwd(x, w, b, pad=1):
    return _ORIG["conv3x3_fwd"](x, w, None, pad)


def _swapped_taps_fwd(x, w, b, pad=1):
    return _ORIG["conv3x3_fwd"](x, np.swapaxes(w, 1, 2), b, pad)


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


MUTANTS = [
    ("conv3x3_dx", _flipped_dx, P.test_conv_adjoint_identities, ()),
    ("conv3x3_fwd", _no_bias_fwd, P.test_conv_fwd_brute_force, (1,)),
    ("conv3x3_fwd", _swapped_taps_fwd, P.test_conv_fwd_im2col_route, ()),
    ("softmax_xent", _softmax_sum, P.test_softmax_fd_and_stability, ()),
    ("update_momentum", _momentum_sign, P.test_momentum_constant_gradient_closed_form, ()),
    ("update_adagrad", _adagrad_no_square, P.test_adagrad_constant_gradient_closed_form, ()),
    ("maxpool2x2_fwd", _pool_last_max, P.test_pool_brute_force_with_ties, ()),
    ("version_used", _stale_off_by_one, P.test_constant_delay_matches_explicit_loop, ()),
    ("fc_bwd", _fc_bwd_half_db, P.test_network_gradient_finite_differences, (P.SMALL_MLP,)),
]


@pytest.mark.parametrize("name,mutant,pin,args", MUTANTS, ids=[m[0] + ":" + m[1].__name__ for m in MUTANTS])
def test_pin_catches_planted_mistake(monkeypatch, name, mutant, pin, args):
    monkeypatch.setattr(OM, name, mutant)
    monkeypatch.setattr(O, name, mutant, raising=False)
    with pytest.raises(AssertionError):
        pin(*args)
