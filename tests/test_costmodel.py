"""The SPRINT cost model's host arithmetic (Eq. (4), (6), (9), (10) of the SPRINT
report, Sec. 3.3-3.6): exact recovery of known coefficients, the role table,
and the closed forms. No GPU."""
import numpy as np
import pytest

from stale_weight_sgd_gb300 import costmodel as C
from stale_weight_sgd_gb300 import model


def test_fit_recovers_known_coefficients():
    rng = np.random.default_rng(3)
    true = np.array([2e-15, 3e-12, 1e-12, 4e-12, 5e-9, 2e-9, 7e-9, 4e-6])
    samples = []
    for _ in range(40):
        m, n, k = (int(v) for v in rng.integers(1, 6000, size=3))
        t = (true[0] * m * n * k + true[1] * m * n + true[2] * m * k + true[3] * n * k + true[4] * m + true[5] * n
             + true[6] * k + true[7])
        samples.append((m, n, k, t))
    coef = C.fit_role(samples)
    np.testing.assert_allclose(coef, true, rtol=1e-6)
    m, n, k, t = samples[7]
    assert C.predict(coef, m, n, k) == pytest.approx(t, rel=1e-9)


def test_role_table_of_the_report():
    shapes = model.layer_shapes(dict(input=(3, 8, 8), layers=[("conv", 4, True), ("conv", 6, False), ("fc", 5, False)]))
    N = 7
    first = C.role_dims(shapes[0], N, True)
    assert first == {"convolution": (8 * 8 * N, 4, 27), "dedw": (27, 4, 8 * 8 * N)}
    second = C.role_dims(shapes[1], N, False)
    assert second == {"convolution": (4 * 4 * N, 6, 36), "dedw": (36, 6, 4 * 4 * N), "dedx_conv": (4 * 4 * N, 36, 6)}
    fc = C.role_dims(shapes[2], N, False)
    assert fc == {"fc": (N, 5, 96), "dedw": (96, 5, N), "dedx_fc": (N, 96, 5)}


def test_t_gpu_is_the_sum_over_layers_and_roles():
    shapes = model.layer_shapes(dict(input=(12, 1, 1), layers=[("fc", 9, True), ("fc", 4, False)]))
    unit = {r: np.array([1.0, 0, 0, 0, 0, 0, 0, 0]) for r in C.ROLES}   # cost = m*n*k
    N = 3
    expect = 3 * 9 * 12 + 12 * 9 * 3 + 3 * 4 * 9 + 9 * 4 * 3 + 3 * 9 * 4   # fc, dedw (layer 1); fc, dedw, dedx (layer 2)
    assert C.predict_t_gpu(shapes, N, unit) == expect


def test_minibatch_average_and_epoch_time():
    # Eq. (9): 16 nodes x 3 GPUs x 5 images, one update per 0.2 s, a GPU step of 0.5 s
    nmb = C.n_minibatch_avg(16, 3, 5, 0.2, 0.5)
    assert nmb == pytest.approx(96.0, rel=1e-15)
    # Eq. (10): an epoch of the ILSVRC 2012 training set size (1,281,167 files)
    assert C.t_epoch(1281167, 0.2, nmb) == pytest.approx(1281167 * 0.2 / 96.0, rel=1e-15)
    # one GPU that updates after every step of its own: N_Minibatch_avg = N_Subbatch
    assert C.n_minibatch_avg(1, 1, 128, 0.3, 0.3) == pytest.approx(128.0)


# ---- DistBelief n_fetch / n_push version arithmetic of the trainer (host logic)

@pytest.mark.parametrize("n_fetch,n_push", [(1, 1), (2, 1), (1, 3), (3, 2), (5, 2), (4, 4), (7, 3)])
def test_fetch_push_versions_match_a_step_by_step_server(n_fetch, n_push):
    # brute force: run the server step by step, count its updates, snapshot at fetch steps
    from stale_weight_sgd_gb300.trainer import fetch_push_max_lag, fetch_push_version
    updates, fetched, worst = 0, None, 0
    for t in range(60):
        if t % n_fetch == 0:
            fetched = updates
        assert fetch_push_version(t, n_fetch, n_push) == fetched, t
        worst = max(worst, updates - fetched)
        if (t + 1) % n_push == 0:
            updates += 1
    # the ring (max_lag + 2 slots: the versions read plus the one being written) is enough
    assert worst <= fetch_push_max_lag(n_fetch, n_push)


def test_trainer_rejects_inconsistent_schedules_before_touching_the_gpu():
    from stale_weight_sgd_gb300.trainer import StaleSGD
    net = dict(input=(12, 1, 1), classes=4, layers=[("fc", 9, True), ("fc", 4, False)])
    bad = [dict(stage_delays=[1, 0]),                                          # no stage map
           dict(stage_delays=[1], stage_of_layer=[0, 1]),                      # stage without a delay
           dict(stage_delays=[1, 0], stage_of_layer=[0, 1], max_delay=2),      # two delay models
           dict(n_fetch=2, max_delay=1),
           dict(n_fetch=0, n_push=1),
           dict(hybrid_switch=3),                                              # hybrid without a pipeline
           dict(max_delay=-1)]
    for kw in bad:
        with pytest.raises(ValueError):
            StaleSGD(net, 8, **kw)
