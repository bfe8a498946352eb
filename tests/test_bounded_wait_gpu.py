"""The failure path of the bounded waits: a wait that runs out sets a bit in
the device status word, the kernel returns, sprint_device_status reports it,
and the context stays usable. The wait is made to run out on an mbarrier that
nothing completes (sprint_selftest_bounded_wait: no copy or MMA in flight), so
no GPU fault, trap or hang is involved."""
import numpy as np
import pytest

import oracle as O
import synth
from helpers import TOL_TF32, dev, host, rel_inf

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def test_wait_runs_out_sets_flag_and_device_stays_usable():
    import ctypes

    from stale_weight_sgd_gb300 import sprint as S
    S.lib()
    torch.cuda.set_device(0)
    assert S.sprint_device_status(reset=True) == 0
    limit_ns = 3_000_000
    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    S.sprint_selftest_bounded_wait(limit_ns)
    e.record()
    torch.cuda.synchronize()
    assert a.elapsed_time(e) >= limit_ns / 1e6 * 0.9      # it did wait about the limit
    v = ctypes.c_int(0)
    rc = S.lib().sprint_device_status(ctypes.byref(v), 1)   # read and clear
    assert rc == 6 and v.value & 8, (rc, v.value)           # SPRINT_ERR_DEVICE_FLAG, self-test bit
    assert "bounded wait" in S.sprint_last_error()
    assert S.sprint_device_status(reset=True) == 0
    # the context still runs the pipelined tensor-core kernels correctly
    M, K, N = 256, 320, 192
    x = synth.normal(1, "x", (M, K))
    w = synth.normal(1, "w", (N, K), 0.05)
    b = synth.normal(1, "b", N)
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    S.sprint_fc_fwd(dev(x), dev(w), dev(b), y, M, K, N, 0)
    assert rel_inf(host(y), O.fc_fwd(x, w, b)) <= TOL_TF32
    assert S.sprint_device_status(reset=True) == 0


def test_selftest_limit_is_validated():
    from stale_weight_sgd_gb300 import sprint as S
    with pytest.raises(S.SprintError) as e:
        S.sprint_selftest_bounded_wait(10)
    assert e.value.status == 1
