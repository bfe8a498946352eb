"""The FC backward entry point that allocates nothing (sprint_fc_bwd_static_scratch).

Its scratch is a fixed array inside the library, for callers that cannot
allocate device memory (a memory manager owns all of it, or the path must not
call cudaMalloc/cudaFree, which may synchronise the device). It runs the same
kernels as sprint_fc_bwd with a caller workspace, so on the same inputs it must
give the same bits, on repeated calls (the array keeps the previous call's
contents); both agree with the FP64 oracle within the TF32 tolerance. It must
reject shapes whose scratch need exceeds the array, accept the ones that fit
only because no transposed weight copy is formed (dx not asked for), and leave
the device's allocations untouched. This file is collected last on purpose."""
import numpy as np
import pytest

import oracle as O
import synth
from helpers import TOL_FP32, TOL_TF32, dev, host, rel_inf

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def S():
    from stale_weight_sgd_gb300 import sprint
    sprint.lib()
    return sprint


def _case(seed, N, fin, fout):
    x = np.maximum(synth.normal(seed, "x", (N, fin)), 0)
    w = synth.normal(seed, "w", (fout, fin), np.sqrt(2.0 / fin))
    dy = synth.normal(seed, "dy", (N, fout))
    return x, w, dy


def _with_workspace(S, x, w, wT, dy, N, fin, fout, accumulate, dw0, db0, want_dx=True):
    nb = S.sprint_fc_workspace_size(N, fin, fout, wT is not None or not want_dx)
    ws = torch.empty(nb // 4 + 64, dtype=torch.float32, device="cuda")
    dx = torch.empty((N, fin), dtype=torch.float32, device="cuda") if want_dx else None
    dw, db = dev(dw0), dev(db0)
    xd = dev(x)
    S.sprint_fc_bwd(xd, dev(w), wT, dev(dy), xd, dx, dw, db, 0.5, accumulate, N, fin, fout, ws, nb)
    return (host(dx) if want_dx else None), host(dw), host(db)


def _static(S, x, w, wT, dy, N, fin, fout, accumulate, dw0, db0, want_dx=True):
    dx = torch.empty((N, fin), dtype=torch.float32, device="cuda") if want_dx else None
    dw, db = dev(dw0), dev(db0)
    xd = dev(x)
    S.sprint_fc_bwd_static_scratch(xd, dev(w), wT, dev(dy), xd, dx, dw, db, 0.5, accumulate, N, fin, fout)
    return (host(dx) if want_dx else None), host(dw), host(db)


def _oracle(x, w, dy, accumulate, dw0, db0):
    """dx masked by the layer input's ReLU, dw/db = accumulate*old + 0.5*gradient."""
    dx, dw, db = O.fc_bwd(x, w, dy)
    dx = dx * O.relu_mask(x)
    keep = 1.0 if accumulate else 0.0
    return dx, keep * np.asarray(dw0, np.float64) + 0.5 * dw, keep * np.asarray(db0, np.float64) + 0.5 * db


@pytest.mark.parametrize("N,fin,fout,with_wT", [(512, 320, 384, 1), (300, 200, 136, 0), (64, 256, 512, 1)])
def test_static_scratch_matches_workspace_version_twice(S, N, fin, fout, with_wT):
    for call, seed in enumerate((21, 22)):       # two calls in a row, different data
        x, w, dy = _case(seed + N, N, fin, fout)
        dw0 = synth.normal(seed, "dw0", (fout, fin))
        db0 = synth.normal(seed, "db0", fout)
        wT = dev(np.ascontiguousarray(w.T)) if with_wT else None
        acc = call % 2
        ref = _with_workspace(S, x, w, wT, dy, N, fin, fout, acc, dw0, db0)
        got = _static(S, x, w, wT, dy, N, fin, fout, acc, dw0, db0)
        for g, r in zip(got, ref):
            assert np.array_equal(g, r)          # the same kernels on the same inputs: the same bits
        for g, r, tol in zip(got, _oracle(x, w, dy, acc, dw0, db0), (TOL_TF32, TOL_TF32, TOL_FP32)):
            assert rel_inf(g, r) <= tol
    assert S.sprint_device_status(reset=True) == 0


def test_static_scratch_without_dx_fits_without_the_weight_copy(S):
    """dx not asked for and wT absent: no transposed weight copy is formed, so a
    shape whose scratch need is over the limit with that copy but under it
    without is accepted, and matches sprint_fc_bwd bit for bit."""
    cap = S.sprint_fc_bwd_static_scratch_bytes()
    N, fin, fout = 256, 2048, 2560
    assert S.sprint_fc_workspace_size(N, fin, fout, 0) > cap >= S.sprint_fc_workspace_size(N, fin, fout, 1)
    for call, seed in enumerate((41, 42)):
        x, w, dy = _case(seed, N, fin, fout)
        dw0 = synth.normal(seed, "dw0", (fout, fin))
        db0 = synth.normal(seed, "db0", fout)
        ref = _with_workspace(S, x, w, None, dy, N, fin, fout, call, dw0, db0, want_dx=False)
        got = _static(S, x, w, None, dy, N, fin, fout, call, dw0, db0, want_dx=False)
        assert np.array_equal(got[1], ref[1]) and np.array_equal(got[2], ref[2])
        o = _oracle(x, w, dy, call, dw0, db0)
        assert rel_inf(got[1], o[1]) <= TOL_TF32 and rel_inf(got[2], o[2]) <= TOL_FP32
    # with dx asked for and no wT the same shape needs the weight copy too: rejected
    with pytest.raises(S.SprintError) as e:
        S.sprint_fc_bwd_static_scratch(16, 16, None, 16, None, 16, 16, None, 1.0, 0, N, fin, fout)
    assert e.value.status == 7


def test_static_scratch_allocates_nothing(S):
    """After a first call (which looks up the array's address), further calls
    change neither the device's free memory nor the caching allocator's count."""
    N, fin, fout = 128, 512, 384
    x, w, dy = _case(5, N, fin, fout)
    xd, wd, dyd = dev(x), dev(w), dev(dy)
    dx = torch.empty((N, fin), dtype=torch.float32, device="cuda")
    dw = torch.empty((fout, fin), dtype=torch.float32, device="cuda")
    db = torch.empty(fout, dtype=torch.float32, device="cuda")
    S.sprint_fc_bwd_static_scratch(xd, wd, None, dyd, xd, dx, dw, db, 1.0, 0, N, fin, fout)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    alloc0 = torch.cuda.memory_allocated()
    for _ in range(5):
        S.sprint_fc_bwd_static_scratch(xd, wd, None, dyd, xd, dx, dw, db, 1.0, 1, N, fin, fout)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == alloc0
    assert free1 == free0
    assert S.sprint_device_status(reset=True) == 0


def test_static_scratch_rejects_oversize(S):
    cap = S.sprint_fc_bwd_static_scratch_bytes()
    assert cap == 24 << 20
    N, fin, fout = 1024, 8192, 8192     # x^T and dy^T alone need 64 MiB
    assert S.sprint_fc_workspace_size(N, fin, fout, 1) > cap
    with pytest.raises(S.SprintError) as e:
        S.sprint_fc_bwd_static_scratch(16, 16, 16, 16, None, 16, 16, None, 1.0, 0, N, fin, fout)
    assert e.value.status == 7 and "static scratch" in str(e.value)
