"""The FC backward entry point that allocates nothing (sprint_fc_bwd_static_scratch).

Its scratch is a fixed array inside the library, for callers that cannot
allocate device memory (a memory manager owns all of it, or the path must not
call cudaMalloc/cudaFree, which may synchronise the device). It must give the
same results as sprint_fc_bwd with a caller workspace, on repeated calls (the
array keeps the previous call's contents), and reject shapes whose scratch need
exceeds the array. This file is collected last on purpose."""
import numpy as np
import pytest

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


def _with_workspace(S, x, w, wT, dy, N, fin, fout, accumulate, dw0, db0):
    nb = S.sprint_fc_workspace_size(N, fin, fout, wT is not None)
    ws = torch.empty(nb // 4 + 64, dtype=torch.float32, device="cuda")
    dx = torch.empty((N, fin), dtype=torch.float32, device="cuda")
    dw, db = dev(dw0), dev(db0)
    xd = dev(x)
    S.sprint_fc_bwd(xd, dev(w), wT, dev(dy), xd, dx, dw, db, 0.5, accumulate, N, fin, fout, ws, nb)
    return host(dx), host(dw), host(db)


def _static(S, x, w, wT, dy, N, fin, fout, accumulate, dw0, db0):
    dx = torch.empty((N, fin), dtype=torch.float32, device="cuda")
    dw, db = dev(dw0), dev(db0)
    xd = dev(x)
    S.sprint_fc_bwd_static_scratch(xd, dev(w), wT, dev(dy), xd, dx, dw, db, 0.5, accumulate, N, fin, fout)
    return host(dx), host(dw), host(db)


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
        for g, r, tol in zip(got, ref, (TOL_TF32, TOL_TF32, TOL_FP32)):
            assert rel_inf(g, r) <= tol
    assert S.sprint_device_status(reset=True) == 0


def test_static_scratch_rejects_oversize(S):
    cap = S.sprint_fc_bwd_static_scratch_bytes()
    assert cap == 24 << 20
    N, fin, fout = 1024, 8192, 8192     # x^T and dy^T alone need 64 MiB
    assert S.sprint_fc_workspace_size(N, fin, fout, 1) > cap
    with pytest.raises(S.SprintError) as e:
        S.sprint_fc_bwd_static_scratch(16, 16, 16, 16, None, 16, 16, None, 1.0, 0, N, fin, fout)
    assert e.value.status == 7 and "static scratch" in str(e.value)
