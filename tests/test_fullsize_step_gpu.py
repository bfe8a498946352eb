"""Whole training steps at the configured sizes against the FP64 oracle.

  * SMLPs (3072 -> 5000 x5 -> 10), 4 replicas x batch 512, seeded delays in
    {0..3}, eta 0.01: steps 1 and 2 checked step-locally and layer-locally
    (every layer's output, every gradient tensor, the loss, the update);
  * VGG-16 CIFAR-shaped at batch 128, momentum 0.9, pipeline stages delayed
    3,2,1,0: step 3 (the first whose four stages read four different
    versions) checked the same way;
  * VGG-16 ILSVRC-shaped, 8 replicas x batch 64, delays in {0..7}, eta 0.005,
    issued exactly as the bench issues it (replica streams, update stream):
    step 1 of replicas 0 and 7 checked on what the oracle can compute one by
    one at this size: every layer's output on sampled pixels (full FC
    outputs), pool outputs and argmaxes bit-exact on sampled windows, the loss
    against the oracle softmax of the GPU logits, the gradients of the last
    six layers (conv5_1 .. fc3) in full by replaying the oracle's backward pass
    on the GPU's saved activations, and the update on sampled parameters.
The replayed decisions (ReLU masks, pool argmaxes) are read from the kernel's
values on both sides, as in the smaller step tests."""
import math

import numpy as np
import pytest

import oracle as O
import synth
from helpers import TOL_TF32, TOL_UPDATE, at_pixels as _at, crops3x3 as _crops, rel_inf, sample_pixels as _pixels
from test_step_gpu import _check_step_local, _run_gpu

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def test_smlps_full_size_steps():
    arch = O.ARCHS["smlps"]
    kw = dict(replicas=4, max_delay=3, schedule_seed=11, eta=0.01)
    run = _run_gpu(arch, 512, 3, 8, 3, kw, keep_steps=(1, 2))
    _check_step_local(arch, run, kw, check_steps=(1, 2))


def test_vgg_c_full_size_pipelined_step():
    from stale_weight_sgd_gb300.model import VGG_C_STAGES
    arch = O.ARCHS["vgg_c"]
    kw = dict(optimizer="momentum", eta=0.01, stage_of_layer=VGG_C_STAGES, stage_delays=[3, 2, 1, 0])
    run = _run_gpu(arch, 128, 4, 4, 3, kw, keep_steps=(3,))
    _check_step_local(arch, run, kw, check_steps=(3,))


def test_vgg_i_full_size_bench_configuration():
    # as the bench: the trainer issues on a high-priority stream of its own
    with torch.cuda.stream(torch.cuda.Stream(priority=-1)):
        _vgg_i_full_size()


def _vgg_i_full_size():
    from stale_weight_sgd_gb300 import model
    from stale_weight_sgd_gb300.trainer import StaleSGD
    net = model.NETWORKS["vgg_i"]
    shapes = model.layer_shapes(net)
    layers = O.build_layers(O.ARCHS["vgg_i"])
    N, R, P, eta = 64, 8, 16, 0.005
    tr = StaleSGD(net, N, replicas=R, max_delay=7, schedule_seed=1234, optimizer="sgd", eta=eta)
    w0 = np.concatenate([np.concatenate([synth.normal(7, f"w{i}", (L.w_numel,), math.sqrt(2.0 / L.fan_in)),
                                         np.zeros(L.cout, np.float32)]) for i, L in enumerate(shapes)])
    tr.load_weights(w0)
    xs = synth.device_normal(1000, "x", (P, N, 224 * 224 * 3))
    g = torch.Generator(device="cuda")
    g.manual_seed(1001)
    ys = torch.randint(0, 1000, (P, N), generator=g, device="cuda", dtype=torch.int32)
    tr.set_batch_pool(xs, ys)
    tr.step()
    tr.step()
    tr.join()
    torch.cuda.synchronize()
    t = 1
    from stale_weight_sgd_gb300 import sprint as S
    assert S.sprint_device_status(reset=True) == 0
    w_after = tr.weights(2).astype(np.float64)
    offs, _ = O.param_offsets(layers)
    gbufs = [model.unpack(shapes, tr.gradbuf[r].cpu().numpy()) for r in range(R)]
    worst = dict(fwd=0.0, grad=0.0)
    for r in (0, 7):
        v = tr._version(t, r, 0)
        params = O.unflatten(layers, tr.weights(v).astype(np.float64))
        A = tr.acts[r]
        bi = (t * R + r) % P
        inp = xs[bi].reshape(N, 224, 224, 3)
        saved = []
        for li, (L, (w, b)) in enumerate(zip(layers, params)):
            if L.kind == "conv":
                y = A["outs"][li].reshape(N, L.h, L.w, L.cout)
                n, h, ww = _pixels(li * 10 + r, N, L.h, L.w, 192)
                ref = O.relu(O.conv3x3_fwd(_crops(inp, n, h, ww), w, b, pad=0))[:, 0, 0, :]
                e = rel_inf(_at(y, n, h, ww), ref)
                worst["fwd"] = max(worst["fwd"], e)
                assert e <= TOL_TF32, ("forward", r, li, e)
                nxt = y
                if L.pool:
                    arg = A["argmax"][li].reshape(N, L.h // 2, L.w // 2, L.cout)
                    pooled = A["pooled"][li].reshape(N, L.h // 2, L.w // 2, L.cout)
                    pn, ph, pw = _pixels(li * 10 + r + 5, N, L.h // 2, L.w // 2, 192)
                    win = np.stack([_at(y, pn, 2 * ph + dy_, 2 * pw + dx_) for dy_ in (0, 1) for dx_ in (0, 1)], 1)
                    win = win.reshape(-1, 2, 2, L.cout).astype(np.float32)
                    p_ref, a_ref = O.maxpool2x2_fwd(win)
                    assert (_at(arg, pn, ph, pw).astype(np.uint8) == a_ref[:, 0, 0, :]).all(), ("argmax", r, li)
                    assert (_at(pooled, pn, ph, pw) == p_ref[:, 0, 0, :]).all(), ("pooled", r, li)
                    nxt = pooled
                saved.append((inp, y, A["argmax"][li].reshape(N, L.h // 2, L.w // 2, L.cout) if L.pool else None))
                inp = nxt
            else:
                x2 = inp.reshape(N, -1).double().cpu().numpy()
                y = A["outs"][li].reshape(N, L.cout).double().cpu().numpy()
                ref = O.fc_fwd(x2, w, b)
                ref = O.relu(ref) if L.relu else ref
                e = rel_inf(y, ref)
                worst["fwd"] = max(worst["fwd"], e)
                assert e <= TOL_TF32, ("forward", r, li, e)
                saved.append((x2, y, None))
                inp = A["outs"][li].reshape(N, L.cout)
        labels = ys[bi].cpu().numpy()
        loss_ref, dz = O.softmax_xent(saved[-1][1], labels)
        loss_gpu = float(tr.loss[r, 0].item())
        if math.isfinite(loss_ref):
            assert abs(loss_gpu - loss_ref) <= 1e-5 * abs(loss_ref), ("loss", r, loss_gpu, loss_ref)
        # the backward pass of conv5_1 .. fc3, replayed on the GPU's saved activations
        k = 10
        replay = []
        for L, (a, yy, arg) in zip(layers[k:], saved[k:]):
            to_np = (lambda z: z.double().cpu().numpy()) if torch.is_tensor(a) else (lambda z: z)
            replay.append((to_np(a), to_np(yy) if torch.is_tensor(yy) else yy,
                           arg.cpu().numpy() if torch.is_tensor(arg) else arg))
        grads = O.flatten(O.backward(layers[k:], params[k:], replay, dz))
        base = offs[k][0]
        for i, L in enumerate(layers[k:], start=k):
            a, b = offs[i]
            for lo, hi in ((a, b), (b, b + L.cout)):
                e = rel_inf(gbufs[r][lo:hi], grads[lo - base:hi - base])
                worst["grad"] = max(worst["grad"], e)
                assert e <= TOL_TF32, ("gradient", r, i, lo, hi, e)
    # the update W(2) = W(1) - eta * sum_r GradBuf_r, on sampled parameters
    idx = np.sort(np.random.default_rng(5).choice(w_after.size, 1_000_000, replace=False))
    w1 = tr.weights(1).astype(np.float64)[idx]
    w_pred, _ = O.apply_update(w1, [gb[idx].astype(np.float64) for gb in gbufs], optimizer="sgd", eta=eta)
    e = rel_inf(w_after[idx], w_pred)
    assert e <= TOL_UPDATE, ("update", e)
    print(f"VGG-I full size, step 1, replicas 0 and 7: forward {worst['fwd']:.2e}, gradients (conv5_1..fc3) "
          f"{worst['grad']:.2e}, update {e:.2e}")
