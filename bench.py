"""Throughput of the stale-weight SGD hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config vgg_i|vgg_c|smlps|tiny|vgg_c_hybrid|smlps_fetch_push|ps]

A step is one pass of the whole hot path over one batch per logical replica:
every replica's forward, softmax cross-entropy and backward (gradients fused
into its GradBuf), then the parameter-server update that writes the next
weight version. Default workload: the ILSVRC-shaped VGG-16 (3x224x224 input,
13 conv3x3 layers, FC 25088-4096-4096-1000, N_Param 138,357,544), batch 64 per
replica, 8 replicas with seeded delays in {0..7}, GradBuf sum then
W -= eta * sum, eta = 0.005.

Prints one JSON line (rank 0). `value` is images/s with inputs resident in HBM;
`e2e` is the same metric with every step's inputs copied from pinned host
memory and the loss read back inside the timed region. `roofline` is the
dominant convolution kernel's achieved TF32 FLOP/s inside the timed steps
(CUDA events around the layers' per-replica launch groups) against the
measured peak. `breakdown` times one extra step issued serially, one event pair
per library call, and splits it into the SGEMM roles of the SPRINT cost model
(Eq. (4)). `--config ps` sweeps the parameter-server update instead (GB/s per
point). `--impl reference` times the FP64 CPU oracle on the same workload, each
step a bounded sample. Multi-GPU (torchrun): every rank runs an independent
replica of the workload (no data-path collective); value = the sum over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "CNN train images/s on 1 GB300; conv-GEMM % TF32 peak; update GB/s vs HBM peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TF32_OVER_BF16 = 1.1 / 2.25   # nominal dense tensor ratio (tf32 1.1 PF vs bf16 2.25 PF)

CONFIGS = {
    "vgg_i": dict(net="vgg_i", batch=64, replicas=8, max_delay=7, optimizer="sgd", eta=0.005,
                  desc="VGG-16 ILSVRC-shaped fp32 (3x224x224, N_Param 138,357,544), batch 64/replica, ASGD 8 "
                       "replicas, seeded delays {0..7}, GradBuf sum then W -= eta*sum, SGD eta=0.005"),
    "vgg_c": dict(net="vgg_c", batch=128, replicas=1, max_delay=0, optimizer="momentum", eta=0.01,
                  stage_delays=[3, 2, 1, 0],
                  desc="VGG-16 CIFAR-shaped fp32, batch 128, momentum 0.9, 4 pipeline stages s_k=3,2,1,0"),
    "smlps": dict(net="smlps", batch=512, replicas=4, max_delay=3, optimizer="sgd", eta=0.01,
                  desc="SMLPs MLP 3072-5000x5-10 fp32, batch 512/replica, ASGD 4 replicas, delays {0..3}, SGD eta=0.01"),
    "tiny": dict(net="tiny", batch=8, replicas=1, max_delay=0, optimizer="sgd", eta=0.01,
                 desc="tiny CNN (conv16-pool-conv32-pool-fc10), batch 8, SGD eta=0.01"),
    # the widened rows: hybrid pipelined -> non-pipelined training with Nesterov momentum and
    # weight decay, and DistBelief n_fetch / n_push
    "vgg_c_hybrid": dict(net="vgg_c", batch=128, replicas=1, max_delay=0, optimizer="nesterov", eta=0.01,
                         weight_decay=5e-4, stage_delays=[3, 2, 1, 0], hybrid_switch=12,
                         desc="VGG-16 CIFAR-shaped fp32, batch 128, Nesterov 0.9 + weight decay 5e-4, 4 pipeline "
                              "stages s_k=3,2,1,0 switched to non-pipelined at step 12 (hybrid)"),
    "smlps_fetch_push": dict(net="smlps", batch=512, replicas=4, max_delay=0, optimizer="adagrad", eta=0.001,
                             n_fetch=3, n_push=2,
                             desc="SMLPs MLP 3072-5000x5-10 fp32, batch 512/replica, 4 replicas, DistBelief "
                                  "n_fetch=3 / n_push=2, Adagrad eta=0.001"),
    "ps": dict(desc="parameter-server update sweep fp32: n = 1M / 16M / 138M parameters, k = 1, 2, 4, 8, 16 pending "
                    "GradBufs, SGD / momentum 0.9 / Adagrad (eta 0.01, eps 1e-8, G0 0.1)"),
}
DEFAULT_CONFIG = "vgg_i"

# The conv roofline's headline layer: VGG conv3_2 (no pool after it), batch
# 64 per replica, as (N, H, W, Cin, Cout); its launches in the timed steps give
# `achieved`, the other tensor-core layers without a pool are listed beside it.
ROOF_CONV_SHAPE = (64, 56, 56, 256, 256)
ROOF_CONV_KERNEL = ("tc_gemm_kernel<CONV_IMPL> (implicit-GEMM conv forward, TF32), VGG conv3_2 "
                    "56x56x256->256, batch 64")

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the
# roofline kernel, from one ncu capture of that kernel on the same shape; must
# be re-measured whenever that kernel or its tile choice changes (then absent).
PROFILED_TRAFFIC = {
    # one call: the GEMM kernel 461.8 + 47.0 MB and its tail reduction 17.1 MB (one ncu capture)
    "tc_gemm_kernel (grouped FC forward, 4 x 512x5000x5000, TF32)": 525.9e6,
    # the GEMM kernel alone: 210.3 MB read + 170.8 MB written (one ncu capture, --set full;
    # algorithmic 412 MB: x and y 205.5 MB each, the weights 2.4 MB)
    ROOF_CONV_KERNEL: 381.1e6,
}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def tf32_peaks():
    """(burst, sustained) TF32 TFLOP/s: the measured bf16 peaks times the nominal ratio."""
    peaks, src = load_peaks()
    burst = peaks["bf16_tflops"] * TF32_OVER_BF16
    sust = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) * TF32_OVER_BF16
    return burst, sust, src


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


class GemmProbe:
    """Records CUDA events, on the launching stream, around the forward FC
    GEMM launches of the given (in, out) shapes: one grouped tensor-core
    kernel per call, covering every replica of the layer. Installed by the
    bench only; the library is untouched."""

    def __init__(self, sprint_mod, torch, shapes):
        self.S = sprint_mod
        self.torch = torch
        self.shapes = set(shapes)
        self.active = False
        self.events = []
        self.desc = None
        self.orig = sprint_mod.sprint_fc_fwd_batched
        probe = self

        def fc_fwd_batched(x, w, b, y, N, i, o, relu, ws=None, ws_bytes=0, stream=None, yT=None):
            if not (probe.active and (i, o) in probe.shapes):
                return probe.orig(x, w, b, y, N, i, o, relu, ws, ws_bytes, stream, yT)
            st = (torch.cuda.ExternalStream(stream) if isinstance(stream, int) and stream != 0
                  else torch.cuda.current_stream())
            a = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            a.record(st)
            r = probe.orig(x, w, b, y, N, i, o, relu, ws, ws_bytes, stream, yT)
            e.record(st)
            probe.events.append((a, e, 2.0 * N * i * o * len(x)))
            probe.desc = f"tc_gemm_kernel (grouped FC forward, {len(x)} x {N}x{o}x{i}, TF32)"
            return r
        sprint_mod.sprint_fc_fwd_batched = fc_fwd_batched

    def summary(self):
        if not self.events:
            return None
        ms = np.array([a.elapsed_time(e) for a, e, _ in self.events])
        fl = np.array([f for _, _, f in self.events])
        return {"launches": len(ms), "mean_ms": float(ms.mean()), "total_ms": float(ms.sum()),
                "flops_per_launch": float(fl.mean()), "kernel": self.desc, "how": "events around each grouped call"}


class ConvSpanProbe:
    """Times the per-replica convolution forward groups of chosen layers inside
    the timed steps: the trainer's span hook records an event on the main
    stream before the replicas' launches are forked and one after they have
    joined, so the pair brackets exactly the R launches of that layer (which
    share the GPU: each persistent launch fills every SM). Per-launch time =
    span / R; work = 2 * pixels * Cout * 9 * Cin per launch."""

    def __init__(self, torch, tr, layers):
        self.torch = torch
        self.tr = tr
        self.layers = set(layers)
        self.active = False
        self.open = {}
        self.spans = []   # (layer, begin, end)
        tr.span_hook = self.hook

    def hook(self, tag, phase, stream):
        kind, li = tag
        if not self.active or kind != "fwd" or li not in self.layers:
            return
        ev = self.torch.cuda.Event(enable_timing=True)
        ev.record(stream)
        if phase == 0:
            self.open[li] = ev
        else:
            self.spans.append((li, self.open.pop(li), ev))

    def summary(self, shapes, N, R, desc, head=None):
        """head: the layer indices the headline figure covers (default: all probed layers);
        per_layer lists every probed layer."""
        if not self.spans:
            return None
        ms_all = np.array([a.elapsed_time(e) for _, a, e in self.spans])
        fl_all = np.array([2.0 * N * shapes[li].h * shapes[li].w * shapes[li].cout * 9 * shapes[li].cin
                           for li, _, _ in self.spans])
        sel = np.array([head is None or li in head for li, _, _ in self.spans])
        ms, fl = ms_all[sel], fl_all[sel]
        per_layer = {}
        for (li, _, _), m, f in zip(self.spans, ms_all, fl_all):
            d = per_layer.setdefault(li, [0.0, 0.0, 0])
            d[0] += m
            d[1] += f * R
            d[2] += 1
        L = shapes
        return {"launches": int(len(ms) * R), "mean_ms": float(ms.sum() / (len(ms) * R)),
                "total_ms": float(ms.sum()), "flops_per_launch": float(fl.mean()), "kernel": desc,
                "how": f"events on the main stream around each layer's {R} per-replica launches (fork to join); "
                       "per-launch time = span / replicas",
                "per_layer": {f"conv{li} {L[li].h}x{L[li].w}x{L[li].cin}->{L[li].cout}":
                              {"tflops": round(v[1] / (v[0] / 1e3) / 1e12, 1), "ms_per_launch": round(v[0] / v[2] / R, 4)}
                              for li, v in per_layer.items()}}


# the roles of the SPRINT cost model's Eq. (4) / Sec. 3.3 table, per library call
ROLE_OF_CALL = {
    "sprint_conv_fwd": "convolution",
    "sprint_conv_dW": "dedw+dedb conv",
    "sprint_conv_dX": "dedx conv",
    "sprint_fc_fwd_batched": "fc",
    "sprint_fc_bwd_batched": "fc backward (dedx fc + dedw + dedb)",
    "sprint_pool_fwd": "pool",
    "sprint_pool_bwd": "pool",
    "sprint_softmax_xent_batched": "softmax",
    "sprint_apply_update": "update",
    "sprint_apply_update_t": "update",
}


class CallProbe:
    """Wraps every library call the trainer makes with a CUDA event pair on the
    call's stream (a serial step: one stream, so the pairs are exact)."""

    def __init__(self, sprint_mod, torch):
        self.S = sprint_mod
        self.torch = torch
        self.active = False
        self.calls = []   # (name, flops, a, e)
        for name in list(ROLE_OF_CALL) + ["sprint_transpose"]:
            self._wrap(name)

    def _wrap(self, name):
        orig = getattr(self.S, name)
        torch = self.torch
        probe = self

        def wrapped(*args, **kw):
            if not probe.active:
                return orig(*args, **kw)
            a = torch.cuda.Event(enable_timing=True)
            e = torch.cuda.Event(enable_timing=True)
            st = torch.cuda.current_stream()
            a.record(st)
            r = orig(*args, **kw)
            e.record(st)
            probe.calls.append((name, probe._flops(name, args), a, e, probe._conv_key(name, args)))
            return r
        setattr(self.S, name, wrapped)

    @staticmethod
    def _flops(name, a):
        if name == "sprint_conv_fwd" or name == "sprint_conv_dW":
            N, H, W, Ci, Co = a[4:9] if name == "sprint_conv_fwd" else a[6:11]
            return 2.0 * N * H * W * Co * 9 * Ci
        if name == "sprint_conv_dX":
            N, H, W, Ci, Co = a[5:10]
            return 2.0 * N * H * W * Co * 9 * Ci
        if name == "sprint_fc_fwd_batched":
            return 2.0 * a[4] * a[5] * a[6] * len(a[0])
        if name == "sprint_fc_bwd_batched":
            N, fin, fout = a[10:13]
            return (2.0 if a[5] is None else 4.0) * N * fin * fout * len(a[0])
        return 0.0

    @staticmethod
    def _conv_key(name, a):
        op = {"sprint_conv_fwd": "fwd", "sprint_conv_dX": "dX", "sprint_conv_dW": "dW"}.get(name)
        if op is None:
            return None
        i = {"fwd": 4, "dX": 5, "dW": 6}[op]
        N, H, W, Ci, Co = a[i:i + 5]
        return f"{op} {H}x{W}x{Ci}->{Co}"

    def summary(self):
        roles, flops, conv = {}, {}, {}
        total = 0.0
        for name, f, a, e, key in self.calls:
            ms = a.elapsed_time(e)
            r = ROLE_OF_CALL.get(name, "other")
            roles[r] = roles.get(r, 0.0) + ms
            flops[r] = flops.get(r, 0.0) + f
            total += ms
            if key:
                c = conv.setdefault(key, [0.0, 0.0])
                c[0] += ms
                c[1] += f
        return {"serial_ms_per_step": round(total, 3), "calls": len(self.calls),
                "roles_ms": {r: round(v, 3) for r, v in sorted(roles.items(), key=lambda kv: -kv[1])},
                "roles_share": {r: round(v / total, 4) for r, v in roles.items()} if total else {},
                "roles_tflops": {r: round(flops[r] / (roles[r] / 1e3) / 1e12, 1) for r in roles if flops.get(r)},
                # every conv call of the step by op and layer shape (all replicas together)
                "conv_calls": {k: {"ms": round(v[0], 3), "tflops": round(v[1] / (v[0] / 1e3) / 1e12, 1)}
                               for k, v in sorted(conv.items(), key=lambda kv: -kv[1][0])}}


def dense_init(shapes, seed):
    import synth
    return np.concatenate([np.concatenate([synth.normal(seed, f"w{i}", (L.w_numel,), np.sqrt(2.0 / L.fan_in)),
                                           np.zeros(L.cout, np.float32)]) for i, L in enumerate(shapes)])


def make_trainer(cfg, N, R, concurrent, StaleSGD, model):
    net = model.NETWORKS[cfg["net"]]
    kw = dict(replicas=R, max_delay=cfg["max_delay"], schedule_seed=1234, optimizer=cfg["optimizer"], eta=cfg["eta"],
              weight_decay=cfg.get("weight_decay", 0.0))
    if "stage_delays" in cfg:
        kw = dict(stage_of_layer=model.VGG_C_STAGES, stage_delays=cfg["stage_delays"], optimizer=cfg["optimizer"],
                  eta=cfg["eta"], weight_decay=cfg.get("weight_decay", 0.0), hybrid_switch=cfg.get("hybrid_switch"))
    if "n_fetch" in cfg:
        kw.update(max_delay=0, n_fetch=cfg["n_fetch"], n_push=cfg["n_push"])
    return StaleSGD(net, N, concurrent=concurrent, **kw)


def run_ours(args, cfg, rank, world, local_rank):
    import torch

    from stale_weight_sgd_gb300 import model, sprint
    from stale_weight_sgd_gb300.trainer import StaleSGD

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    # a dedicated stream (not the legacy default stream) for the whole run: the
    # trainer issues on it, and the probes' events are recorded on it. It runs at
    # high priority so that the training step's kernels (the critical path) are
    # scheduled ahead of the trainer's low-priority update stream
    torch.cuda.set_stream(torch.cuda.Stream(dev, priority=-1))
    net = model.NETWORKS[cfg["net"]]
    shapes = model.layer_shapes(net)
    N, R = cfg["batch"], cfg["replicas"]
    c, h, w = net["input"]
    feat = c * h * w
    classes = shapes[-1].cout
    P = max(2 * R, 8)
    tr = make_trainer(cfg, N, R, not args.serial, StaleSGD, model)
    # synthetic data generated on the device (seeded), weights He-normal
    g = torch.Generator(device=dev)
    g.manual_seed(1000 + rank)
    xs = torch.randn((P, N, feat), generator=g, device=dev, dtype=torch.float32)
    ys = torch.randint(0, classes, (P, N), generator=g, device=dev, dtype=torch.int32)
    tr.set_batch_pool(xs, ys)
    wd = dense_init(shapes, 7)
    tr.load_weights(wd)

    has_conv = any(L.kind == "conv" for L in shapes)
    # roofline probe: the implicit-GEMM conv forward of the tensor-core layers without a
    # pool (their per-replica group holds conv launches only), or the grouped FC forward
    conv_layers = [i for i, L in enumerate(shapes) if L.kind == "conv" and not L.pool and
                   sprint.sprint_conv_plan(sprint.SPRINT_CONV_FWD, N, L.h, L.w, L.cin, L.cout)["path"] == "tc"]
    span_probe = ConvSpanProbe(torch, tr, conv_layers) if (has_conv and not tr.use_graphs and conv_layers) else None
    big = [(L.cin, L.cout) for L in shapes if L.kind == "fc" and L.cin * L.cout >= 20_000_000]
    gemm_probe = GemmProbe(sprint, torch, big) if not has_conv else None

    first_nonfinite = None
    for i in range(args.warmup):
        tr.step()
        if first_nonfinite is None and not math.isfinite(tr.step_loss()):
            first_nonfinite = i
    tr.prepare_graphs()   # periodic schedules: capture every step graph of a period now, replay later
    torch.cuda.synchronize()
    barrier(world)
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    for p in (span_probe, gemm_probe):
        if p is not None:
            p.active = True
    launches0 = sprint.sprint_launch_count() + tr.graph_launch_adjust
    t_first = tr.t
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(tr.main_stream)
    host_t0 = time.perf_counter()
    for _ in range(args.steps):
        tr.step()
    host_issue_ms = (time.perf_counter() - host_t0) * 1e3 / args.steps
    tr.join()   # the last step's per-layer updates are inside the timed region
    end.record(tr.main_stream)
    torch.cuda.synchronize()
    for p in (span_probe, gemm_probe):
        if p is not None:
            p.active = False
    launches = sprint.sprint_launch_count() + tr.graph_launch_adjust - launches0   # replayed graph kernels included
    clk = clocks.stop()
    ms = start.elapsed_time(end)
    ms_max = allreduce_max(ms, world)
    barrier(world)
    loss = tr.step_loss()
    if first_nonfinite is None and not math.isfinite(loss):
        first_nonfinite = f"between step {args.warmup} and step {tr.t - 1} (the timed steps)"

    # end to end, pipelined like a training loop: every step's inputs are copied from
    # pinned host memory (on a copy stream, into one of two device buffers, while the
    # previous step computes) and every step's loss is read back to pinned memory;
    # the host waits for each loss one step behind, and for the last one at the end
    hx = torch.empty((R, N, feat), dtype=torch.float32).pin_memory()
    hy = torch.empty((R, N), dtype=torch.int32).pin_memory()
    hx.copy_(xs[:R].cpu())
    hy.copy_(ys[:R].cpu())
    dxs = [torch.empty((R, N, feat), dtype=torch.float32, device=dev) for _ in range(2)]
    dys = [torch.empty((R, N), dtype=torch.int32, device=dev) for _ in range(2)]
    hloss = [torch.empty(tuple(tr.loss.shape), dtype=torch.float32).pin_memory() for _ in range(2)]
    cs = torch.cuda.Stream(dev)
    main = tr.main_stream
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_loss = [torch.cuda.Event() for _ in range(2)]

    def h2d(b):
        with torch.cuda.stream(cs):
            dxs[b].copy_(hx, non_blocking=True)
            dys[b].copy_(hy, non_blocking=True)

    if tr.lookahead:
        # step i also issues step i + 1's forward pass: one pool of two batch slots
        # (step t reads slot t % 2), step i + 1's copy made before step i is issued. The
        # forward pass the last timed step issued ahead read the old pool: dropped, so
        # the first step here computes its own (from its copied inputs)
        tr.drop_lookahead()
        pool_x = torch.empty((2 * R, N, feat), dtype=torch.float32, device=dev)
        pool_y = torch.empty((2 * R, N), dtype=torch.int32, device=dev)
        dxs = [pool_x[b * R:(b + 1) * R] for b in range(2)]
        dys = [pool_y[b * R:(b + 1) * R] for b in range(2)]
        tr.set_batch_pool(pool_x, pool_y)
        tr.prepare_graphs()
    else:
        for b in range(2):   # the step graphs read the batch buffers: capture for both
            tr.set_batch_pool(dxs[b], dys[b])
            tr.prepare_graphs()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    s0 = tr.t
    if tr.lookahead:   # step t reads slot t % 2
        h2d(s0 % 2)
        h2d((s0 + 1) % 2)
    else:              # step i reads buffer i % 2
        h2d(0)
    for i in range(args.steps):
        b = i % 2
        if not tr.lookahead:
            tr.set_batch_pool(dxs[b], dys[b])
        tr.mark_inputs(cs)          # step i waits for its copy (and, ahead, step i + 1's)
        tr.step()
        tr.join()
        ev_done[b].record(main)
        with torch.cuda.stream(main):
            hloss[b].copy_(tr.loss, non_blocking=True)   # contiguous [R][4]; column 0 = replica loss
        ev_loss[b].record(main)
        if tr.lookahead:
            if i + 2 <= args.steps:
                cs.wait_event(ev_done[b])   # step i no longer reads its slot: step i + 2's goes there
                h2d((s0 + i) % 2)
        elif i + 1 < args.steps:
            cs.wait_event(ev_done[1 - b])   # step i-1 no longer reads the other buffer
            h2d(1 - b)
        if i > 0:
            ev_loss[1 - b].synchronize()    # the host reads step i-1's loss
    ev_loss[(args.steps - 1) % 2].synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_s = allreduce_max(e2e_s, world)

    # one more step issued serially (one stream, eager, no update overlap) with an event
    # pair around every library call: the per-role split of the SPRINT cost model, Eq. (4)
    breakdown = None
    if not args.no_breakdown:
        tr.join()
        torch.cuda.synchronize()
        call_probe = CallProbe(sprint, torch)
        saved = (tr.fork, tr.upd_stream, tr.use_graphs, tr.span_hook, tr.split_bwd, tr.lookahead)
        tr.fork, tr.upd_stream, tr.use_graphs, tr.span_hook, tr.split_bwd = False, tr.main_stream, False, None, False
        # one whole step on one stream: the forward pass the last step issued ahead is
        # dropped (finished above) and issued again inside the probed step
        tr.drop_lookahead()
        tr.lookahead = False
        tr._graph_steps = False
        with torch.cuda.stream(tr.main_stream):
            call_probe.active = True
            tr.step()
            tr.join()
            call_probe.active = False
        torch.cuda.synchronize()
        tr.fork, tr.upd_stream, tr.use_graphs, tr.span_hook, tr.split_bwd, tr.lookahead = saved
        breakdown = call_probe.summary()

    imgs = R * N * args.steps * world
    value, _ = weak_scaling_value(R * N * args.steps, ms / 1e3, world)
    e2e_value = imgs / e2e_s
    burst, sust, peak_src = tf32_peaks()
    if span_probe is not None:
        # headline: the layer shape the profiled traffic was captured on, when the net has it
        head = [li for li in conv_layers if (N, shapes[li].h, shapes[li].w, shapes[li].cin, shapes[li].cout)
                == ROOF_CONV_SHAPE]
        if head:
            summ = span_probe.summary(shapes, N, R, ROOF_CONV_KERNEL, head)
        else:
            summ = span_probe.summary(shapes, N, R, "tc_gemm_kernel<CONV_IMPL> (implicit-GEMM conv forward, TF32), "
                                                    "every tensor-core layer without a pool")
    else:
        summ = gemm_probe.summary() if gemm_probe is not None else None
    roof = None
    if summ:
        achieved = summ["flops_per_launch"] / (summ["mean_ms"] / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": round(burst, 1), "unit": "TFLOP/s",
                "frac": round(achieved / burst, 4), "traffic": PROFILED_TRAFFIC.get(summ["kernel"]),
                "kernel": summ["kernel"],
                "peak_source": f"{peak_src}: bf16 burst x 1.1/2.25 (nominal tf32/bf16 dense ratio); the timed "
                               "steps ran at the clocks below",
                "peak_sustained": round(sust, 1), "frac_of_sustained": round(achieved / sust, 4),
                "launches": summ["launches"], "mean_ms": round(summ["mean_ms"], 4), "how": summ["how"]}
        if "per_layer" in summ:
            roof["per_layer"] = summ["per_layer"]
    elif breakdown:
        roof = {"note": "no in-step probe for CUDA-graph replays; see breakdown.roles_tflops (serial step)"}
    flops_step = model.train_flops_per_image(net) * R * N
    step_tflops = flops_step * args.steps / (ms_max / 1e3) / 1e12 * world
    out = {
        "metric": METRIC,
        "value": round(value, 1), "unit": "images/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_max / args.steps, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32 (tf32 tensor-core GEMMs, fp32 accumulate)",
        "data": "synthetic (seeded N(0,1) inputs, uniform labels, He-normal init)",
        "config": {"workload": cfg["desc"], "global_batch": R * N * world, "replicas_per_gpu": R,
                   "parallelism": f"replicas only x{world}" if world > 1 else "1 GPU",
                   "l2": "working set (weights, GradBufs, activations) far larger than L2; no flush needed",
                   **({"staleness_first_step": tr.staleness(t_first), "staleness_last_step": tr.staleness(tr.t - 1)}
                      if tr.pipeline else {})},
        "e2e": {"value": round(e2e_value, 1), "unit": "images/s",
                "h2d_bytes_per_step": int(hx.numel() * 4 + hy.numel() * 4),
                "d2h_bytes_per_step": int(hloss[0].numel() * 4),
                "pipelined": "step i's input copy overlaps step i-1; the host waits for each loss one step behind",
                "host_ms_per_step": round(e2e_s * 1e3 / args.steps, 3)},
        "gpu_launches": int(launches),
        "roofline": roof,
        "achieved_step_tflops": round(step_tflops, 1),
        "step_frac_of_tf32_burst": round(step_tflops / world / burst, 4),
        "breakdown": breakdown,
        "clocks": clk,
        # JSON has no NaN: a diverged run reports null
        "loss_last": loss if math.isfinite(loss) else None,
        "kernels_per_step": int(launches // args.steps),
        "host_issue_ms_per_step": round(host_issue_ms, 3),
    }
    if first_nonfinite is not None:
        out["numerics"] = {
            "loss_first_nonfinite_step": first_nonfinite,
            "note": "the configured eta with the replicas' gradients summed (no normalisation, no batch norm) "
                    "diverges; the FP64 oracle diverges the same way on the reduced net. Steps after that run on "
                    "non-finite values; the kernels' work and time do not depend on the values"}
    return out


# ---------------------------------------------------------------- the FP64 oracle on the host

def _oracle_sample_step(O, layers, w0, n_img, frac_update, R, opt, arch, tag):
    """One bounded sample of a training step: forward + backward of n_img images
    of one replica, and the parameter-server update of the same share
    (n_img / (R * batch)) of the parameter vector over R buffers."""
    import synth
    c, h, w = arch["input"]
    x = synth.images_nhwc(3, f"cpu{tag}", n_img, c, h, w)
    if layers[0].kind == "fc":
        x = x.reshape(n_img, -1)
    y = synth.labels(3, f"cpuy{tag}", n_img, layers[-1].cout)
    n_upd = max(1, int(round(w0.size * frac_update)))
    t0 = time.perf_counter()
    _, grads = O.gradient(layers, w0, x, y)
    g = np.asarray(grads, np.float64)[:n_upd]
    O.apply_update(w0[:n_upd], [g] * R, optimizer=opt["optimizer"], eta=opt["eta"],
                   state=O.initial_state(opt["optimizer"], n_upd))
    return time.perf_counter() - t0


def oracle_rate(cfg, budget_s):
    """Images/s of the FP64 oracle's training step on bounded samples at the
    workload's full layer sizes (forward + backward of a few images of one
    replica plus the same share of the update), over about budget_s seconds."""
    import oracle as O
    import synth
    arch = O.ARCHS[cfg["net"]]
    layers = O.build_layers(arch)
    w0 = np.concatenate([np.concatenate([synth.normal(7, f"w{i}", (int(np.prod(L.w_shape)),), O.he_std(L)),
                                         np.zeros(L.cout, np.float32)]) for i, L in enumerate(layers)]).astype(np.float64)
    opt = dict(optimizer=cfg["optimizer"], eta=cfg["eta"])
    per_step = cfg["replicas"] * cfg["batch"]
    _oracle_sample_step(O, layers, w0, 1, 1 / per_step, cfg["replicas"], opt, arch, "warm")   # page faults
    n, done, elapsed = 1, 0, 0.0
    while True:
        dt = _oracle_sample_step(O, layers, w0, n, n / per_step, cfg["replicas"], opt, arch, f"{n}.{done}")
        done += n
        elapsed += dt
        if elapsed >= budget_s or dt * 4 + elapsed > budget_s * 2:
            break
        n = min(n * 2, cfg["batch"])
    return done / elapsed, done, elapsed


def host_threads():
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def oracle_rate_one_thread(config, budget_s):
    """The same rate with the numpy BLAS limited to one thread (a child process:
    the thread count is fixed when numpy's BLAS is loaded)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               BLIS_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    try:
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-rate", config, str(budget_s)],
                           env=env, capture_output=True, text=True, timeout=budget_s * 6 + 60)
        d = json.loads(r.stdout.strip().splitlines()[-1])
        return d
    except Exception as e:   # reported, never fatal
        return {"error": str(e)[:200]}


def cpu_baseline(cfg, config_name, budget_s=10.0):
    rate, done, elapsed = oracle_rate(cfg, budget_s)
    one = oracle_rate_one_thread(config_name, budget_s * 0.6)
    return {"value": round(rate, 3), "unit": "images/s", "cores": host_threads(), "kind": "oracle",
            "sample": f"{done} images of one replica's forward + backward at full layer sizes, plus the matching "
                      f"share of the update ({elapsed:.1f} s)",
            "one_thread": ({"value": round(one["rate"], 3), "unit": "images/s", "cores": 1,
                            "sample": f"{one['images']} images ({one['seconds']:.1f} s)"} if "rate" in one else one)}


REF_IMAGES = {"tiny": 8, "smlps": 256, "vgg_c": 8, "vgg_i": 1}


def run_reference(args, cfg, config_name):
    """The reference arm: the FP64 oracle as it stands, W warm-up and K timed
    steps, each a bounded sample of the workload (a few images of one replica's
    forward + backward and the matching share of the update)."""
    import oracle as O
    import synth
    if config_name == "ps":
        return run_reference_ps(args, cfg)
    arch = O.ARCHS[cfg["net"]]
    layers = O.build_layers(arch)
    w0 = np.concatenate([np.concatenate([synth.normal(7, f"w{i}", (int(np.prod(L.w_shape)),), O.he_std(L)),
                                         np.zeros(L.cout, np.float32)]) for i, L in enumerate(layers)]).astype(np.float64)
    opt = dict(optimizer=cfg["optimizer"], eta=cfg["eta"])
    per_step = cfg["replicas"] * cfg["batch"]
    # images per sample step, fixed per workload (about 0.5-3 s of oracle work on 16
    # host cores): the oracle has a fixed cost per call (it converts and copies every
    # parameter), so an MLP sample needs many images to time the per-image work
    n = min(cfg["batch"], REF_IMAGES.get(cfg["net"], 1))
    _oracle_sample_step(O, layers, w0, 1, 1 / per_step, cfg["replicas"], opt, arch, "c0")   # page faults
    for i in range(args.warmup):
        _oracle_sample_step(O, layers, w0, n, n / per_step, cfg["replicas"], opt, arch, f"w{i}")
    times = [_oracle_sample_step(O, layers, w0, n, n / per_step, cfg["replicas"], opt, arch, f"s{i}")
             for i in range(args.steps)]
    total = float(sum(times))
    rate = n * args.steps / total
    sample = (f"each step: {n} image(s) of one replica's forward + backward at full layer sizes plus "
              f"{n}/{per_step} of the parameter-server update ({args.steps} steps, {total:.1f} s)")
    return {"impl": "reference", "metric": METRIC, "value": round(rate, 3), "unit": "images/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 1),
            "images_per_step": n, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": cfg["desc"], "global_batch": per_step,
                                            "replicas_per_gpu": cfg["replicas"], "parallelism": "host cores"},
            "cpu_baseline": {"value": round(rate, 3), "unit": "images/s", "cores": host_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(rate, 3), "unit": "images/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------- parameter-server update sweep

PS_SIZES = (1_000_000, 16_000_000, 138_000_000)
PS_KS = (1, 2, 4, 8, 16)
PS_OPTS = ("sgd", "momentum", "adagrad")


def ps_bytes(opt, k, n):
    """Algorithmic bytes of one apply: k buffers and W read, W' written, plus the
    optimizer state read and written (momentum's v, Adagrad's G)."""
    return (4.0 * k + 8.0 + (8.0 if opt != "sgd" else 0.0)) * n


def run_ps(args, world, rank, local_rank):
    """Times sprint_apply_update over the sweep: W ~ N(0, 0.01^2), buffers ~ N(0,
    1e-6), per point W warm-up and K timed launches, each timed alone (events on
    the launching stream) after a 256 MB write that evicts L2."""
    import torch

    from stale_weight_sgd_gb300 import sprint as S
    S.lib()
    torch.cuda.set_device(local_rank)
    st = torch.cuda.Stream()
    torch.cuda.set_stream(st)
    g = torch.Generator(device="cuda")
    g.manual_seed(17 + rank)
    nmax, kmax = max(PS_SIZES), max(PS_KS)
    W = torch.randn(nmax, generator=g, device="cuda") * 0.01
    Wout = torch.empty(nmax, device="cuda")
    bufs = [torch.randn(nmax, generator=g, device="cuda") * 1e-3 for _ in range(kmax)]
    state = torch.empty(nmax, device="cuda")
    flush = torch.empty(64 * 1024 * 1024, device="cuda")   # 256 MB > L2
    hp = {"sgd": 0.0, "momentum": 0.9, "adagrad": 1e-8}
    peaks, src = load_peaks()
    points = []
    barrier(world)
    clocks = ClockSampler(local_rank)
    clocks.start()
    launches0 = S.sprint_launch_count()
    tot_bytes, tot_ms = 0.0, 0.0
    for n in PS_SIZES:
        for k in PS_KS:
            for opt in PS_OPTS:
                state[:n].fill_(0.1 if opt == "adagrad" else 0.0)
                ms_l = []
                for i in range(args.warmup + args.steps):
                    flush.zero_()
                    a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(st)
                    S.sprint_apply_update(opt, W, Wout, state if opt != "sgd" else None, bufs[:k], n, 0.01, hp[opt],
                                          0.0, st)
                    e.record(st)
                    if i >= args.warmup:
                        ms_l.append((a, e))
                torch.cuda.synchronize()
                ms = float(np.mean([a.elapsed_time(e) for a, e in ms_l]))
                b = ps_bytes(opt, k, n)
                gbs = b / (ms / 1e3) / 1e9
                tot_bytes += b * args.steps
                tot_ms += ms * args.steps
                points.append({"n": n, "k": k, "opt": opt, "ms": round(ms, 4), "GB/s": round(gbs, 1),
                               "frac_hbm": round(gbs / peaks["hbm_gbs"], 4)})
    clk = clocks.stop()
    launches = S.sprint_launch_count() - launches0
    big = [p for p in points if p["n"] >= 16_000_000]
    value = tot_bytes / (tot_ms / 1e3) / 1e9
    return {"metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(tot_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded N(0,0.01^2) W, "
            "N(0,1e-6) buffers)",
            "config": {"workload": CONFIGS["ps"]["desc"], "l2": "a 256 MB write evicts L2 before every timed launch",
                       "value": "all points' algorithmic bytes over their summed launch times"},
            "roofline": {"bound": "hbm", "achieved": round(value, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(value / peaks["hbm_gbs"], 4), "traffic": None,
                         "kernel": "update_kernel (all points)", "peak_source": f"{src}: hbm copy",
                         "frac_min_n_ge_16M": min(p["frac_hbm"] for p in big),
                         "frac_median_n_ge_16M": float(np.median([p["frac_hbm"] for p in big]))},
            "sweep": points, "gpu_launches": int(launches), "clocks": clk}


def run_reference_ps(args, cfg):
    """The reference arm of the update sweep: the oracle's SGD apply over k = 4
    buffers on a 1M-element sample, W warm-up and K timed steps."""
    import oracle as O
    n, k = 1_000_000, 4
    rng = np.random.default_rng(3)
    w = rng.normal(0, 0.01, n)
    bufs = [rng.normal(0, 1e-3, n) for _ in range(k)]
    for _ in range(args.warmup):
        O.apply_update(w, bufs, optimizer="sgd", eta=0.01)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        O.apply_update(w, bufs, optimizer="sgd", eta=0.01)
    dt = time.perf_counter() - t0
    gbs = ps_bytes("sgd", k, n) * args.steps / dt / 1e9
    return {"impl": "reference", "metric": METRIC, "value": round(gbs, 3), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg["desc"]},
            "cpu_baseline": {"value": round(gbs, 3), "unit": "GB/s", "cores": host_threads(), "kind": "oracle",
                             "sample": f"SGD apply, n = 1M, k = 4 (of the sweep), {args.steps} steps"},
            "e2e": {"value": round(gbs, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


KERNELS = {
    # name: description; every case holds well under a few GB on the device
    "fc_fwd": "FC forward GEMM of an SMLPs hidden layer, 512 x 5000 x 5000 (TF32)",
    "fc_bwd": "FC backward (dX + dW + db) of an SMLPs hidden layer, 512 x 5000 x 5000, with w^T given",
    "conv_fwd": "conv forward, VGG conv3_2 shape 56x56x256->256, batch 16 (TF32 implicit GEMM)",
    "conv_dx": "conv input gradient, VGG conv3_2 shape, batch 16",
    "conv_dw": "conv weight gradient, VGG conv3_2 shape, batch 16",
    "conv_dw_xT": "conv weight gradient with the x^T copy made ahead (as the training step calls it, "
                  "sprint_conv_dW_xT), VGG conv3_2 shape, batch 16 (use --batch 64 for the blocked copies)",
    "fc_fwd_grouped": "grouped FC forward of the SMLPs hidden layer over 4 replicas, 4 x 512 x 5000 x 5000 (TF32), "
                      "with bias and the transposed output copy, as in the step",
    "fc_bwd_grouped": "grouped FC backward (dX + dW + db) of the SMLPs hidden layer over 4 replicas, with w^T, "
                      "x^T + ones row, dy^T given and dx^T written, as in the step",
    "conv_dw_224x64": "conv weight gradient, VGG conv1_2 shape 224x224x64->64, batch 16",
    "conv_dw_224x64_xT": "conv weight gradient with the x^T copy made ahead (sprint_conv_dW_xT), VGG conv1_2 "
                         "shape 224x224x64->64, batch 16 (use --batch 64)",
    "conv_fwd_224x64": "conv forward, VGG conv1_2 shape 224x224x64->64, batch 16",
    "conv_dx_224x64": "conv input gradient (ReLU mask), VGG conv1_2 shape 224x224x64->64, batch 16",
    "conv_fwd_224x3": "conv forward, VGG conv1_1 shape 224x224x3->64, batch 16",
    "conv_dw_224x3": "conv weight gradient + bias gradient, VGG conv1_1 shape 224x224x3->64, batch 16 "
                     "(direct CUDA-core kernel)",
    "update_sgd": "parameter-server SGD apply, n = 16M, k = 16 buffers",
    "update_momentum": "parameter-server momentum apply, n = 16M, k = 4 buffers",
    "update_nesterov_wd": "parameter-server Nesterov apply with weight decay, n = 16M, k = 4 buffers",
    "update_t_sgd": "parameter-server SGD apply writing W' and W'^T, 5000 x 5000 (+ bias), k = 4 buffers",
    "pool_fwd": "2x2 max-pool forward with argmax, VGG-I pool1 64x224x224x64 -> 112x112",
    "pool_bwd": "max-pool backward routed by argmax with the ReLU mask, VGG-I pool1 shape",
    "softmax_xent": "softmax cross-entropy (loss + dlogits) of 8 replicas x 64 x 1000 classes",
    "conv_xT": "the weight gradient's blocked copy x -> [H][W*N/32][C][32] (sprint_conv_xT), VGG conv3_2 input "
               "56x56x256, batch 16 (use --batch 64, --conv-shape)",
    "transpose": "2-D transpose [16*56*56][256] -> [256][16*56*56] (the bytes of one conv weight-gradient operand "
                 "re-layout at the VGG conv3_2 shape, batch 16)",
}


def run_kernel(args):
    """Times one hot kernel at a workload shape with CUDA events (on the
    launching stream), after warm-up; prints one JSON line."""
    import torch

    from stale_weight_sgd_gb300 import sprint as S
    S.lib()
    torch.cuda.set_device(0)
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    rnd = lambda *shape, std=1.0: torch.randn(shape, generator=g, device="cuda") * std
    k = args.kernel
    peaks, src = load_peaks()
    if k.endswith("_grouped"):
        M, K, N, G = 512, 5000, 5000, 4
        x = [rnd(M, K).relu_() for _ in range(G)]
        w = [[rnd(N, K, std=0.02) for _ in range(G)] for _ in range(2)]   # two sets: > L2 between launches
        wT = [[t.t().contiguous() for t in ws_] for ws_ in w]
        y = [torch.empty(M, N, device="cuda") for _ in range(G)]
        dy = [rnd(M, N) for _ in range(G)]
        dx = [torch.empty(M, K, device="cuda") for _ in range(G)]
        dw = [torch.empty(N, K, device="cuda") for _ in range(G)]
        db = [torch.empty(N, device="cuda") for _ in range(G)]
        # the calls as the training step makes them: bias, transposed copies (y^T, dx^T),
        # x^T with its row of ones (db from the weight-gradient GEMM), dy^T given
        b = [rnd(N, std=0.1) for _ in range(G)]
        yT = [torch.empty(N + 1, M, device="cuda") for _ in range(G)]
        xT1 = [torch.cat([t.t(), torch.ones(1, M, device="cuda")]).contiguous() for t in x]
        dyT = [t.t().contiguous() for t in dy]
        dxT = [torch.empty(K, M, device="cuda") for _ in range(G)]
        nb = S.sprint_fc_batched_workspace_size(G, M, K, N, 1)
        ws = torch.empty(nb // 4 + 64, device="cuda")
        if k == "fc_fwd_grouped":
            fn = lambda i: S.sprint_fc_fwd_batched(x, w[i % 2], b, y, M, K, N, 1, ws, nb, yT=yT)
            work = 2.0 * M * N * K * G
        else:
            fn = lambda i: S.sprint_fc_bwd_batched(x, w[i % 2], wT[i % 2], dy, x, dx, dw, db, 1.0, 0, M, K, N, ws, nb,
                                                   xT1=xT1, dyT=dyT, dxT=dxT)
            work = 4.0 * M * N * K * G
        unit = "TFLOP/s"
    elif k.startswith("fc"):
        M, K, N = 512, 5000, 5000
        x = rnd(M, K).relu_()
        w = [rnd(N, K, std=0.02) for _ in range(2)]     # two weight matrices: > L2 between launches
        wT = [t.t().contiguous() for t in w]
        y = torch.empty(M, N, device="cuda")
        dy = rnd(M, N)
        dx = torch.empty(M, K, device="cuda")
        dw = torch.empty(N, K, device="cuda")
        db = torch.empty(N, device="cuda")
        nb = S.sprint_fc_workspace_size(M, K, N, 1)
        ws = torch.empty(nb // 4 + 64, device="cuda")
        if k == "fc_fwd":
            fn = lambda i: S.sprint_fc_fwd(x, w[i % 2], None, y, M, K, N, 1)
            work, unit = 2.0 * M * N * K, "TFLOP/s"
        else:
            fn = lambda i: S.sprint_fc_bwd(x, w[i % 2], wT[i % 2], dy, x, dx, dw, db, 1.0, 0, M, K, N, ws, nb)
            work, unit = 4.0 * M * N * K, "TFLOP/s"
    elif k in ("conv_dw_224x64", "conv_dw_224x64_xT", "conv_fwd_224x64", "conv_dx_224x64", "conv_fwd_224x3",
               "conv_dw_224x3"):
        Nb, H, W = args.batch or 16, 224, 224
        Ci = 64 if "224x64" in k else 3
        Co = 64
        x = rnd(Nb, H, W, Ci).relu_()
        w = rnd(Co, 3, 3, Ci, std=(2.0 / (9 * Ci)) ** 0.5)
        b = torch.zeros(Co, device="cuda")
        y = torch.empty(Nb, H, W, Co, device="cuda")
        dy = rnd(Nb, H, W, Co)
        nbytes = max(S.sprint_conv_workspace_size(op, Nb, H, W, Ci, Co, 1) for op in range(3))
        ws = torch.empty(nbytes // 4 + 64, device="cuda")
        dwt = torch.empty(Co, 3, 3, Ci, device="cuda")
        dbt = torch.empty(Co, device="cuda")
        work, unit = 2.0 * Nb * H * W * Co * 9 * Ci, "TFLOP/s"
        if k in ("conv_dw_224x64", "conv_dw_224x3"):
            fn = lambda i: S.sprint_conv_dW(x, dy, dwt, dbt, 1.0, 0, Nb, H, W, Ci, Co, 1, ws, nbytes)
        elif k == "conv_dw_224x64_xT":
            xT = torch.empty(max(S.sprint_conv_xT_size(Nb, H, W, Ci, Co, 1) // 4, 1), device="cuda")
            S.sprint_conv_xT(x, xT, Nb, H, W, Ci, Co, 1)
            fn = lambda i: S.sprint_conv_dW_xT(x, xT, dy, dwt, dbt, 1.0, 0, Nb, H, W, Ci, Co, 1, ws, nbytes)
        elif k == "conv_dx_224x64":
            dx = torch.empty(Nb, H, W, Ci, device="cuda")
            fn = lambda i: S.sprint_conv_dX(dy, w, None, x, dx, Nb, H, W, Ci, Co, 1, ws, nbytes)
        else:
            fn = lambda i: S.sprint_conv_fwd(x, w, b, y, Nb, H, W, Ci, Co, 1, 1, ws, nbytes)
    elif k.startswith("conv"):
        Nb = args.batch or 16
        H, W, Ci, Co = (int(v) for v in args.conv_shape.split(",")) if args.conv_shape else (56, 56, 256, 256)
        x = rnd(Nb, H, W, Ci).relu_()
        w = rnd(Co, 3, 3, Ci, std=(2.0 / (9 * Ci)) ** 0.5)
        wT = w.reshape(Co, 9 * Ci).t().contiguous()
        b = torch.zeros(Co, device="cuda")
        y = torch.empty(Nb, H, W, Co, device="cuda")
        dx = torch.empty(Nb, H, W, Ci, device="cuda")
        dy = rnd(Nb, H, W, Co)
        nbytes = max(S.sprint_conv_workspace_size(op, Nb, H, W, Ci, Co, 1) for op in range(3))
        ws = torch.empty(nbytes // 4 + 64, device="cuda")
        dwt = torch.empty(Co, 3, 3, Ci, device="cuda")
        dbt = torch.empty(Co, device="cuda")
        work, unit = 2.0 * Nb * H * W * Co * 9 * Ci, "TFLOP/s"
        if k == "conv_xT":   # reads x, writes its blocked copy
            xT = torch.empty(max(S.sprint_conv_xT_size(Nb, H, W, Ci, Co, 1) // 4, 1), device="cuda")
            fn = lambda i: S.sprint_conv_xT(x, xT, Nb, H, W, Ci, Co, 1)
            work, unit = 8.0 * Nb * H * W * Ci, "GB/s"
        elif k == "conv_fwd":
            fn = lambda i: S.sprint_conv_fwd(x, w, b, y, Nb, H, W, Ci, Co, 1, 1, ws, nbytes)
        elif k == "conv_dx":
            fn = lambda i: S.sprint_conv_dX(dy, w, wT, x, dx, Nb, H, W, Ci, Co, 1, ws, nbytes)
        elif k == "conv_dw_xT":
            xT = torch.empty(max(S.sprint_conv_xT_size(Nb, H, W, Ci, Co, 1) // 4, 1), device="cuda")
            S.sprint_conv_xT(x, xT, Nb, H, W, Ci, Co, 1)
            fn = lambda i: S.sprint_conv_dW_xT(x, xT, dy, dwt, dbt, 1.0, 0, Nb, H, W, Ci, Co, 1, ws, nbytes)
        else:
            fn = lambda i: S.sprint_conv_dW(x, dy, dwt, dbt, 1.0, 0, Nb, H, W, Ci, Co, 1, ws, nbytes)
    elif k in ("pool_fwd", "pool_bwd"):
        Nb, H, W, C = 64, 224, 224, 64
        x = rnd(Nb, H, W, C).relu_()
        y = torch.empty(Nb, H // 2, W // 2, C, device="cuda")
        arg = torch.empty(Nb, H // 2, W // 2, C, dtype=torch.uint8, device="cuda")
        S.sprint_pool_fwd(x, y, arg, Nb, H, W, C)
        big, small = 4.0 * Nb * H * W * C, 4.0 * Nb * (H // 2) * (W // 2) * C
        if k == "pool_fwd":   # reads x, writes y and the uint8 argmax
            fn = lambda i: S.sprint_pool_fwd(x, y, arg, Nb, H, W, C)
            work = big + small + small / 4
        else:                 # reads dy, argmax and the pooled output (ReLU mask), writes dx
            dy = rnd(Nb, H // 2, W // 2, C)
            dx = torch.empty_like(x)
            fn = lambda i: S.sprint_pool_bwd(dy, arg, y, dx, Nb, H, W, C)
            work = big + 2 * small + small / 4
        unit = "GB/s"
    elif k == "softmax_xent":
        R, Nb, C = 8, 64, 1000
        z = [rnd(Nb, C) for _ in range(R)]
        lab = [torch.randint(0, C, (Nb,), generator=g, device="cuda", dtype=torch.int32) for _ in range(R)]
        loss = [torch.empty(4, device="cuda") for _ in range(R)]
        dz = [torch.empty(Nb, C, device="cuda") for _ in range(R)]
        fn = lambda i: S.sprint_softmax_xent_batched(z, lab, loss, dz, Nb, C)
        work = R * (8.0 * Nb * C + 4.0 * Nb)
        unit = "GB/s"
    elif k == "transpose":
        rows, cols = 16 * 56 * 56, 256
        srcs = [rnd(rows, cols) for _ in range(2)]     # two sources: > L2 between launches
        dst = torch.empty(cols, rows, device="cuda")
        fn = lambda i: S.sprint_transpose(srcs[i % 2], dst, rows, cols)
        work = 8.0 * rows * cols
        unit = "GB/s"
    else:
        n = 16_000_000
        kb = 16 if k == "update_sgd" else 4
        wv = rnd(n, std=0.01)
        bufs = [rnd(n, std=1e-3) for _ in range(kb)]
        st = torch.zeros(n, device="cuda")
        if k == "update_sgd":
            fn = lambda i: S.sprint_apply_update_sgd(wv, wv, bufs, n, 0.01)
            work = (4.0 * kb + 8) * n
        elif k == "update_momentum":
            fn = lambda i: S.sprint_apply_update_momentum(wv, wv, st, bufs, n, 0.01, 0.9)
            work = (4.0 * kb + 16) * n
        elif k == "update_nesterov_wd":
            fn = lambda i: S.sprint_apply_update("nesterov", wv, wv, st, bufs, n, 0.01, 0.9, 5e-4)
            work = (4.0 * kb + 16) * n
        else:   # update_t_sgd: reads k buffers and W, writes W' and W'^T
            rows, cols = 5000, 5000
            n = rows * cols + rows
            wv = rnd(n, std=0.01)
            bufs = [rnd(n, std=1e-3) for _ in range(kb)]
            wo = torch.empty(n, device="cuda")
            wT = torch.empty(rows * cols, device="cuda")
            fn = lambda i: S.sprint_apply_update_t("sgd", wv, wo, wT, None, bufs, rows, cols, 0.01, n_total=n)
            work = (4.0 * kb + 8) * n + 4.0 * rows * cols
        unit = "GB/s"
    for i in range(args.warmup):
        fn(i)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    a.record()
    for i in range(args.steps):
        fn(i)
    e.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(e) / args.steps
    achieved = work / (ms / 1e3) / (1e12 if unit == "TFLOP/s" else 1e9)
    if unit == "TFLOP/s":
        peak = peaks["bf16_tflops"] * TF32_OVER_BF16
        psrc = f"{src}: bf16 burst x 1.1/2.25"
    else:
        peak = peaks["hbm_gbs"]
        psrc = f"{src}: hbm copy"
    shape = f" (shape {args.conv_shape})" if args.conv_shape and k.startswith("conv") else ""
    print(json.dumps({"kernel": k, "workload": KERNELS[k] + (f" (batch {args.batch})" if args.batch else "") + shape,
                      "ms": round(ms, 4), "achieved": round(achieved, 1),
                      "unit": unit, "peak": round(peak, 1), "frac": round(achieved / peak, 4), "peak_source": psrc,
                      "flags": S.sprint_device_status()}))
    return 0


def init_dist(world, local_rank):
    """One process per GPU (NCCL); on a machine without GPUs the same host
    logic runs over gloo (the multi-process CPU tests)."""
    if world <= 1:
        return
    import torch
    import torch.distributed as dist
    if torch.cuda.is_available():
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    else:
        dist.init_process_group("gloo")


def weak_scaling_value(imgs_per_rank, seconds_local, world):
    """Replicas-only scaling: every rank runs the whole workload; the job's
    images/s are all ranks' images over the slowest rank's time."""
    s_max = allreduce_max(seconds_local, world)
    return imgs_per_rank * world / s_max, s_max


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(v, world):
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64, device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_cost_model(args):
    """Refits the SPRINT report's SGEMM cost model (Eq. (6), per role) to this
    library's calls on one GPU and checks its prediction of a replica's
    forward + backward time (Eq. (4)); evaluates Eq. (9) / (10) for the
    SMLPs workload with the measured update time. Prints one JSON line."""
    import torch

    from stale_weight_sgd_gb300 import costmodel as C
    from stale_weight_sgd_gb300 import model
    from stale_weight_sgd_gb300 import sprint as S
    S.lib()
    torch.cuda.set_device(0)
    st = torch.cuda.Stream()
    torch.cuda.set_stream(st)
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    rnd = lambda *shape, std=1.0: torch.randn(shape, generator=g, device="cuda") * std

    def timed(fn, reps=8):
        for _ in range(2):
            fn()
        a, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        for _ in range(reps):
            fn()
        e.record(st)
        torch.cuda.synchronize()
        return a.elapsed_time(e) / reps / 1e3

    samples = {r: [] for r in C.ROLES}
    measured = {}   # (net, N) -> sum of the measured per-layer call times (a replica's forward + backward GEMMs)
    sweeps = (("smlps", (64, 128, 256, 512, 1024)), ("vgg_c", (8, 16, 32, 64, 128)))
    for name, Ns in sweeps:
        shapes = model.layer_shapes(model.NETWORKS[name])
        for N in Ns:
            total = 0.0
            for i, L in enumerate(shapes):
                dims = C.role_dims(L, N, i == 0)
                if L.kind == "fc":
                    x, w, b = rnd(N, L.cin).relu_(), rnd(L.cout, L.cin, std=0.02), rnd(L.cout)
                    wT, y, dy = w.t().contiguous(), torch.empty(N, L.cout, device="cuda"), rnd(N, L.cout)
                    dx, dw, db = torch.empty(N, L.cin, device="cuda"), torch.empty_like(w), torch.empty_like(b)
                    nb = S.sprint_fc_workspace_size(N, L.cin, L.cout, 1)
                    ws = torch.empty(nb // 4 + 64, device="cuda")
                    t_f = timed(lambda: S.sprint_fc_fwd(x, w, b, y, N, L.cin, L.cout, 1, st.cuda_stream))
                    t_w = timed(lambda: S.sprint_fc_bwd(x, w, wT, dy, None, None, dw, db, 1.0, 0, N, L.cin, L.cout,
                                                        ws, nb, st.cuda_stream))
                    samples["fc"].append((*dims["fc"], t_f))
                    samples["dedw"].append((*dims["dedw"], t_w))
                    total += t_f + t_w
                    if i > 0:
                        t_b = timed(lambda: S.sprint_fc_bwd(x, w, wT, dy, x, dx, dw, db, 1.0, 0, N, L.cin, L.cout,
                                                            ws, nb, st.cuda_stream))
                        samples["dedx_fc"].append((*dims["dedx_fc"], max(t_b - t_w, 0.0)))
                        total += max(t_b - t_w, 0.0)
                else:
                    x = rnd(N, L.h, L.w, L.cin).relu_()
                    w, b = rnd(L.cout, 3, 3, L.cin, std=0.05), rnd(L.cout)
                    wT = w.reshape(L.cout, -1).t().contiguous()
                    y, dy = torch.empty(N, L.h, L.w, L.cout, device="cuda"), rnd(N, L.h, L.w, L.cout)
                    dx, dw, db = torch.empty_like(x), torch.empty_like(w), torch.empty_like(b)
                    nb = max(S.sprint_conv_workspace_size(op, N, L.h, L.w, L.cin, L.cout, 1)
                             for op in (S.SPRINT_CONV_FWD, S.SPRINT_CONV_DX, S.SPRINT_CONV_DW))
                    ws = torch.empty(nb // 4 + 64, device="cuda")
                    t_f = timed(lambda: S.sprint_conv_fwd(x, w, b, y, N, L.h, L.w, L.cin, L.cout, 1, 1, ws, nb,
                                                          st.cuda_stream))
                    t_w = timed(lambda: S.sprint_conv_dW(x, dy, dw, db, 1.0, 0, N, L.h, L.w, L.cin, L.cout, 1, ws, nb,
                                                         st.cuda_stream))
                    samples["convolution"].append((*dims["convolution"], t_f))
                    samples["dedw"].append((*dims["dedw"], t_w))
                    total += t_f + t_w
                    if i > 0:
                        t_x = timed(lambda: S.sprint_conv_dX(dy, w, wT, x, dx, N, L.h, L.w, L.cin, L.cout, 1, ws, nb,
                                                             st.cuda_stream))
                        samples["dedx_conv"].append((*dims["dedx_conv"], t_x))
                        total += t_x
            measured[(name, N)] = total
    coefs = {r: C.fit_role(samples[r]) for r in C.ROLES}
    fit = {}
    for r in C.ROLES:
        y = np.array([t for *_, t in samples[r]])
        p = np.array([C.predict(coefs[r], m, n, k) for m, n, k, _ in samples[r]])
        fit[r] = {"samples": len(y), "max_rel_err": round(float(np.max(np.abs(p - y) / y)), 4),
                  "r2": round(float(1 - np.sum((p - y) ** 2) / np.sum((y - y.mean()) ** 2)), 5),
                  "coef": [float(f"{c:.4e}") for c in coefs[r]]}
    pred = {}
    for (name, N), t in measured.items():
        tp = C.predict_t_gpu(model.layer_shapes(model.NETWORKS[name]), N, coefs)
        pred[f"{name}@{N}"] = {"measured_ms": round(t * 1e3, 4), "predicted_ms": round(tp * 1e3, 4),
                               "rel_err": round(abs(tp - t) / t, 4)}
    # Eq. (9) / (10) for the SMLPs workload: 4 replicas on one GPU (N_Node = 1, N_GPU = 4),
    # N_Subbatch = 512, T_GPU from the model, T_Update = the measured update of all layers
    shapes = model.layer_shapes(model.NETWORKS["smlps"])
    n = model.padded_size(shapes)
    wv = rnd(n, std=0.01)
    bufs = [rnd(n, std=1e-3) for _ in range(4)]
    t_update = timed(lambda: S.sprint_apply_update_sgd(wv, wv, bufs, n, 0.01, st.cuda_stream))
    t_gpu = C.predict_t_gpu(shapes, 512, coefs)
    nmb = C.n_minibatch_avg(1, 4, 512, t_update, t_gpu)
    out = {"cost_model": "SPRINT Eq. (6) per SGEMM role, refitted on this GPU", "fit": fit, "t_gpu": pred,
           "smlps_eq9": {"t_update_ms": round(t_update * 1e3, 4), "t_gpu_ms": round(t_gpu * 1e3, 4),
                         "n_minibatch_avg": round(nmb, 2),
                         "t_epoch_s_cifar10": round(C.t_epoch(50000, t_update, nmb), 4)}}
    print(json.dumps(out))
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=sorted(CONFIGS), default=DEFAULT_CONFIG)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-breakdown", action="store_true", help="skip the serial per-role breakdown step")
    ap.add_argument("--serial", action="store_true",
                    help="issue everything on one stream (no update overlap, no side-by-side replica convolutions)")
    ap.add_argument("--kernel", choices=sorted(KERNELS), default=None,
                    help="time one hot kernel at a workload shape instead of the training step")
    ap.add_argument("--batch", type=int, default=None,
                    help="--kernel conv_*: batch size in place of the case's 16")
    ap.add_argument("--conv-shape", default=None, metavar="H,W,CIN,COUT",
                    help="--kernel conv_fwd / conv_dx / conv_dw / conv_dw_xT: layer shape in place of 56,56,256,256")
    ap.add_argument("--cost-model", action="store_true",
                    help="refit the SPRINT report's SGEMM cost model to this GPU and check its T_GPU prediction")
    ap.add_argument("--oracle-rate", nargs=2, metavar=("CONFIG", "SECONDS"), default=None,
                    help=argparse.SUPPRESS)   # child process of the one-thread oracle timing
    args = ap.parse_args(argv)
    if args.oracle_rate:
        rate, done, elapsed = oracle_rate(CONFIGS[args.oracle_rate[0]], float(args.oracle_rate[1]))
        print(json.dumps({"rate": rate, "images": done, "seconds": elapsed}))
        return 0
    if args.kernel:
        return run_kernel(args)
    if args.cost_model:
        return run_cost_model(args)
    cfg = CONFIGS[args.config]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, cfg, args.config)))
        return 0

    init_dist(world, local_rank)
    if args.config == "ps":
        out = run_ps(args, world, rank, local_rank)
    else:
        out = run_ours(args, cfg, rank, world, local_rank)
        if rank == 0 and not args.no_cpu_baseline:
            out["cpu_baseline"] = cpu_baseline(cfg, args.config)
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
