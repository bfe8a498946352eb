"""Stale-weight SGD on one GPU: the worker step of every logical replica,
then the parameter-server update, all through libsprint's C ABI.

Asynchrony is simulated deterministically (SPRINT report, IPSJ SIG Technical
Report Vol.2016-HPC-155 No.8, Sec. 1 / Fig. 1 and Algorithms 1-2; DistBelief
blog summary: replicas fetch w, push dw, the server applies w' := w - eta*dw):

  * weight versions live in a device ring of S+1 slots; W(t), the version
    before step t's update, is slot t mod (S+1). The update reads slot t and
    writes slot t+1 out of place, so no version is ever copied;
  * replica r at step t computes its gradient on W(max(0, t - s[t, r])) with
    s from the seeded SplitMix64 schedule (sprint_staleness_schedule), or —
    for a pipeline ("Pipelined training of deep CNNs with stale weights",
    Sec. 4.1) — layer l of stage k uses W_l(max(0, t - s_k)) in both its
    forward and backward pass;
  * each replica writes its raw gradient into its own GradBuf (Algorithm 1:
    assign when empty), fused into the dW/db GEMM epilogues;
  * the input-gradient GEMMs read transposed weights (the TF32 tensor-core
    MMA takes k-contiguous operands only): a second ring holds W^T of every
    version, written once when the version is created and shared by every
    replica that reads that version;
  * the update sums the R GradBufs in replica order and applies SGD, momentum
    or Adagrad (Algorithm 2; one fused kernel).

Replica r draws batch (t*R + r) mod P from a pool of P device-resident
batches. Replicas run on their own CUDA streams (independent work that fills
the GPU together); the update of step t waits for all of them. A replica of
step t waits only for the newest weight version it reads (so a replica with
delay >= 1 need not wait for update t-1) and for update t-2, the last reader
of its GradBuf set: GradBufs are double-buffered by step parity. Nothing here
computes: every operation is a libsprint call.
"""
from __future__ import annotations

import numpy as np
import torch

from . import sprint as S
from .model import layer_shapes, pack, padded_size, unpack


class StaleSGD:
    def __init__(self, net, batch, *, replicas=1, max_delay=0, schedule_seed=0, stage_of_layer=None,
                 stage_delays=None, optimizer="sgd", eta=0.01, nu=0.9, eps=1e-8, g0=0.1, concurrent=True,
                 device="cuda"):
        S.lib()  # fail loudly if the CUDA library is missing
        self.net = net
        self.shapes = layer_shapes(net)
        self.n = padded_size(self.shapes)
        self.N = int(batch)
        self.R = int(replicas)
        self.pipeline = stage_delays is not None
        if self.pipeline:
            assert stage_of_layer is not None and len(stage_of_layer) == len(self.shapes)
            self.stage_of_layer = list(stage_of_layer)
            self.stage_delays = [int(s) for s in stage_delays]
            self.S = max(self.stage_delays)
        else:
            self.S = int(max_delay)
        self.seed = int(schedule_seed)
        self.optimizer = optimizer
        self.eta, self.nu, self.eps, self.g0 = float(eta), float(nu), float(eps), float(g0)
        self.dev = torch.device(device)
        f32 = dict(dtype=torch.float32, device=self.dev)

        self.ring = torch.zeros((self.S + 1, self.n), **f32)
        self.ringT = torch.zeros((self.S + 1, self.n), **f32)   # W^T of every layer that needs dX
        self.gradbuf_sets = torch.zeros((2, self.R, self.n), **f32)   # step t writes set t % 2
        self.gradbuf = self.gradbuf_sets[0]
        if optimizer == "momentum":
            self.opt_state = torch.zeros(self.n, **f32)
        elif optimizer == "adagrad":
            self.opt_state = torch.full((self.n,), self.g0, **f32)
        elif optimizer == "sgd":
            self.opt_state = None
        else:
            raise ValueError(optimizer)
        self.loss = torch.zeros((self.R, 4), **f32)  # row r, column 0 = replica r's loss

        # per-replica activations, saved for the backward pass
        self.acts = [self._alloc_acts() for _ in range(self.R)]
        self.classes = self.shapes[-1].cout

        main = torch.cuda.current_stream(self.dev)
        self.main_stream = main
        self.streams = [torch.cuda.Stream(self.dev) for _ in range(self.R)] if concurrent else [main] * self.R
        self.ev_update = torch.cuda.Event()      # the latest update has finished
        self.ev_done = [torch.cuda.Event() for _ in range(self.R)]
        self.ev_ver = [torch.cuda.Event() for _ in range(self.S + 3)]  # version v exists: ev_ver[v % (S+3)]
        self.ev_update.record(main)
        self.ev_ver[0].record(main)
        self.ev_inputs = torch.cuda.Event()
        self.inputs_pending = False
        self._sched = np.zeros((0, self.R), np.int32)
        self.batches_x = None
        self.batches_y = None
        self.t = 0

    # ------------------------------------------------------------------ buffers
    def _alloc_acts(self):
        f32 = dict(dtype=torch.float32, device=self.dev)
        outs, pooled, argmax = [], [], []
        big = 0       # largest activation / gradient tensor (elements)
        ws_bytes = 0  # largest workspace any call of this replica needs
        for L in self.shapes:
            if L.kind == "conv":
                numel = self.N * L.h * L.w * L.cout
                big = max(big, numel, self.N * L.h * L.w * L.cin)
                outs.append(torch.empty(numel, **f32))
                if L.pool:
                    ph, pw = L.out_hw
                    pooled.append(torch.empty(self.N * ph * pw * L.cout, **f32))
                    argmax.append(torch.empty(self.N * ph * pw * L.cout, dtype=torch.uint8, device=self.dev))
                else:
                    pooled.append(None)
                    argmax.append(None)
                for op in (S.SPRINT_CONV_FWD, S.SPRINT_CONV_DX, S.SPRINT_CONV_DW):
                    ws_bytes = max(ws_bytes, S.sprint_conv_workspace_size(op, self.N, L.h, L.w, L.cin, L.cout, 1))
            else:
                numel = self.N * L.cout
                big = max(big, numel, self.N * L.cin)
                outs.append(torch.empty(numel, **f32))
                pooled.append(None)
                argmax.append(None)
                ws_bytes = max(ws_bytes, S.sprint_fc_workspace_size(self.N, L.cin, L.cout, 1))
        g = [torch.empty(big, **f32), torch.empty(big, **f32)]
        ws = torch.empty(max(ws_bytes // 4 + 64, 64), **f32)
        return dict(outs=outs, pooled=pooled, argmax=argmax, g=g, ws=ws, ws_bytes=ws.numel() * 4)

    # ------------------------------------------------------------------ data / weights
    def load_weights(self, dense: np.ndarray):
        """Sets W(0) from a dense [W0 b0 W1 b1 ...] fp32 vector."""
        w = torch.from_numpy(pack(self.shapes, np.asarray(dense, np.float32)))
        self.ring[0].copy_(w.to(self.dev))
        self._transpose_slot(0, self.main_stream)
        if self.optimizer == "momentum":
            self.opt_state.zero_()
        elif self.optimizer == "adagrad":
            self.opt_state.fill_(self.g0)
        self.t = 0
        torch.cuda.synchronize(self.dev)
        self.ev_update.record(self.main_stream)
        self.ev_ver[0].record(self.main_stream)

    def load_batches(self, batches):
        """Uploads the pool of (x, labels) batches; x is NHWC (or [N][features])."""
        xs = np.stack([np.asarray(x, np.float32).reshape(self.N, -1) for x, _ in batches])
        ys = np.stack([np.asarray(y, np.int32).reshape(self.N) for _, y in batches])
        self.batches_x = torch.from_numpy(xs).to(self.dev)
        self.batches_y = torch.from_numpy(ys).to(self.dev)

    def set_batch_pool(self, x: torch.Tensor, y: torch.Tensor):
        """Uses device tensors [P][N][...] and [P][N] (int32) as the batch pool."""
        self.batches_x = x.reshape(x.shape[0], self.N, -1)
        self.batches_y = y

    def mark_inputs(self, stream):
        """The batch pool was (re)written on `stream`: the next step's replicas
        wait for that work before reading it."""
        self.ev_inputs.record(stream)
        self.inputs_pending = True

    def weights(self, version=None) -> np.ndarray:
        """Dense copy of W(version) (default: the current version)."""
        v = self.t if version is None else version
        torch.cuda.synchronize(self.dev)
        return unpack(self.shapes, self.ring[v % (self.S + 1)].cpu().numpy())

    def _transpose_slot(self, slot, stream):
        """W^T of every layer after the first (they need dE/dX) into ringT[slot]."""
        src = self.ring[slot].data_ptr()
        dst = self.ringT[slot].data_ptr()
        for L in self.shapes[1:]:
            rows, cols = (L.cout, 9 * L.cin) if L.kind == "conv" else (L.cout, L.cin)
            S.sprint_transpose(src + 4 * L.w_off, dst + 4 * L.w_off, rows, cols, stream.cuda_stream)

    def schedule(self, steps) -> np.ndarray:
        if self._sched.shape[0] < steps:
            n = max(steps, 2 * self._sched.shape[0], 256)
            self._sched = S.sprint_staleness_schedule(self.seed, n, self.R, self.S)
        return self._sched[:steps]

    # ------------------------------------------------------------------ one step
    def _version(self, t, r, layer):
        if self.pipeline:
            return max(0, t - self.stage_delays[self.stage_of_layer[layer]])
        s = int(self.schedule(t + 1)[t, r]) if self.S > 0 else 0
        return max(0, t - s)

    def _replica(self, t, r, stream):
        """Forward, softmax cross-entropy and backward of replica r (Algorithm 1)."""
        A = self.acts[r]
        N = self.N
        ring_ptr = self.ring.data_ptr()
        row = self.n * 4
        gb = self.gradbuf_sets[t % 2][r].data_ptr()
        bi = (t * self.R + r) % self.batches_x.shape[0]
        x = self.batches_x[bi]
        y = self.batches_y[bi]
        ringT_ptr = self.ringT.data_ptr()
        wptr, wtptr = [], []
        for li, L in enumerate(self.shapes):
            slot = self._version(t, r, li) % (self.S + 1)
            base = ring_ptr + slot * row
            wptr.append((base + 4 * L.w_off, base + 4 * L.b_off))
            wtptr.append(ringT_ptr + slot * row + 4 * L.w_off)
        ws, wsb = A["ws"], A["ws_bytes"]
        sh = stream.cuda_stream

        # forward
        inp = [None] * len(self.shapes)
        cur = x.data_ptr()
        for li, L in enumerate(self.shapes):
            inp[li] = cur
            out = A["outs"][li]
            if L.kind == "conv":
                S.sprint_conv_fwd(cur, wptr[li][0], wptr[li][1], out, N, L.h, L.w, L.cin, L.cout, 1, 1, ws, wsb, sh)
                if L.pool:
                    S.sprint_pool_fwd(out, A["pooled"][li], A["argmax"][li], N, L.h, L.w, L.cout, sh)
                    cur = A["pooled"][li].data_ptr()
                else:
                    cur = out.data_ptr()
            else:
                S.sprint_fc_fwd(cur, wptr[li][0], wptr[li][1], out, N, L.cin, L.cout, int(L.relu), sh)
                cur = out.data_ptr()
        g, h = A["g"]
        S.sprint_softmax_xent(cur, y, N, self.classes, self.loss[r], g, 0, sh)

        # backward (g holds dE/d(pre-activation output) of layer li)
        for li in range(len(self.shapes) - 1, -1, -1):
            L = self.shapes[li]
            dw, db = gb + 4 * L.w_off, gb + 4 * L.b_off
            prev = self.shapes[li - 1] if li > 0 else None
            if L.kind == "fc":
                relu_src = None
                if prev is not None and not (prev.kind == "conv" and prev.pool) and prev.relu:
                    relu_src = inp[li]
                S.sprint_fc_bwd(inp[li], wptr[li][0], wtptr[li] if prev is not None else None, g, relu_src,
                                h if prev is not None else None, dw, db, 1.0, 0, N, L.cin, L.cout, ws, wsb, sh)
            else:
                S.sprint_conv_dW(inp[li], g, dw, db, 1.0, 0, N, L.h, L.w, L.cin, L.cout, 1, ws, wsb, sh)
                if prev is not None:
                    relu_src = None if prev.pool else inp[li]
                    S.sprint_conv_dX(g, wptr[li][0], wtptr[li], relu_src, h, N, L.h, L.w, L.cin, L.cout, 1, ws, wsb,
                                     sh)
            if prev is None:
                break
            g, h = h, g
            if prev.kind == "conv" and prev.pool:
                # h (free) <- routed gradient of the pre-pool ReLU output, masked
                S.sprint_pool_bwd(g, A["argmax"][li - 1], A["pooled"][li - 1], h, N, prev.h, prev.w, prev.cout, sh)
                g, h = h, g

    def _update(self, t, stream):
        """SumGradient + UpdateWeights (Algorithm 2): W(t+1) into ring slot t+1."""
        w_in = self.ring[t % (self.S + 1)]
        w_out = self.ring[(t + 1) % (self.S + 1)]
        bufs = [self.gradbuf_sets[t % 2][r] for r in range(self.R)]
        sh = stream.cuda_stream
        if self.optimizer == "sgd":
            S.sprint_apply_update_sgd(w_in, w_out, bufs, self.n, self.eta, sh)
        elif self.optimizer == "momentum":
            S.sprint_apply_update_momentum(w_in, w_out, self.opt_state, bufs, self.n, self.eta, self.nu, sh)
        else:
            S.sprint_apply_update_adagrad(w_in, w_out, self.opt_state, bufs, self.n, self.eta, self.eps, sh)
        self._transpose_slot((t + 1) % (self.S + 1), stream)

    def step(self):
        """One global step: every replica's gradient, then one update. Asynchronous."""
        t = self.t
        L = len(self.ev_ver)
        for r in range(self.R):
            st = self.streams[r]
            newest = max(self._version(t, r, li) for li in range(len(self.shapes)))
            # the newest version this replica reads, and update t-2 (last reader of GradBuf set t % 2)
            st.wait_event(self.ev_ver[max(newest, t - 1, 0) % L])
            if self.inputs_pending:
                st.wait_event(self.ev_inputs)
            self._replica(t, r, st)
            self.ev_done[r].record(st)
        for r in range(self.R):
            self.main_stream.wait_event(self.ev_done[r])
        self._update(t, self.main_stream)
        self.ev_update.record(self.main_stream)
        self.ev_ver[(t + 1) % L].record(self.main_stream)
        self.gradbuf = self.gradbuf_sets[t % 2]   # the GradBufs of the step just issued
        self.inputs_pending = False
        self.t = t + 1

    def step_loss(self) -> float:
        """Mean over replicas of the last step's loss (synchronises)."""
        self.main_stream.synchronize()
        return float(self.loss[:, 0].mean().item())
