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
    or Adagrad (Algorithm 2; one fused kernel per layer).

Execution is layer-major: the R replicas of a layer are one batch of
problems. An FC layer is one grouped tensor-core launch for all replicas
(each problem with its own weight version); a convolution runs replica after
replica (each already fills the GPU); the softmax of all replicas is one
launch. All of it is issued on one stream. The update is split by layer: as
soon as the backward pass of layer l has finished for every replica, a second
stream applies the update of layer l (and writes its W^T) while the backward
pass of the layers below runs, so only the update of the first layer remains
between two steps. Per-layer events order everything else:
  * the forward pass of layer l at step t waits for the newest version of
    layer l that any replica reads;
  * the backward pass of layer l at step t waits for version t-1 of layer l,
    i.e. for update t-2, the last reader of GradBuf set t mod 2 (GradBufs
    are double-buffered by step parity);
  * the update of layer l at step t overwrites ring slot (t+1) mod (S+1),
    whose version t-S is read by nobody once layer l's backward pass of step
    t is done.
Replica r draws batch (t*R + r) mod P from a pool of P device-resident
batches. Nothing here computes: every operation is a libsprint call.
"""
from __future__ import annotations

import numpy as np
import torch

from . import sprint as S
from .model import layer_shapes, pack, padded_size, stale_weight_percent, staleness_degrees, unpack


def fetch_push_version(t, n_fetch, n_push):
    """DistBelief n_fetch / n_push: the server version (count of updates applied)
    a replica computes on at step t — the one of its last fetch step, t rounded
    down to a multiple of n_fetch; updates end steps n_push - 1, 2 n_push - 1, ..."""
    return (t // n_fetch * n_fetch) // n_push


def fetch_push_max_lag(n_fetch, n_push):
    """A bound on how many server updates a replica's copy can be behind the
    newest version (the versions of steps f .. f + n_fetch - 1 differ by at most
    this; not always reached)."""
    return (n_fetch - 1) // n_push + 1


class StaleSGD:
    def __init__(self, net, batch, *, replicas=1, max_delay=0, schedule_seed=0, stage_of_layer=None,
                 stage_delays=None, hybrid_switch=None, n_fetch=None, n_push=None, optimizer="sgd", eta=0.01,
                 nu=0.9, eps=1e-8, g0=0.1, weight_decay=0.0, concurrent=True, graphs="auto", lookahead="auto",
                 device="cuda"):
        """Delays: seeded per-replica delays up to max_delay (ASGD), fixed per-stage
        delays (pipeline: stage_of_layer, stage_delays; hybrid_switch = N_p turns
        them to 0 from step N_p on, "Pipelined training of deep CNNs with stale
        weights" Sec. 4.2), or DistBelief's n_fetch / n_push (every replica
        computes on the server's parameters of its last fetch step, t % n_fetch ==
        0, accumulates its gradients in its GradBuf and pushes them at steps with
        (t + 1) % n_push == 0, when the server applies the R buffers once).
        optimizer: "sgd", "momentum", "nesterov" or "adagrad"; weight_decay adds
        lambda*W to the summed gradient at the server.
        concurrent: run the per-layer updates on a second stream, overlapping
        the rest of the backward pass (False: everything on one stream).
        graphs: replay captured CUDA graphs of the step ("auto": when the delay
        schedule is periodic — pipeline stages or no delay — so the same few
        steps recur; the seeded random ASGD schedule is issued step by step).
        lookahead: with pipeline stage delays, step t also issues the forward
        pass of step t + 1, on a stream of its own beside step t's backward
        pass: a stage whose weights are s_k >= 1 steps old needs none of step
        t's updates ("Pipelined training of deep CNNs with stale weights"
        Sec. 4.1: the stages of different minibatches run at the same time);
        layers with s_k = 0 wait for step t's update of their weights. Two
        activation sets alternate by step parity. The softmax then opens the
        backward pass. Step t + 1's batch must be in the pool when step t is
        issued ("auto": on for pipeline delays without replica streams)."""
        S.lib()  # fail loudly if the CUDA library is missing
        self.net = net
        self.shapes = layer_shapes(net)
        self.n = padded_size(self.shapes)
        self.N = int(batch)
        self.R = int(replicas)
        self.pipeline = stage_delays is not None
        self.fetch_push = n_fetch is not None or n_push is not None
        self.hybrid_switch = None if hybrid_switch is None else int(hybrid_switch)
        if self.pipeline:
            if stage_of_layer is None or len(stage_of_layer) != len(self.shapes):
                raise ValueError("stage_delays needs stage_of_layer with one stage per layer")
            if self.fetch_push or max_delay:
                raise ValueError("pipeline stage delays exclude max_delay and n_fetch / n_push")
            self.stage_of_layer = list(stage_of_layer)
            self.stage_delays = [int(s) for s in stage_delays]
            if min(self.stage_delays) < 0 or max(self.stage_of_layer) >= len(self.stage_delays):
                raise ValueError("stage delays must be >= 0 and cover every stage of stage_of_layer")
            self.S = max(self.stage_delays)
        elif self.fetch_push:
            if max_delay or self.hybrid_switch is not None:
                raise ValueError("n_fetch / n_push exclude max_delay and hybrid_switch")
            self.n_fetch = 1 if n_fetch is None else int(n_fetch)
            self.n_push = 1 if n_push is None else int(n_push)
            if self.n_fetch < 1 or self.n_push < 1:
                raise ValueError("n_fetch and n_push must be >= 1")
            # versions count server updates: at most D behind the current one
            self.S = fetch_push_max_lag(self.n_fetch, self.n_push)
        else:
            if self.hybrid_switch is not None:
                raise ValueError("hybrid_switch needs pipeline stage delays")
            if max_delay < 0:
                raise ValueError("max_delay must be >= 0")
            self.S = int(max_delay)
        self.RS = self.S + 2 if self.fetch_push else self.S + 1   # weight-version ring slots
        self.seed = int(schedule_seed)
        self.optimizer = optimizer
        self.eta, self.nu, self.eps, self.g0 = float(eta), float(nu), float(eps), float(g0)
        self.weight_decay = float(weight_decay)
        self.dev = torch.device(device)
        f32 = dict(dtype=torch.float32, device=self.dev)

        self.ring = torch.zeros((self.RS, self.n), **f32)
        self.ringT = torch.zeros((self.RS, self.n), **f32)   # W^T of every layer that needs dX
        # the gradients pushed by update j live in set j % 2 (step t's update index: _cur(t))
        self.gradbuf_sets = torch.zeros((2, self.R, self.n), **f32)
        self.gradbuf = self.gradbuf_sets[0]
        if optimizer in ("momentum", "nesterov"):
            self.opt_state = torch.zeros(self.n, **f32)
        elif optimizer == "adagrad":
            self.opt_state = torch.full((self.n,), self.g0, **f32)
        elif optimizer == "sgd":
            self.opt_state = None
        else:
            raise ValueError(optimizer)
        self.loss = torch.zeros((self.R, 4), **f32)  # row r, column 0 = replica r's loss
        self.classes = self.shapes[-1].cout
        # parameter span of each layer (W then b, padded): the per-layer update range
        ends = [L.w_off for L in self.shapes[1:]] + [self.n]
        self.span = [(L.w_off, e - L.w_off) for L, e in zip(self.shapes, ends)]
        self.lookahead = (self.pipeline and concurrent and not (self.R > 1 and any(L.kind == "conv" for L in self.shapes))
                          if lookahead == "auto" else bool(lookahead))
        self._alloc_acts()

        main = torch.cuda.current_stream(self.dev)
        self.main_stream = main
        # lowest priority: on a higher-priority caller stream the backward GEMMs are
        # scheduled first and the updates take what the GPU has left
        self.upd_stream = torch.cuda.Stream(self.dev, priority=0) if concurrent else main
        # convolutions of different replicas run side by side (each with its own
        # workspace): the small late layers alone leave most SMs idle
        self.fork = concurrent and self.R > 1 and any(L.kind == "conv" for L in self.shapes)
        if self.fork:
            self.rep_streams = [torch.cuda.Stream(self.dev) for _ in range(self.R)]
            self.rep_ws = [torch.empty(max(self.conv_ws_bytes // 4 + 64, 64), **f32) for _ in range(self.R)]
            self.ev_fork = torch.cuda.Event()
            self.ev_join = [torch.cuda.Event() for _ in range(self.R)]
        else:
            self.rep_streams = [main] * self.R
            self.rep_ws = [self.ws] * self.R
        # a conv layer's weight gradient runs on a stream of its own (per replica, with its
        # own workspace) beside the input-gradient chain of the layers below, and the
        # gradient buffers rotate through three so that it can still read its dy while the
        # next two layers' gradients are written
        self.split_bwd = concurrent and any(L.kind == "conv" for L in self.shapes)
        if self.split_bwd:
            self.dw_streams = [torch.cuda.Stream(self.dev) for _ in range(self.R)]
            self.ws_dw = [torch.empty(max(self.conv_ws_bytes // 4 + 64, 64), **f32) for _ in range(self.R)]
            self.gspare = torch.empty_like(self.g)
            self.ev_gready = [[torch.cuda.Event() for _ in range(self.R)] for _ in self.shapes]
            self.ev_dw = [[torch.cuda.Event() for _ in range(self.R)] for _ in self.shapes]
            # the weight gradients' copies of their inputs (blocked x^T), made on the weight-
            # gradient streams during the forward pass, beside the forward GEMMs
            self.ev_xready = [[torch.cuda.Event() for _ in range(self.R)] for _ in self.shapes]
            for A in self._sets:
                for li, L in enumerate(self.shapes):
                    nb = S.sprint_conv_xT_size(self.N, L.h, L.w, L.cin, L.cout, 1) if L.kind == "conv" else 0
                    A["xT"][li] = torch.empty((self.R, (nb // 4 + 63) // 64 * 64), **f32) if nb else None
            self.xT_bufs = self._sets[0]["xT"]
        self.K = self.RS + 2   # version v of layer l exists: ev_layer[l][v % K]
        self.ev_layer = [[torch.cuda.Event() for _ in range(self.K)] for _ in self.shapes]
        self.ev_bwd = [torch.cuda.Event() for _ in self.shapes]
        for evs in self.ev_layer:
            evs[0].record(main)
        self.ev_inputs = torch.cuda.Event()
        self.inputs_pending = False
        # lookahead: the forward pass of step t + 1 on its own stream; _ahead = the step whose
        # forward pass has been issued already (or None)
        self.ahead_stream = torch.cuda.Stream(self.dev) if self.lookahead else None
        self._ahead = None
        self._ahead_graph = False   # that forward pass is part of a replayed (joined) step
        self.ev_fwd_done = [torch.cuda.Event() for _ in range(2)]
        self.ev_fwd_cap = torch.cuda.Event()
        self.ev_dw_cap = [torch.cuda.Event() for _ in range(self.R)]
        self.ev_bwd_done = [torch.cuda.Event() for _ in range(2)]
        self.ev_ahead_fork = torch.cuda.Event()
        self.ev_upd_cap = [torch.cuda.Event() for _ in self.shapes]   # per layer, inside one captured step
        self._sched = np.zeros((0, self.R), np.int32)
        self.batches_x = None
        self.batches_y = None
        self.t = 0
        periodic = (self.pipeline or self.S == 0) and not self.fetch_push
        self.use_graphs = periodic if graphs == "auto" else bool(graphs)
        self._graphs = {}            # step key -> captured CUDA graph
        self._graph_steps = False    # the last step ran as a graph replay
        self._graph_kernels = {}     # step key -> kernels in the graph
        self.graph_launch_adjust = 0  # kernels replayed minus kernels counted while capturing
        self.ev_graph_upd = torch.cuda.Event()
        self._cap_stream = None
        self.span_hook = None   # optional timing hook around each layer's per-replica convolution group

    # ------------------------------------------------------------------ buffers
    def _alloc_acts(self):
        """Per layer one [R][...] tensor (replica r's slice is row r), the
        gradient ping-pong pair [R][big], and one workspace for the largest call."""
        f32 = dict(dtype=torch.float32, device=self.dev)
        R, N = self.R, self.N

        def rows(numel, dtype=torch.float32):
            # [R][numel] with each replica's row starting on a 256-byte boundary
            stride = (numel + 255) // 256 * 256
            return torch.empty((R, stride), dtype=dtype, device=self.dev)[:, :numel]

        # one activation set per step parity when the next step's forward pass runs ahead
        self._sets = []
        big = 0
        ws_bytes = 0
        conv_ws = 0
        for _ in range(2 if self.lookahead else 1):
            outs, pooled, argmax = [], [], []
            # FC layers followed by an FC layer also keep their output transposed,
            # [out + 1][N] with a last row of ones (the next layer's xT1 operand:
            # its weight-gradient GEMM reads it as is and yields db in the same pass)
            outsT = []
            for li, L in enumerate(self.shapes):
                if L.kind == "conv":
                    numel = N * L.h * L.w * L.cout
                    big = max(big, numel, N * L.h * L.w * L.cin)
                    outs.append(rows(numel))
                    if L.pool:
                        ph, pw = L.out_hw
                        pooled.append(rows(N * ph * pw * L.cout))
                        argmax.append(rows(N * ph * pw * L.cout, torch.uint8))
                    else:
                        pooled.append(None)
                        argmax.append(None)
                    for op in (S.SPRINT_CONV_FWD, S.SPRINT_CONV_DX, S.SPRINT_CONV_DW):
                        conv_ws = max(conv_ws, S.sprint_conv_workspace_size(op, N, L.h, L.w, L.cin, L.cout, 1))
                else:
                    numel = N * L.cout
                    big = max(big, numel, N * L.cin)
                    outs.append(rows(numel))
                    pooled.append(None)
                    argmax.append(None)
                    ws_bytes = max(ws_bytes, S.sprint_fc_batched_workspace_size(R, N, L.cin, L.cout, 1),
                                   S.sprint_fc_batched_workspace_size(R, N, L.cin, L.cout, 0))
                nxt = self.shapes[li + 1] if li + 1 < len(self.shapes) else None
                if L.kind == "fc" and nxt is not None and nxt.kind == "fc":
                    t = rows((L.cout + 1) * N)
                    t[:, L.cout * N:].fill_(1.0)
                    outsT.append(t)
                else:
                    outsT.append(None)
            self._sets.append(dict(outs=outs, pooled=pooled, argmax=argmax, outsT=outsT, xT=[None] * len(outs)))
        self.outs, self.pooled, self.argmax, self.outsT = (self._sets[0][k] for k in ("outs", "pooled", "argmax",
                                                                                       "outsT"))
        self._acts_par = 0   # the set holding the last issued step's forward pass
        self.g = rows(big)
        self.h = rows(big)
        # dE/dy of FC layers transposed ([out][N]), written by the dX GEMM of the layer above
        self.gT = rows(big)
        self.hT = rows(big)
        self.ws = torch.empty(max(max(ws_bytes, conv_ws) // 4 + 64, 64), **f32)
        self.ws_bytes = self.ws.numel() * 4
        # the forward pass that runs ahead has a workspace of its own
        self.ws_ahead = torch.empty_like(self.ws) if self.lookahead else None
        self.conv_ws_bytes = conv_ws

    @property
    def acts(self):
        """Per-replica views of the last step's forward tensors (what replica r's
        pass read and wrote): outs, pooled and argmax per layer."""
        A = self._sets[self._acts_par]
        return [dict(outs=[o[r] for o in A["outs"]],
                     pooled=[p[r] if p is not None else None for p in A["pooled"]],
                     argmax=[a[r] if a is not None else None for a in A["argmax"]])
                for r in range(self.R)]

    # ------------------------------------------------------------------ data / weights
    def load_weights(self, dense: np.ndarray):
        """Sets W(0) from a dense [W0 b0 W1 b1 ...] fp32 vector."""
        torch.cuda.synchronize(self.dev)
        w = torch.from_numpy(pack(self.shapes, np.asarray(dense, np.float32)))
        self.ring[0].copy_(w.to(self.dev))
        for li in range(1, len(self.shapes)):
            self._transpose_layer(li, 0, self.main_stream)
        if self.optimizer in ("momentum", "nesterov"):
            self.opt_state.zero_()
        elif self.optimizer == "adagrad":
            self.opt_state.fill_(self.g0)
        self.t = 0
        self._graph_steps = False   # eager again until the schedule is periodic
        torch.cuda.synchronize(self.dev)
        for evs in self.ev_layer:
            evs[0].record(self.main_stream)

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
        """The batch pool was (re)written on `stream`: the next step waits for
        that work before reading it."""
        self.ev_inputs.record(stream)
        self.inputs_pending = True

    def weights(self, version=None) -> np.ndarray:
        """Dense copy of W(version) (default: the current version). Versions are
        steps (W(t) is the version before step t's update), or server updates
        with n_fetch / n_push."""
        v = self._cur(self.t) if version is None else version
        torch.cuda.synchronize(self.dev)
        return unpack(self.shapes, self.ring[v % self.RS].cpu().numpy())

    def staleness(self, t=None):
        """Stale-weight metrics of a pipeline at step t (default: the next step),
        "Pipelined training of deep CNNs with stale weights" Sec. 4.1: the degree
        of staleness of every stage pair (the steps its weights lag) and the
        percentage of the parameters held by stages with stale weights."""
        if not self.pipeline:
            raise ValueError("staleness metrics are defined for pipeline stages")
        t = self.t if t is None else t
        delays = [self._stage_delay(k, t) for k in range(len(self.stage_delays))]
        return dict(degrees=staleness_degrees(delays),
                    stale_weight_percent=stale_weight_percent(self.shapes, self.stage_of_layer, delays))

    def _transpose_layer(self, li, slot, stream):
        """W_l^T of version slot `slot` into ringT (layers after the first need dE/dX)."""
        L = self.shapes[li]
        rows, cols = (L.cout, 9 * L.cin) if L.kind == "conv" else (L.cout, L.cin)
        src = self.ring[slot].data_ptr() + 4 * L.w_off
        dst = self.ringT[slot].data_ptr() + 4 * L.w_off
        S.sprint_transpose(src, dst, rows, cols, stream.cuda_stream)

    def schedule(self, steps) -> np.ndarray:
        if self._sched.shape[0] < steps:
            n = max(steps, 2 * self._sched.shape[0], 256)
            self._sched = S.sprint_staleness_schedule(self.seed, n, self.R, self.S)
        return self._sched[:steps]

    # ------------------------------------------------------------------ one step
    def _stage_delay(self, k, t):
        """Delay of pipeline stage k at step t (0 from the hybrid switch on)."""
        if self.hybrid_switch is not None and t >= self.hybrid_switch:
            return 0
        return self.stage_delays[k]

    def _cur(self, t):
        """Index of the newest weight version before step t's update: steps, or
        server updates with n_fetch / n_push (pushes end steps n_push-1, 2n_push-1, ...)."""
        return t // self.n_push if self.fetch_push else t

    def _pushes(self, t):
        """Step t ends with a server update."""
        return not self.fetch_push or (t + 1) % self.n_push == 0

    def _first(self, t):
        """Step t assigns (rather than adds to) the GradBufs: the first step of a push window."""
        return not self.fetch_push or t % self.n_push == 0

    def _version(self, t, r, layer):
        if self.pipeline:
            return max(0, t - self._stage_delay(self.stage_of_layer[layer], t))
        if self.fetch_push:   # the server's version at the replica's last fetch step
            return fetch_push_version(t, self.n_fetch, self.n_push)
        s = int(self.schedule(t + 1)[t, r]) if self.S > 0 else 0
        return max(0, t - s)

    def _update_layer(self, t, li, stream):
        """SumGradient + UpdateWeights (Algorithm 2) of layer li: W_l(t+1) into
        ring slot t+1 in one launch, with W's transpose written in the same pass
        (layers after the first)."""
        off, cnt = self.span[li]
        j = self._cur(t)
        slot_in, slot_out = j % self.RS, (j + 1) % self.RS
        sh = stream.cuda_stream
        hp = self.eps if self.optimizer == "adagrad" else self.nu
        gb = self.gradbuf_sets[j % 2]

        def ptrs(o):
            return (self.ring[slot_in].data_ptr() + 4 * o, self.ring[slot_out].data_ptr() + 4 * o,
                    self.opt_state.data_ptr() + 4 * o if self.opt_state is not None else None,
                    [gb[r].data_ptr() + 4 * o for r in range(self.R)])

        w_in, w_out, st, bufs = ptrs(off)
        if li == 0:   # no input gradient: no transpose; W, b and padding in one pass
            S.sprint_apply_update(self.optimizer, w_in, w_out, st, bufs, cnt, self.eta, hp, self.weight_decay, sh)
            return
        L = self.shapes[li]
        rows, cols = (L.cout, 9 * L.cin) if L.kind == "conv" else (L.cout, L.cin)
        wT = self.ringT[slot_out].data_ptr() + 4 * L.w_off
        # W (transposed copy too), then the rest of the span (b and padding) in the same launch
        S.sprint_apply_update_t(self.optimizer, w_in, w_out, wT, st, bufs, rows, cols, self.eta, hp, sh, n_total=cnt,
                                weight_decay=self.weight_decay)

    def _per_replica(self, fn, tag=None, main=None, ws=None):
        """fn(r, stream_handle, ws, ws_bytes) for every replica: on the replica
        streams (forked from and joined back into the main stream) or in order
        on the main stream (default: self.main_stream; ws: its workspace, default
        self.ws). If span_hook is set, it is called with (tag, 0, main stream)
        before the group and (tag, 1, main stream) after it has joined, so events
        it records there bracket the whole group."""
        main = self.main_stream if main is None else main
        ws = self.ws if ws is None else ws
        hook = self.span_hook if tag is not None else None
        if hook:
            hook(tag, 0, main)
        if not self.fork:
            for r in range(self.R):
                fn(r, main.cuda_stream, ws, ws.numel() * 4)
        else:
            self.ev_fork.record(main)
            for r in range(self.R):
                st = self.rep_streams[r]
                st.wait_event(self.ev_fork)
                fn(r, st.cuda_stream, self.rep_ws[r], self.rep_ws[r].numel() * 4)
                self.ev_join[r].record(st)
            for r in range(self.R):
                main.wait_event(self.ev_join[r])
        if hook:
            hook(tag, 1, main)

    def _graph_key(self, t):
        """Everything a captured step bakes in: weight slots, GradBuf parity, batches."""
        nL = len(self.shapes)
        P = self.batches_x.shape[0]
        slots = tuple(self._version(t, r, li) % self.RS for r in range(self.R) for li in range(nL))
        bx = tuple(self.batches_x[(t * self.R + r) % P].data_ptr() for r in range(self.R))
        by = tuple(self.batches_y[(t * self.R + r) % P].data_ptr() for r in range(self.R))
        key = (slots, self._cur(t) % 2, self._first(t), self._pushes(t), bx, by)
        if self.lookahead:   # the captured step also holds step t + 1's forward pass
            slots1 = tuple(self._version(t + 1, r, li) % self.RS for r in range(self.R) for li in range(nL))
            bx1 = tuple(self.batches_x[((t + 1) * self.R + r) % P].data_ptr() for r in range(self.R))
            key = key + (slots1, bx1, t % 2)
        return key

    def _capture(self, t, key):
        """Captures step t's graph (not run): on a stream of our own (capture needs
        a non-default stream), standing in for the main stream while it is issued."""
        main = self.main_stream
        if self._cap_stream is None:
            self._cap_stream = torch.cuda.Stream(self.dev)
        g = torch.cuda.CUDAGraph()
        n0 = S.sprint_launch_count()
        self.main_stream = self._cap_stream
        state = (self._ahead, self._ahead_graph, self._acts_par)   # issuing records them; capturing runs nothing
        try:
            with torch.cuda.graph(g, stream=self._cap_stream, capture_error_mode="relaxed"):
                self._issue(t, graph=True)
        finally:
            self.main_stream = main
            self._ahead, self._ahead_graph, self._acts_par = state
        self._graphs[key] = g
        self._graph_kernels[key] = S.sprint_launch_count() - n0
        self.graph_launch_adjust -= self._graph_kernels[key]   # captured, not run
        return g

    def prepare_graphs(self):
        """Captures (without running them) the graphs of every step of one period of
        the schedule from the current step on, so later steps only replay; returns
        how many graphs are cached. No-op unless graphs are in use."""
        if not self.use_graphs:
            return 0
        P = self.batches_x.shape[0]
        period = int(np.lcm.reduce([self.S + 1, 2, P // np.gcd(P, self.R) if P else 1]))
        t0 = max(self.t, self.S)
        starts = [t0]
        if self.hybrid_switch is not None and self.hybrid_switch + self.S > t0:
            # the steps around and after the switch to non-pipelined training recur too
            starts.append(max(t0, self.hybrid_switch))
        for a in starts:
            for t in range(a, a + period + self.S):
                key = self._graph_key(t)
                if key not in self._graphs:
                    self._capture(t, key)
        return len(self._graphs)

    def step(self):
        """One global step: every replica's gradient, then the update, layer by
        layer. Asynchronous."""
        t = self.t
        main = self.main_stream
        if self.inputs_pending:
            main.wait_event(self.ev_inputs)
            if self.lookahead:
                self.ahead_stream.wait_event(self.ev_inputs)
            self.inputs_pending = False
        if self._ahead == t:
            if not self._ahead_graph:   # (a replayed step joined its forward pass ahead itself)
                main.wait_event(self.ev_fwd_done[t % 2])   # this step's forward pass ran ahead
        elif self.lookahead:
            # prologue: the first step (or one after a step without lookahead) issues its
            # own forward pass first
            if self._graph_steps:
                self.join()
            self._issue_forward(t, False, main, self.ws)
            self._ahead = None
        # Periodic schedules: once past the first S steps (whose versions are clamped
        # at 0) a step is a replay of the graph captured for its key. A captured step
        # ends with the update stream joined into the main stream, so replays are
        # ordered by the main stream alone and need none of the per-layer events.
        if self.use_graphs and t >= self.S:
            if not self._graph_steps:
                self.join()   # the eager steps' updates still in flight
            key = self._graph_key(t)
            g = self._graphs.get(key)
            if g is None:
                g = self._capture(t, key)
            with torch.cuda.stream(main):
                g.replay()
            self.graph_launch_adjust += self._graph_kernels[key]
            self._graph_steps = True
            if self.lookahead:
                self._ahead = t + 1
                self._ahead_graph = True
                self._acts_par = t % 2
            self.gradbuf = self.gradbuf_sets[self._cur(t) % 2]
            self.t = t + 1
            return
        if self._ahead == t and not self.lookahead:
            # forward pass ahead issued while lookahead was on: this step has it already
            self._ahead = None
            dw_last = self._issue_backward(t, False)
            if dw_last is not None:
                for ev in dw_last:
                    main.wait_event(ev)
            self.gradbuf = self.gradbuf_sets[self._cur(t) % 2]
            self.t = t + 1
            return
        self._issue(t, graph=False)

    def _step_refs(self, t):
        """Per-step constants: weight-version slots per replica and layer, the batch
        indices, and pointer helpers into the weight ring."""
        R, nL = self.R, len(self.shapes)
        row = self.n * 4
        ring, ringT = self.ring.data_ptr(), self.ringT.data_ptr()
        ver = [[self._version(t, r, li) for li in range(nL)] for r in range(R)]
        slot = [[v % self.RS for v in vr] for vr in ver]
        P = self.batches_x.shape[0]
        bidx = [(t * R + r) % P for r in range(R)]

        def W(r, li):
            return ring + slot[r][li] * row + 4 * self.shapes[li].w_off

        def B(r, li):
            return ring + slot[r][li] * row + 4 * self.shapes[li].b_off

        def WT(r, li):
            return ringT + slot[r][li] * row + 4 * self.shapes[li].w_off

        return ver, bidx, W, B, WT

    def _fwd_ptrs(self, t):
        """Step t's layer inputs (per layer, per replica) and logits, in activation
        set t % sets (no work issued)."""
        R = self.R
        A = self._sets[t % len(self._sets)]
        _, bidx, _, _, _ = self._step_refs(t)
        cur = [self.batches_x[b].data_ptr() for b in bidx]
        inp = []
        for li, L in enumerate(self.shapes):
            inp.append(cur)
            if L.kind == "conv" and L.pool:
                cur = [A["pooled"][li][r].data_ptr() for r in range(R)]
            else:
                cur = [A["outs"][li][r].data_ptr() for r in range(R)]
        return inp, cur

    def _issue_forward(self, t, graph, stream, ws, cap_waits=None):
        """Forward pass of step t on `stream` into activation set t % sets (the
        softmax opens the backward pass). Eagerly every layer first waits for the
        version of its weights it reads; inside a capture, cap_waits {layer: event}
        holds the updates of the same captured step it must follow."""
        R, N, K = self.R, self.N, self.K
        sh = stream.cuda_stream
        A = self._sets[t % len(self._sets)]
        ver, bidx, W, B, WT = self._step_refs(t)
        wsb = ws.numel() * 4
        cur = [self.batches_x[b].data_ptr() for b in bidx]
        for li, L in enumerate(self.shapes):
            if not graph:
                stream.wait_event(self.ev_layer[li][max(ver[r][li] for r in range(R)) % K])
            elif cap_waits and li in cap_waits:
                stream.wait_event(cap_waits[li])
            outs = [A["outs"][li][r].data_ptr() for r in range(R)]
            if L.kind == "conv":
                def fwd(r, st, rws, rwsb, li=li, L=L, src=cur, outs=outs):
                    if self.split_bwd and A["xT"][li] is not None:
                        ev = self.ev_xready[li][r]
                        ev.record(self.rep_streams[r] if self.fork else stream)
                        dws = self.dw_streams[r]
                        dws.wait_event(ev)
                        S.sprint_conv_xT(src[r], A["xT"][li][r], N, L.h, L.w, L.cin, L.cout, 1, dws.cuda_stream)
                    S.sprint_conv_fwd(src[r], W(r, li), B(r, li), outs[r], N, L.h, L.w, L.cin, L.cout, 1, 1, rws,
                                      rwsb, st)
                    if L.pool:
                        S.sprint_pool_fwd(outs[r], A["pooled"][li][r], A["argmax"][li][r], N, L.h, L.w, L.cout, st)
                self._per_replica(fwd, ("fwd", li), main=stream, ws=ws)
                cur = [A["pooled"][li][r].data_ptr() for r in range(R)] if L.pool else outs
            else:
                yT = None if A["outsT"][li] is None else [A["outsT"][li][r].data_ptr() for r in range(R)]
                S.sprint_fc_fwd_batched(cur, [W(r, li) for r in range(R)], [B(r, li) for r in range(R)], outs, N,
                                        L.cin, L.cout, int(L.relu), ws, wsb, sh, yT=yT)
                cur = outs
        self._acts_par = t % len(self._sets)

    def _issue_backward(self, t, graph):
        """Softmax cross-entropy and backward pass of step t (reading activation set
        t % sets), each layer's update on the update stream as soon as its
        gradients are final. Returns the events of the weight-gradient streams the
        step's end must wait for (or None)."""
        R, N, K = self.R, self.N, self.K
        main, upd = self.main_stream, self.upd_stream
        sh = main.cuda_stream
        nL = len(self.shapes)
        A = self._sets[t % len(self._sets)]
        ver, bidx, W, B, WT = self._step_refs(t)
        inp, logits = self._fwd_ptrs(t)
        j = self._cur(t)
        gb = [self.gradbuf_sets[j % 2][r].data_ptr() for r in range(R)]
        acc = 0 if self._first(t) else 1   # GradBuf: assign at a window's first step, add afterwards
        ws, wsb = self.ws, self.ws_bytes
        g = [self.g[r].data_ptr() for r in range(R)]
        h = [self.h[r].data_ptr() for r in range(R)]
        # split backward: the three gradient buffers, and for each the event of the weight
        # gradient still reading it (waited for before the buffer is written again)
        bufs = [g, h, [self.gspare[r].data_ptr() for r in range(R)]] if self.split_bwd else None
        readers = [None, None, None]
        gi, hi, si = 0, 1, 2
        dw_last = None
        gT = None   # g transposed, when the layer above wrote it
        hT_all = [self.hT[r].data_ptr() for r in range(R)]
        gT_all = [self.gT[r].data_ptr() for r in range(R)]
        S.sprint_softmax_xent_batched(logits, [self.batches_y[b].data_ptr() for b in bidx],
                                      [self.loss[r].data_ptr() for r in range(R)], g, N, self.classes, 0, sh)

        # backward (g holds dE/d(pre-activation output) of layer li)
        for li in range(nL - 1, -1, -1):
            L = self.shapes[li]
            prev = self.shapes[li - 1] if li > 0 else None
            # update j-2 (the last reader of GradBuf set j % 2) of this layer has finished
            if not graph:
                main.wait_event(self.ev_layer[li][max(j - 1, 0) % K])
            dw = [gb[r] + 4 * L.w_off for r in range(R)]
            db = [gb[r] + 4 * L.b_off for r in range(R)]
            hT = None
            if L.kind == "fc":
                relu_src = None
                if prev is not None and not (prev.kind == "conv" and prev.pool) and prev.relu:
                    relu_src = inp[li]
                xT1 = None
                if prev is not None and A["outsT"][li - 1] is not None:
                    xT1 = [A["outsT"][li - 1][r].data_ptr() for r in range(R)]
                    hT = hT_all   # the layer below is FC too: it reads dE/dy transposed
                S.sprint_fc_bwd_batched(inp[li], [W(r, li) for r in range(R)],
                                        [WT(r, li) for r in range(R)] if prev is not None else None, g, relu_src,
                                        h if prev is not None else None, dw, db, 1.0, acc, N, L.cin, L.cout, ws, wsb,
                                        sh, xT1=xT1, dyT=gT, dxT=hT)
            elif self.split_bwd:
                if dw_last is None:   # the first conv layer: pick up the buffers the FC layers left
                    gi = next(i for i, bb in enumerate(bufs) if bb is g)
                    hi = next(i for i, bb in enumerate(bufs) if bb is h)
                    si = 3 - gi - hi
                g, h = bufs[gi], bufs[hi]
                rd_h, rd_s = readers[hi], readers[si]

                def bwd(r, st, rws, rwsb, li=li, L=L, prev=prev, g=g, h=h, s_=bufs[si], dw=dw, db=db, rd_h=rd_h,
                        rd_s=rd_s):
                    stream = self.rep_streams[r] if self.fork else main
                    dws = self.dw_streams[r]
                    ev = self.ev_gready[li][r]
                    ev.record(stream)
                    dws.wait_event(ev)
                    if A["xT"][li] is not None:   # x^T made during the forward pass, on this stream
                        S.sprint_conv_dW_xT(inp[li][r], A["xT"][li][r], g[r], dw[r], db[r], 1.0, acc, N, L.h,
                                            L.w, L.cin, L.cout, 1, self.ws_dw[r], self.ws_dw[r].numel() * 4,
                                            dws.cuda_stream)
                    else:
                        S.sprint_conv_dW(inp[li][r], g[r], dw[r], db[r], 1.0, acc, N, L.h, L.w, L.cin, L.cout, 1,
                                         self.ws_dw[r], self.ws_dw[r].numel() * 4, dws.cuda_stream)
                    self.ev_dw[li][r].record(dws)
                    if prev is None:
                        return
                    if rd_h is not None:
                        stream.wait_event(rd_h[r])
                    relu_src = None if prev.pool else inp[li][r]
                    S.sprint_conv_dX(g[r], W(r, li), WT(r, li), relu_src, h[r], N, L.h, L.w, L.cin, L.cout, 1,
                                     rws, rwsb, st)
                    if prev.kind == "conv" and prev.pool:
                        if rd_s is not None:
                            stream.wait_event(rd_s[r])
                        S.sprint_pool_bwd(h[r], A["argmax"][li - 1][r], A["pooled"][li - 1][r], s_[r], N, prev.h,
                                          prev.w, prev.cout, st)
                self._per_replica(bwd, ("bwd", li))
                readers[gi] = dw_last = self.ev_dw[li]
                if prev is not None:
                    readers[hi] = None
                    if prev.kind == "conv" and prev.pool:
                        readers[si] = None
                        gi, si = si, gi            # the routed gradient is next; h is free again
                    else:
                        gi, hi, si = hi, si, gi    # dx is next; the spare takes the next dx
            else:
                def bwd(r, st, rws, rwsb, li=li, L=L, prev=prev, g=g, h=h, dw=dw, db=db):
                    S.sprint_conv_dW(inp[li][r], g[r], dw[r], db[r], 1.0, acc, N, L.h, L.w, L.cin, L.cout, 1, rws,
                                     rwsb, st)
                    if prev is not None:
                        relu_src = None if prev.pool else inp[li][r]
                        S.sprint_conv_dX(g[r], W(r, li), WT(r, li), relu_src, h[r], N, L.h, L.w, L.cin, L.cout, 1,
                                         rws, rwsb, st)
                        if prev.kind == "conv" and prev.pool:
                            # g[r] (free) <- routed gradient of the pre-pool ReLU output, masked
                            S.sprint_pool_bwd(h[r], A["argmax"][li - 1][r], A["pooled"][li - 1][r], g[r], N, prev.h,
                                              prev.w, prev.cout, st)
                self._per_replica(bwd, ("bwd", li))
            # layer li's gradients are final: its update overlaps the layers below
            if self._pushes(t):
                self.ev_bwd[li].record(main)
                upd.wait_event(self.ev_bwd[li])
                if self.split_bwd and L.kind == "conv":
                    for ev in self.ev_dw[li]:
                        upd.wait_event(ev)
                self._update_layer(t, li, upd)
                if not graph:
                    self.ev_layer[li][(j + 1) % K].record(upd)
                else:
                    self.ev_upd_cap[li].record(upd)   # the forward pass running ahead may wait for it
            if prev is None:
                break
            if self.split_bwd and L.kind == "conv":
                continue   # the buffers rotated above
            if prev.kind == "conv" and prev.pool:
                if L.kind == "fc":
                    # the FC input gradient (in h) routed through the pool into g (free), masked
                    for r in range(R):
                        S.sprint_pool_bwd(h[r], A["argmax"][li - 1][r], A["pooled"][li - 1][r], g[r], N, prev.h,
                                          prev.w, prev.cout, sh)
                # the conv branch routed into g already: g holds the next layer's gradient
            else:
                g, h = h, g
                gT, hT_all, gT_all = hT, gT_all, hT_all
        return dw_last

    def _issue(self, t, graph):
        """Issues step t (graph: being captured — no waits on events recorded by
        earlier steps, no per-layer version events, the update stream joined at the
        end). With lookahead, step t's forward pass was issued before (ahead, or as
        the prologue) and step t + 1's is issued here beside the backward pass."""
        main, upd = self.main_stream, self.upd_stream
        j = self._cur(t)
        if not self.lookahead:
            self._issue_forward(t, graph, main, self.ws)
            dw_last = self._issue_backward(t, graph)
        else:
            ahead = self.ahead_stream
            if graph:
                self.ev_ahead_fork.record(main)   # the forward pass ahead depends on nothing before it
            dw_last = self._issue_backward(t, graph)
            if graph:
                ahead.wait_event(self.ev_ahead_fork)
                # layers whose step-(t + 1) weights are this step's update follow it
                waits = {li: self.ev_upd_cap[li] for li in range(len(self.shapes))
                         if self._pushes(t) and max(self._version(t + 1, r, li) for r in range(self.R)) > j}
            else:
                ahead.wait_event(self.ev_bwd_done[(t + 1) % 2])   # step t - 1 no longer reads that set
                waits = None
            self._issue_forward(t + 1, graph, ahead, self.ws_ahead, waits)
            # (an event recorded inside a capture cannot be waited for outside it: captures
            # join the forward pass ahead through an event of their own)
            (self.ev_fwd_cap if graph else self.ev_fwd_done[(t + 1) % 2]).record(ahead)
            self._ahead = t + 1
            self._ahead_graph = graph
            self._acts_par = t % 2   # tr.acts: the step being issued
        if dw_last is not None:
            # the next step overwrites activations the weight gradients read
            for ev in dw_last:
                main.wait_event(ev)
        if self.lookahead and not graph:
            self.ev_bwd_done[t % 2].record(main)
        if graph:
            if self.lookahead:   # join the forward pass ahead (and its x^T copies)
                main.wait_event(self.ev_fwd_cap)
                if self.split_bwd:
                    for r in range(self.R):
                        self.ev_dw_cap[r].record(self.dw_streams[r])
                        main.wait_event(self.ev_dw_cap[r])
            # join the update stream: the next replay starts after this step's updates
            self.ev_graph_upd.record(upd)
            main.wait_event(self.ev_graph_upd)
            return
        self.gradbuf = self.gradbuf_sets[j % 2]   # the GradBufs of the step just issued
        self.t = t + 1

    def join(self, stream=None):
        """Makes `stream` (default: the main stream) wait for every update
        issued so far (the last step's updates may still run on the update
        stream when step() returns)."""
        st = self.main_stream if stream is None else stream
        if self._ahead is not None and not self._ahead_graph:   # the forward pass running ahead
            st.wait_event(self.ev_fwd_done[self._ahead % 2])
        if self._graph_steps:   # graph replays end with the update stream joined
            if st is not self.main_stream:
                ev = torch.cuda.Event()
                ev.record(self.main_stream)
                st.wait_event(ev)
            return
        for evs in self.ev_layer:
            st.wait_event(evs[self._cur(self.t) % self.K])

    def drop_lookahead(self):
        """Waits for the forward pass issued ahead (if any) and forgets it: the next
        step issues its own forward pass again (after the batch pool or the weights
        were changed from outside, or to time one whole step)."""
        self.join()
        self.main_stream.synchronize()
        self._ahead = None
        self._ahead_graph = False

    def step_loss(self) -> float:
        """Mean over replicas of the last step's loss (synchronises)."""
        self.join()
        self.main_stream.synchronize()
        return float(self.loss[:, 0].mean().item())
