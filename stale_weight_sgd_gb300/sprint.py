"""Python binding of libsprint (include/sprint.h): argument marshalling only.

Every function has the C name and argument order. Tensor arguments may be
torch tensors (their data_ptr() is passed) or plain integers (raw device
addresses); ``stream`` defaults to torch's current CUDA stream. A non-zero
status raises SprintError with the library's message. There is no fallback:
if libsprint.so is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "libsprint.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "sprint.h")

SPRINT_OK = 0
STATUS_NAMES = {
    0: "SPRINT_OK", 1: "SPRINT_ERR_INVALID_ARG", 2: "SPRINT_ERR_SHAPE", 3: "SPRINT_ERR_ALIGN",
    4: "SPRINT_ERR_UNSUPPORTED", 5: "SPRINT_ERR_CUDA", 6: "SPRINT_ERR_DEVICE_FLAG", 7: "SPRINT_ERR_WORKSPACE",
}
SPRINT_CONV_FWD, SPRINT_CONV_DX, SPRINT_CONV_DW = 0, 1, 2


class SprintError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} -> {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


_lib = None

P = ctypes.c_void_p
I = ctypes.c_int
F = ctypes.c_float
SZ = ctypes.c_size_t

_SIGS = {
    "sprint_last_error": ([], ctypes.c_char_p),
    "sprint_version": ([], I),
    "sprint_launch_count": ([], ctypes.c_uint64),
    "sprint_device_status": ([ctypes.POINTER(I), I], I),
    "sprint_selftest_bounded_wait": ([ctypes.c_uint64, P], I),
    "sprint_conv_plan": ([I, I, I, I, I, I, I, I, P, I], I),
    "sprint_gemm_plan": ([I, I, I, I, I, P, I], I),
    "sprint_im2col": ([P, I, I, I, I, I, P, P, P], I),
    "sprint_conv_fwd": ([P, P, P, P, I, I, I, I, I, I, I, P, SZ, P], I),
    "sprint_conv_dX": ([P, P, P, P, P, I, I, I, I, I, I, P, SZ, P], I),
    "sprint_conv_workspace_size": ([I, I, I, I, I, I, I], SZ),
    "sprint_conv_dW": ([P, P, P, P, F, I, I, I, I, I, I, I, P, SZ, P], I),
    "sprint_conv_xT_size": ([I, I, I, I, I, I], SZ),
    "sprint_conv_xT": ([P, P, I, I, I, I, I, I, P], I),
    "sprint_conv_dW_xT": ([P, P, P, P, P, F, I, I, I, I, I, I, I, P, SZ, P], I),
    "sprint_fc_fwd": ([P, P, P, P, I, I, I, I, P], I),
    "sprint_fc_bwd": ([P, P, P, P, P, P, P, P, F, I, I, I, I, P, SZ, P], I),
    "sprint_fc_workspace_size": ([I, I, I, I], SZ),
    "sprint_fc_bwd_static_scratch": ([P, P, P, P, P, P, P, P, F, I, I, I, I, P], I),
    "sprint_fc_bwd_static_scratch_bytes": ([], SZ),
    "sprint_fc_fwd_batched": ([P, P, P, P, P, I, I, I, I, I, P, SZ, P], I),
    "sprint_fc_fwd_batched_workspace_size": ([], SZ),
    "sprint_fc_batched_workspace_size": ([I, I, I, I, I], SZ),
    "sprint_fc_bwd_batched": ([P, P, P, P, P, P, P, P, P, P, P, F, I, I, I, I, I, P, SZ, P], I),
    "sprint_apply_update": ([I, P, P, P, P, I, SZ, F, F, F, P], I),
    "sprint_apply_update_t": ([I, P, P, P, P, P, I, I, I, SZ, F, F, F, P], I),
    "sprint_fc_bwd_update_batched": ([P, P, P, P, P, P, P, P, P, P, P, F, I, I, I, I, I, I, P, P, P, P, P, P, P, F, F, F,
                                      P, SZ, P], I),
    "sprint_transpose": ([P, P, I, I, P], I),
    "sprint_pool_fwd": ([P, P, P, I, I, I, I, P], I),
    "sprint_pool_bwd": ([P, P, P, P, I, I, I, I, P], I),
    "sprint_softmax_xent": ([P, P, I, I, P, P, I, P], I),
    "sprint_softmax_xent_batched": ([P, P, P, P, I, I, I, I, P], I),
    "sprint_gradbuf_accumulate": ([P, P, SZ, F, I, P], I),
    "sprint_apply_update_sgd": ([P, P, P, I, SZ, F, P], I),
    "sprint_apply_update_momentum": ([P, P, P, P, I, SZ, F, F, P], I),
    "sprint_apply_update_adagrad": ([P, P, P, P, I, SZ, F, F, P], I),
    "sprint_staleness_schedule": ([ctypes.c_uint64, I, I, I, P], I),
}


def header_functions() -> list[str]:
    """Names of the functions include/sprint.h declares."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(sprint_[a-zA-Z0-9_]+)\s*\(", txt)))


def lib() -> ctypes.CDLL:
    """Loads libsprint.so (built by stale_weight_sgd_gb300.build); raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libsprint.so not built ({LIB_PATH}); run python -m stale_weight_sgd_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, ret) in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ret
        _lib = L
    return _lib


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _s(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(name, rc):
    if rc != SPRINT_OK:
        raise SprintError(name, rc, lib().sprint_last_error().decode())
    return rc


def sprint_last_error() -> str:
    return lib().sprint_last_error().decode()


def sprint_version() -> int:
    return lib().sprint_version()


def sprint_launch_count() -> int:
    return int(lib().sprint_launch_count())


PLAN_FIELDS = ("path", "bn", "pair", "splits", "tail_splits", "wg_tpt", "wg_rows", "num_kt", "box_w", "box_h",
               "box_img", "wg_blocked", "wg_fact", "conv_fact", "conv_halo", "conv_rgb", "conv_hflip")
PATH_NAMES = {0: "simt", 1: "tc", 2: "smallc", 3: "im2col"}


def _plan(name, *args):
    buf = (ctypes.c_int32 * len(PLAN_FIELDS))()
    _check(name, getattr(lib(), name)(*args, ctypes.cast(buf, P), len(PLAN_FIELDS)))
    d = dict(zip(PLAN_FIELDS, list(buf)))
    d["path"] = PATH_NAMES[d["path"]]
    return d


def sprint_conv_plan(op, N, H, W, Cin, Cout, pad=1, have_wT=True) -> dict:
    return _plan("sprint_conv_plan", op, N, H, W, Cin, Cout, pad, int(bool(have_wT)))


def sprint_gemm_plan(M, N, K, batch=1, allow_tail=True) -> dict:
    return _plan("sprint_gemm_plan", M, N, K, batch, int(bool(allow_tail)))


def sprint_selftest_bounded_wait(limit_ns: int, stream=None) -> None:
    _check("sprint_selftest_bounded_wait", lib().sprint_selftest_bounded_wait(int(limit_ns), _s(stream)))


def sprint_device_status(reset: bool = True) -> int:
    v = I(0)
    rc = lib().sprint_device_status(ctypes.byref(v), int(reset))
    if rc not in (SPRINT_OK, 6):
        _check("sprint_device_status", rc)
    return v.value


def sprint_im2col(x, N, H, W, C, pad, col, src_index=None, stream=None):
    return _check("sprint_im2col", lib().sprint_im2col(_p(x), N, H, W, C, pad, _p(col), _p(src_index), _s(stream)))


def sprint_conv_workspace_size(op, N, H, W, Cin, Cout, pad) -> int:
    return lib().sprint_conv_workspace_size(op, N, H, W, Cin, Cout, pad)


def sprint_conv_fwd(x, w, b, y, N, H, W, Cin, Cout, pad, relu, ws=None, ws_bytes=0, stream=None):
    return _check("sprint_conv_fwd", lib().sprint_conv_fwd(_p(x), _p(w), _p(b), _p(y), N, H, W, Cin, Cout, pad,
                                                           int(relu), _p(ws), ws_bytes, _s(stream)))


def sprint_conv_dX(dy, w, wT, relu_src, dx, N, H, W, Cin, Cout, pad, ws=None, ws_bytes=0, stream=None):
    return _check("sprint_conv_dX", lib().sprint_conv_dX(_p(dy), _p(w), _p(wT), _p(relu_src), _p(dx), N, H, W, Cin,
                                                         Cout, pad, _p(ws), ws_bytes, _s(stream)))


def sprint_conv_dW(x, dy, dw, db, alpha, accumulate, N, H, W, Cin, Cout, pad, ws=None, ws_bytes=0, stream=None):
    return _check("sprint_conv_dW", lib().sprint_conv_dW(_p(x), _p(dy), _p(dw), _p(db), float(alpha),
                                                         int(accumulate), N, H, W, Cin, Cout, pad, _p(ws), ws_bytes,
                                                         _s(stream)))


def sprint_conv_xT_size(N, H, W, Cin, Cout, pad=1) -> int:
    return lib().sprint_conv_xT_size(N, H, W, Cin, Cout, pad)


def sprint_conv_xT(x, xT, N, H, W, Cin, Cout, pad=1, stream=None):
    return _check("sprint_conv_xT", lib().sprint_conv_xT(_p(x), _p(xT), N, H, W, Cin, Cout, pad, _s(stream)))


def sprint_conv_dW_xT(x, xT, dy, dw, db, alpha, accumulate, N, H, W, Cin, Cout, pad, ws=None, ws_bytes=0,
                      stream=None):
    return _check("sprint_conv_dW_xT", lib().sprint_conv_dW_xT(_p(x), _p(xT), _p(dy), _p(dw), _p(db), float(alpha),
                                                               int(accumulate), N, H, W, Cin, Cout, pad, _p(ws),
                                                               ws_bytes, _s(stream)))


def sprint_fc_fwd(x, w, b, y, N, in_, out, relu, stream=None):
    return _check("sprint_fc_fwd", lib().sprint_fc_fwd(_p(x), _p(w), _p(b), _p(y), N, in_, out, int(relu),
                                                       _s(stream)))


def sprint_fc_bwd(x, w, wT, dy, relu_src, dx, dw, db, alpha, accumulate, N, in_, out, ws=None, ws_bytes=0,
                  stream=None):
    return _check("sprint_fc_bwd", lib().sprint_fc_bwd(_p(x), _p(w), _p(wT), _p(dy), _p(relu_src), _p(dx), _p(dw),
                                                       _p(db), float(alpha), int(accumulate), N, in_, out, _p(ws),
                                                       ws_bytes, _s(stream)))


def sprint_fc_bwd_static_scratch(x, w, wT, dy, relu_src, dx, dw, db, alpha, accumulate, N, in_, out, stream=None):
    return _check("sprint_fc_bwd_static_scratch", lib().sprint_fc_bwd_static_scratch(
        _p(x), _p(w), _p(wT), _p(dy), _p(relu_src), _p(dx), _p(dw), _p(db), float(alpha), int(accumulate), N, in_, out,
        _s(stream)))


def sprint_fc_bwd_static_scratch_bytes() -> int:
    return int(lib().sprint_fc_bwd_static_scratch_bytes())


def sprint_fc_workspace_size(N, in_, out, have_wT) -> int:
    return lib().sprint_fc_workspace_size(N, in_, out, int(have_wT))


def sprint_transpose(src, dst, rows, cols, stream=None):
    return _check("sprint_transpose", lib().sprint_transpose(_p(src), _p(dst), rows, cols, _s(stream)))


def sprint_pool_fwd(x, y, argmax, N, H, W, C, stream=None):
    return _check("sprint_pool_fwd", lib().sprint_pool_fwd(_p(x), _p(y), _p(argmax), N, H, W, C, _s(stream)))


def sprint_pool_bwd(dy, argmax, pooled, dx, N, H, W, C, stream=None):
    return _check("sprint_pool_bwd", lib().sprint_pool_bwd(_p(dy), _p(argmax), _p(pooled), _p(dx), N, H, W, C,
                                                           _s(stream)))


def sprint_softmax_xent(logits, labels, N, C, loss, dlogits, reduction_sum=0, stream=None):
    return _check("sprint_softmax_xent", lib().sprint_softmax_xent(_p(logits), _p(labels), N, C, _p(loss),
                                                                   _p(dlogits), int(reduction_sum), _s(stream)))


def sprint_gradbuf_accumulate(buf, grad, n, alpha, first, stream=None):
    return _check("sprint_gradbuf_accumulate", lib().sprint_gradbuf_accumulate(_p(buf), _p(grad), n, float(alpha),
                                                                               int(first), _s(stream)))


def _ptr_array(bufs):
    arr = (ctypes.c_void_p * len(bufs))(*[_p(b) for b in bufs])
    return arr


def _opt_array(items):
    """Host pointer array for a batched call, or NULL for None (entries may be None)."""
    return None if items is None else _ptr_array(items)


def sprint_fc_fwd_batched(x, w, b, y, N, fin, fout, relu, ws=None, ws_bytes=0, stream=None, yT=None):
    n = len(x)
    return _check("sprint_fc_fwd_batched", lib().sprint_fc_fwd_batched(
        _ptr_array(x), _ptr_array(w), _opt_array(b), _ptr_array(y), _opt_array(yT), n, N, fin, fout, int(relu),
        _p(ws), ws_bytes, _s(stream)))


def sprint_fc_fwd_batched_workspace_size() -> int:
    return lib().sprint_fc_fwd_batched_workspace_size()


def sprint_fc_batched_workspace_size(batch, N, fin, fout, have_wT) -> int:
    return lib().sprint_fc_batched_workspace_size(batch, N, fin, fout, int(have_wT))


def sprint_fc_bwd_batched(x, w, wT, dy, relu_src, dx, dw, db, alpha, accumulate, N, fin, fout, ws=None, ws_bytes=0,
                          stream=None, xT1=None, dyT=None, dxT=None):
    n = len(x)
    return _check("sprint_fc_bwd_batched", lib().sprint_fc_bwd_batched(
        _ptr_array(x), _opt_array(xT1), _ptr_array(w), _opt_array(wT), _ptr_array(dy), _opt_array(dyT),
        _opt_array(relu_src), _opt_array(dx), _opt_array(dxT), _ptr_array(dw), _opt_array(db), float(alpha),
        int(accumulate), n, N, fin, fout, _p(ws), ws_bytes, _s(stream)))


SPRINT_OPT = {"sgd": 0, "momentum": 1, "adagrad": 2, "nesterov": 3}


def sprint_apply_update(opt, w_in, w_out, state, bufs, n, eta, nu_or_eps=0.0, weight_decay=0.0, stream=None):
    return _check("sprint_apply_update", lib().sprint_apply_update(
        SPRINT_OPT.get(opt, opt), _p(w_in), _p(w_out), _p(state), _ptr_array(bufs), len(bufs), n, float(eta),
        float(nu_or_eps), float(weight_decay), _s(stream)))


def sprint_apply_update_t(opt, w_in, w_out, wT_out, state, bufs, rows, cols, eta, nu_or_eps=0.0, stream=None,
                          n_total=None, weight_decay=0.0):
    n = rows * cols if n_total is None else n_total
    return _check("sprint_apply_update_t", lib().sprint_apply_update_t(
        SPRINT_OPT.get(opt, opt), _p(w_in), _p(w_out), _p(wT_out), _p(state), _ptr_array(bufs), len(bufs), rows, cols,
        n, float(eta), float(nu_or_eps), float(weight_decay), _s(stream)))


def sprint_fc_bwd_update_batched(x, w, wT, dy, relu_src, dx, dw, db, alpha, accumulate, N, fin, fout, opt, w_in, b_in,
                                 w_out, b_out, wT_out, w_state, b_state, eta, nu_or_eps, ws=None, ws_bytes=0,
                                 stream=None, xT1=None, dyT=None, dxT=None, weight_decay=0.0):
    n = len(x)
    return _check("sprint_fc_bwd_update_batched", lib().sprint_fc_bwd_update_batched(
        _ptr_array(x), _opt_array(xT1), _ptr_array(w), _opt_array(wT), _ptr_array(dy), _opt_array(dyT),
        _opt_array(relu_src), _opt_array(dx), _opt_array(dxT), _ptr_array(dw), _opt_array(db), float(alpha),
        int(accumulate), n, N, fin, fout, SPRINT_OPT.get(opt, opt), _p(w_in), _p(b_in), _p(w_out), _p(b_out),
        _p(wT_out), _p(w_state), _p(b_state), float(eta), float(nu_or_eps), float(weight_decay), _p(ws), ws_bytes,
        _s(stream)))


def sprint_softmax_xent_batched(logits, labels, loss, dlogits, N, C, reduction_sum=0, stream=None):
    n = len(logits)
    return _check("sprint_softmax_xent_batched", lib().sprint_softmax_xent_batched(
        _ptr_array(logits), _ptr_array(labels), _ptr_array(loss), _ptr_array(dlogits), n, N, C, int(reduction_sum),
        _s(stream)))


def sprint_apply_update_sgd(w_in, w_out, bufs, n, eta, stream=None):
    arr = _ptr_array(bufs)
    return _check("sprint_apply_update_sgd", lib().sprint_apply_update_sgd(_p(w_in), _p(w_out), arr, len(bufs), n,
                                                                           float(eta), _s(stream)))


def sprint_apply_update_momentum(w_in, w_out, v, bufs, n, eta, nu, stream=None):
    arr = _ptr_array(bufs)
    return _check("sprint_apply_update_momentum", lib().sprint_apply_update_momentum(
        _p(w_in), _p(w_out), _p(v), arr, len(bufs), n, float(eta), float(nu), _s(stream)))


def sprint_apply_update_adagrad(w_in, w_out, G, bufs, n, eta, eps, stream=None):
    arr = _ptr_array(bufs)
    return _check("sprint_apply_update_adagrad", lib().sprint_apply_update_adagrad(
        _p(w_in), _p(w_out), _p(G), arr, len(bufs), n, float(eta), float(eps), _s(stream)))


def sprint_staleness_schedule(seed, steps, replicas, max_delay):
    """Returns the [steps][replicas] int32 delay table (numpy)."""
    import numpy as np
    out = np.zeros((steps, replicas), np.int32)
    _check("sprint_staleness_schedule", lib().sprint_staleness_schedule(
        ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF), steps, replicas, max_delay, out.ctypes.data))
    return out
