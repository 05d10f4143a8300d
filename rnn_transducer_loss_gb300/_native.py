"""ctypes binding of librnnt_gb300.so (include/rnnt_gb300.h); argument marshalling only.

The function names mirror the C ABI.  The library is loaded lazily; if it is
missing the call raises (build it with ``python -m rnn_transducer_loss_gb300.build`` or
``__graft_entry__.build()``).  Nothing here computes any part of the loss.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librnnt_gb300.so")

RNNT_OK, RNNT_INVALID_VALUE, RNNT_WORKSPACE_TOO_SMALL = 0, 1, 2
RNNT_LAUNCH_FAILED, RNNT_LOSS_MISMATCH, RNNT_TIMEOUT = 3, 4, 5
RNNT_F32, RNNT_F16, RNNT_BF16 = 0, 1, 2
REDUCTIONS = {"none": 0, "sum": 1, "mean": 2}
MAX_TARGET_LENGTH = 1023
NOALLOC_SCRATCH_BYTES = 32 << 20     # RNNT_NOALLOC_SCRATCH_BYTES

# Every symbol include/rnnt_gb300.h declares.
EXPORTS = ("rnnt_workspace_size", "rnnt_workspace_size_ex", "rnnt_loss_fused", "rnnt_loss_fused_ex",
           "rnnt_loss_fused_staged", "rnnt_grad_scale", "rnnt_set_trace",
           "rnnt_loss_fused_noalloc", "rnnt_selftest_wait_timeout", "rnnt_status_string",
           "rnnt_abi_version", "rnnt_plan")


MAX_BIG_BLANKS = 8                    # RNNT_MAX_BIG_BLANKS
MAX_BIG_BLANK_DURATION = 16           # RNNT_MAX_BIG_BLANK_DURATION


class Options(ctypes.Structure):
    """rnnt_options_t: FastEmit weight, the padded (B, max_T, max_U + 1, V) layout,
    and the multi-blank transducer's big blanks and under-normalisation sigma."""
    _fields_ = [("fastemit_lambda", ctypes.c_float), ("padded", ctypes.c_int32),
                ("max_T", ctypes.c_int32), ("max_U", ctypes.c_int32),
                ("num_big_blanks", ctypes.c_int32),
                ("big_blank_ids", ctypes.c_int32 * MAX_BIG_BLANKS),
                ("big_blank_durations", ctypes.c_int32 * MAX_BIG_BLANKS),
                ("sigma", ctypes.c_float)]


def make_options(fastemit_lambda=0.0, padded=None, big_blanks=(), sigma=0.0) -> Options:
    """padded = (max_T, max_U) or None; big_blanks = [(output index, duration), ...]."""
    o = Options()
    o.fastemit_lambda = float(fastemit_lambda)
    if padded:
        o.padded, o.max_T, o.max_U = 1, int(padded[0]), int(padded[1])
    big = list(big_blanks or ())
    o.num_big_blanks = len(big)
    for i, (idx, dur) in enumerate(big[:MAX_BIG_BLANKS]):
        o.big_blank_ids[i], o.big_blank_durations[i] = int(idx), int(dur)
    o.sigma = float(sigma)
    return o

class Plan(ctypes.Structure):
    """rnnt_plan_t: whether one persistent kernel runs the call, and how many
    kernels the call enqueues."""
    _fields_ = [("persistent", ctypes.c_int32), ("launches", ctypes.c_int32)]


_lib = None


class RNNTError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        super().__init__(f"{where}: {status_string(code)} (status {code})")


def load() -> ctypes.CDLL:
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} not found: the CUDA library is required (there is no fallback); "
            "build it with `python -m rnn_transducer_loss_gb300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                            ctypes.c_size_t)
    lib.rnnt_workspace_size.argtypes = [i32, i64, i32, i32, ctypes.POINTER(sz)]
    lib.rnnt_workspace_size.restype = i32
    lib.rnnt_loss_fused.argtypes = [P, i32, i64, i32, P, i32, P, P, i32, i32, f32, i32, i32,
                                    P, P, P, P, sz, P, P]
    lib.rnnt_loss_fused.restype = i32
    lib.rnnt_workspace_size_ex.argtypes = [i32, i64, i32, i32, ctypes.POINTER(Options),
                                           ctypes.POINTER(sz)]
    lib.rnnt_workspace_size_ex.restype = i32
    lib.rnnt_loss_fused_ex.argtypes = lib.rnnt_loss_fused.argtypes + [ctypes.POINTER(Options)]
    lib.rnnt_loss_fused_ex.restype = i32
    lib.rnnt_loss_fused_staged.argtypes = lib.rnnt_loss_fused.argtypes + [P]
    lib.rnnt_loss_fused_staged.restype = i32
    lib.rnnt_loss_fused_noalloc.argtypes = lib.rnnt_loss_fused.argtypes[:16] + [P, P]
    lib.rnnt_loss_fused_noalloc.restype = i32
    lib.rnnt_grad_scale.argtypes = [P, i32, i64, i32, i32, P, sz, P, i32, P]
    lib.rnnt_grad_scale.restype = i32
    lib.rnnt_selftest_wait_timeout.argtypes = [P, i32, P]
    lib.rnnt_selftest_wait_timeout.restype = i32
    lib.rnnt_set_trace.argtypes = [P, sz]
    lib.rnnt_set_trace.restype = i32
    lib.rnnt_status_string.argtypes = [i32]
    lib.rnnt_status_string.restype = ctypes.c_char_p
    lib.rnnt_abi_version.argtypes = []
    lib.rnnt_abi_version.restype = i32
    lib.rnnt_plan.argtypes = [i32, i64, i32, i32, i32, i32, i32, ctypes.POINTER(Options),
                              ctypes.POINTER(Plan)]
    lib.rnnt_plan.restype = i32
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load().rnnt_status_string(int(code)).decode()


def abi_version() -> int:
    return int(load().rnnt_abi_version())


def rnnt_workspace_size(B: int, rows: int, V: int, dt: int) -> int:
    out = ctypes.c_size_t(0)
    rc = load().rnnt_workspace_size(B, rows, V, dt, ctypes.byref(out))
    if rc != RNNT_OK:
        raise RNNTError(rc, "rnnt_workspace_size")
    return int(out.value)


def rnnt_workspace_size_ex(B: int, rows: int, V: int, dt: int, **options) -> int:
    """Workspace bytes of rnnt_loss_fused_ex; options as make_options."""
    out = ctypes.c_size_t(0)
    opt = make_options(**options)
    rc = load().rnnt_workspace_size_ex(B, rows, V, dt, ctypes.byref(opt), ctypes.byref(out))
    if rc != RNNT_OK:
        raise RNNTError(rc, "rnnt_workspace_size_ex")
    return int(out.value)


def rnnt_loss_fused(logits, dt, rows, V, targets, targets_stride, logit_lengths, target_lengths,
                    B, blank, clamp, fused_log_softmax, reduction, loss, loss_reduced, grad,
                    workspace, workspace_bytes, status_dev, stream) -> int:
    """Raw call; pointer arguments are integers (device addresses) or None."""
    return int(load().rnnt_loss_fused(logits, dt, rows, V, targets, targets_stride,
                                      logit_lengths, target_lengths, B, blank, float(clamp),
                                      int(fused_log_softmax), reduction, loss, loss_reduced, grad,
                                      workspace, workspace_bytes, status_dev, stream))


def rnnt_loss_fused_ex(logits, dt, rows, V, targets, targets_stride, logit_lengths, target_lengths,
                       B, blank, clamp, fused_log_softmax, reduction, loss, loss_reduced, grad,
                       workspace, workspace_bytes, status_dev, stream, fastemit_lambda=0.0,
                       padded=None, big_blanks=(), sigma=0.0) -> int:
    """rnnt_loss_fused with options (make_options): padded = (max_T, max_U) selects the
    padded layout, big_blanks = [(index, duration), ...] and sigma the multi-blank loss."""
    opt = make_options(fastemit_lambda, padded, big_blanks, sigma)
    return int(load().rnnt_loss_fused_ex(logits, dt, rows, V, targets, targets_stride,
                                         logit_lengths, target_lengths, B, blank, float(clamp),
                                         int(fused_log_softmax), reduction, loss, loss_reduced,
                                         grad, workspace, workspace_bytes, status_dev, stream,
                                         ctypes.byref(opt)))


def rnnt_loss_fused_staged(logits, dt, rows, V, targets, targets_stride, logit_lengths,
                           target_lengths, B, blank, clamp, fused_log_softmax, reduction, loss,
                           loss_reduced, grad, workspace, workspace_bytes, status_dev, stream,
                           stage_events) -> int:
    """rnnt_loss_fused recording 7 caller-owned CUDA events (raw handles) at stage boundaries."""
    arr = (ctypes.c_void_p * 7)(*[ctypes.c_void_p(e) if e else None for e in stage_events])
    return int(load().rnnt_loss_fused_staged(logits, dt, rows, V, targets, targets_stride,
                                             logit_lengths, target_lengths, B, blank,
                                             float(clamp), int(fused_log_softmax), reduction,
                                             loss, loss_reduced, grad, workspace,
                                             workspace_bytes, status_dev, stream, arr))


def rnnt_loss_fused_noalloc(logits, dt, rows, V, targets, targets_stride, logit_lengths,
                            target_lengths, B, blank, clamp, fused_log_softmax, reduction, loss,
                            loss_reduced, grad, status_dev, stream) -> int:
    """rnnt_loss_fused over the library's fixed device scratch (no workspace argument)."""
    return int(load().rnnt_loss_fused_noalloc(logits, dt, rows, V, targets, targets_stride,
                                              logit_lengths, target_lengths, B, blank,
                                              float(clamp), int(fused_log_softmax), reduction,
                                              loss, loss_reduced, grad, status_dev, stream))


def rnnt_grad_scale(grad, dt, rows, V, B, workspace, workspace_bytes, factors, per_sample,
                    stream) -> int:
    return int(load().rnnt_grad_scale(grad, dt, rows, V, B, workspace, workspace_bytes, factors,
                                      int(per_sample), stream))


def rnnt_set_trace(buffer, nbytes) -> int:
    return int(load().rnnt_set_trace(buffer, nbytes))


def rnnt_selftest_wait_timeout(status_dev, polls, stream) -> int:
    """Runs the bounded-wait diagnostic; status_dev receives RNNT_TIMEOUT."""
    return int(load().rnnt_selftest_wait_timeout(status_dev, int(polls), stream))


def rnnt_plan(B, rows, V, dt, targets_stride, fused_log_softmax, want_grad=True,
              **options) -> dict:
    """{'persistent': bool, 'launches': int} for a call of this shape on the
    current device (options as make_options)."""
    plan = Plan()
    opt = make_options(**options) if options else None
    rc = load().rnnt_plan(B, rows, V, dt, targets_stride, int(bool(fused_log_softmax)),
                          int(bool(want_grad)), ctypes.byref(opt) if opt is not None else None,
                          ctypes.byref(plan))
    if rc != RNNT_OK:
        raise RNNTError(rc, "rnnt_plan")
    return {"persistent": bool(plan.persistent), "launches": int(plan.launches)}
