"""Float64 CPU oracle for the RNN-T loss on the compact 2D logit layout.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the product package.  It
shares no code with the CUDA path: the arithmetic lives in ``rnnt_oracle.c``
(plain loops in double precision) and in ``brute.py`` (enumeration of every
alignment, for tiny lattices).

Semantics follow torchaudio.functional.rnnt_loss as restated by the
rnnt-loss-ascend README (sections "参数说明", "约束说明"): per-sample rows
``T_b*(U_b+1)`` concatenated in batch order, ``blank`` in [-V, V-1],
``clamp <= 0`` disables clipping, ``reduction`` in none/sum/mean (mean is the
batch mean, README "调用说明" example), ``fused_log_softmax`` selects
raw logits (True) or log-probabilities (False).

Parity status: every function here is pinned in ``tests/test_oracle_pins.py``
by brute-force enumeration, closed forms (T=1 and U=0 lattices, uniform
logits), invariants (alpha/beta loss agreement, per-diagonal occupancy, zero
row sums) and central finite differences.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rnnt_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_rnnt.so")
_lib = None

F32, F16, F64 = 0, 1, 2
_RED = {"none": 0, "sum": 1, "mean": 2}


def build(force: bool = False) -> str:
    """Compile rnnt_oracle.c into a shared library next to it (gcc, OpenMP when available)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=gnu11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    i32, i64, dbl = ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.rnnt_oracle_offsets.argtypes = [i32, P, P, P]
    lib.rnnt_oracle_offsets.restype = None
    lib.rnnt_oracle_forward.argtypes = [P, i32, i32, i32, i32, P, i32, i32, P, P, P, P, P]
    lib.rnnt_oracle_forward.restype = i32
    lib.rnnt_oracle_grad.argtypes = [P, i32, i32, i32, i32, P, i32, i32, P, P, P, P, dbl, dbl,
                                     dbl, i64, i64, P]
    lib.rnnt_oracle_grad.restype = i32
    lib.rnnt_oracle_batch.argtypes = [P, i32, i64, i32, P, i32, P, P, i32, i32, dbl, i32, i32,
                                      dbl, P, P, P, P]
    lib.rnnt_oracle_batch.restype = i32
    lib.rnnt_oracle_num_threads.argtypes = []
    lib.rnnt_oracle_num_threads.restype = i32
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(x: np.ndarray) -> int:
    if x.dtype == np.float32:
        return F32
    if x.dtype == np.float16:
        return F16
    if x.dtype == np.float64:
        return F64
    raise TypeError(f"oracle takes float32, float16 or float64 rows, got {x.dtype}")


def _labels(y, U: int) -> np.ndarray:
    if U <= 0:
        return np.zeros(1, dtype=np.int32)
    return np.ascontiguousarray(np.asarray(y, dtype=np.int32).reshape(-1)[:U])


def num_threads() -> int:
    return int(_load().rnnt_oracle_num_threads())


def offsets(logit_lengths, target_lengths) -> np.ndarray:
    """First row of every sample (exclusive prefix sum of T*(U+1)), int64, B+1 entries."""
    T = np.ascontiguousarray(logit_lengths, dtype=np.int32)
    U = np.ascontiguousarray(target_lengths, dtype=np.int32)
    off = np.zeros(T.shape[0] + 1, dtype=np.int64)
    _load().rnnt_oracle_offsets(T.shape[0], _ptr(T), _ptr(U), _ptr(off))
    return off


@dataclass
class SampleForward:
    """Forward quantities of one sample, arrays in (t, u) row order, natural log."""
    T: int
    U: int
    lpb: np.ndarray
    lpy: np.ndarray
    alpha: np.ndarray
    beta: np.ndarray
    loss_alpha: float
    loss_beta: float

    @property
    def ll(self) -> float:
        return -self.loss_alpha


def sample_forward(x: np.ndarray, T: int, U: int, y, blank: int, fused: bool) -> SampleForward:
    """Log-probs, alpha, beta and both losses of one sample; x is its (T*(U+1), V) block."""
    x = np.ascontiguousarray(x)
    V = x.shape[1]
    n = T * (U + 1)
    if x.ndim != 2 or x.shape[0] != n:
        raise ValueError(f"sample block must have T*(U+1) = {n} rows, got {x.shape}")
    yy = _labels(y, U)
    lpb, lpy, al, be = (np.empty(n) for _ in range(4))
    ls = np.empty(2)
    rc = _load().rnnt_oracle_forward(_ptr(x), _dtype_code(x), V, T, U, _ptr(yy), blank,
                                     int(bool(fused)), _ptr(lpb), _ptr(lpy), _ptr(al), _ptr(be),
                                     _ptr(ls))
    if rc != 0:
        raise ValueError("oracle forward rejected its arguments")
    return SampleForward(T, U, lpb, lpy, al, be, float(ls[0]), float(ls[1]))


def sample_grad(x: np.ndarray, fw: SampleForward, y, blank: int, fused: bool, clamp: float,
                scale: float, r0: int = 0, r1: int | None = None,
                fastemit_lambda: float = 0.0) -> np.ndarray:
    """Gradient rows [r0, r1) of one sample (float64, (r1-r0, V))."""
    x = np.ascontiguousarray(x)
    V = x.shape[1]
    n = fw.T * (fw.U + 1)
    r1 = n if r1 is None else r1
    yy = _labels(y, fw.U)
    g = np.empty((r1 - r0, V))
    rc = _load().rnnt_oracle_grad(_ptr(x), _dtype_code(x), V, fw.T, fw.U, _ptr(yy), blank,
                                  int(bool(fused)), _ptr(fw.lpb), _ptr(fw.lpy), _ptr(fw.alpha),
                                  _ptr(fw.beta), float(clamp), float(scale),
                                  float(fastemit_lambda), r0, r1, _ptr(g))
    if rc != 0:
        raise ValueError("oracle grad rejected its arguments")
    return g


@dataclass
class BatchResult:
    losses: np.ndarray          # per-sample loss from alpha (float64, B)
    losses_beta: np.ndarray     # per-sample loss from beta (float64, B)
    reduced: float              # sum or mean over the batch
    grad: np.ndarray | None     # (rows, V) float64


def rnnt_loss(logits: np.ndarray, targets, logit_lengths, target_lengths, blank: int = -1,
              clamp: float = -1.0, reduction: str = "mean", fused_log_softmax: bool = True,
              want_grad: bool = True, fastemit_lambda: float = 0.0) -> BatchResult:
    """Whole-batch oracle; samples run in parallel on the host cores.

    ``fastemit_lambda`` (>= 0) scales the gradient of every label-emission
    log-probability by 1 + lambda (FastEmit); the losses do not depend on it.
    """
    x = np.ascontiguousarray(logits)
    rows, V = x.shape
    tg = np.ascontiguousarray(np.asarray(targets, dtype=np.int32))
    if tg.ndim == 1:
        tg = tg.reshape(1, -1)
    if tg.shape[1] == 0:
        tg = np.zeros((tg.shape[0], 1), dtype=np.int32)
    T = np.ascontiguousarray(logit_lengths, dtype=np.int32)
    U = np.ascontiguousarray(target_lengths, dtype=np.int32)
    B = T.shape[0]
    losses, losses_b = np.empty(B), np.empty(B)
    red = np.empty(1)
    grad = np.empty((rows, V)) if want_grad else None
    rc = _load().rnnt_oracle_batch(_ptr(x), _dtype_code(x), rows, V, _ptr(tg), tg.shape[1],
                                   _ptr(T), _ptr(U), B, blank, float(clamp),
                                   int(bool(fused_log_softmax)), _RED[reduction],
                                   float(fastemit_lambda), _ptr(losses),
                                   _ptr(losses_b), _ptr(red),
                                   _ptr(grad) if grad is not None else None)
    if rc != 0:
        raise ValueError("oracle batch rejected its arguments")
    return BatchResult(losses, losses_b, float(red[0]), grad)


def rnnt_loss_padded(logits: np.ndarray, targets, logit_lengths, target_lengths,
                     **kw) -> BatchResult:
    """Oracle on the padded (B, max_T, max_U+1, V) layout of the ESPnet GPURNNT docs.

    Node (t, u) of sample b is ``logits[b, t, u]``; entries with t >= T_b or
    u > U_b belong to no lattice, are never read and get a zero gradient.
    The lattices are gathered into the compact layout, ``rnnt_loss`` (or,
    with ``big_blanks``, ``rnnt_loss_multiblank``) runs on it, and the
    gradient is scattered back into a zero (B, max_T, max_U+1, V) array.
    Keyword arguments are those of that function.
    """
    x = np.asarray(logits)
    if x.ndim != 4:
        raise ValueError("padded logits must be (B, max_T, max_U+1, V)")
    B, maxT, maxW, V = x.shape
    T = np.asarray(logit_lengths, dtype=np.int64)
    U = np.asarray(target_lengths, dtype=np.int64)
    if T.shape[0] != B or (T > maxT).any() or (U + 1 > maxW).any():
        raise ValueError("lengths do not fit the padded tensor")
    compact = np.concatenate([x[b, :T[b], :U[b] + 1, :].reshape(-1, V) for b in range(B)])
    if kw.get("big_blanks") or kw.get("sigma"):
        big = kw.pop("big_blanks", [])
        res = rnnt_loss_multiblank(compact, targets, T.astype(np.int32), U.astype(np.int32), big,
                                   **kw)
    else:
        kw.pop("big_blanks", None)
        kw.pop("sigma", None)
        res = rnnt_loss(compact, targets, T.astype(np.int32), U.astype(np.int32), **kw)
    if res.grad is not None:
        g = np.zeros((B, maxT, maxW, V))
        r = 0
        for b in range(B):
            n = int(T[b] * (U[b] + 1))
            g[b, :T[b], :U[b] + 1, :] = res.grad[r:r + n].reshape(int(T[b]), int(U[b]) + 1, V)
            r += n
        res.grad = g
    return res


def rnnt_loss_multiblank(logits: np.ndarray, targets, logit_lengths, target_lengths,
                         big_blanks, blank: int = -1, sigma: float = 0.0, clamp: float = -1.0,
                         reduction: str = "mean", fused_log_softmax: bool = True,
                         want_grad: bool = True, fastemit_lambda: float = 0.0) -> BatchResult:
    """Multi-blank transducer loss on the compact layout (ESPnet
    compute_multiblank_grad_kernel docs): ``big_blanks`` is a list of
    (output index, duration >= 2) pairs, ``sigma`` the logit
    under-normalisation subtracted from every log-probability.  Sample by
    sample in float64 (``rnnt_oracle_mb_sample``); with no big blanks and
    sigma = 0 it is the standard transducer loss."""
    lib = _load()
    if not hasattr(lib, "_mb_ready"):
        P, i32, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
        lib.rnnt_oracle_mb_sample.argtypes = [P, i32, i32, i32, i32, P, i32, i32, i32, P, P, dbl,
                                              dbl, dbl, dbl, P, P]
        lib.rnnt_oracle_mb_sample.restype = i32
        lib._mb_ready = True
    x = np.ascontiguousarray(logits)
    rows, V = x.shape
    T = np.asarray(logit_lengths, dtype=np.int64)
    U = np.asarray(target_lengths, dtype=np.int64)
    B = T.shape[0]
    off = np.zeros(B + 1, dtype=np.int64)
    off[1:] = np.cumsum(T * (U + 1))
    if off[-1] != rows:
        raise ValueError("rows != sum T*(U+1)")
    ids = np.ascontiguousarray([int(i) + (V if int(i) < 0 else 0) for i, _ in big_blanks] or [0],
                               dtype=np.int32)
    durs = np.ascontiguousarray([int(d) for _, d in big_blanks] or [0], dtype=np.int32)
    K = len(big_blanks)
    scale = 1.0 / B if reduction == "mean" else 1.0
    tg = np.asarray(targets, dtype=np.int32).reshape(B, -1)
    losses, losses_b = np.empty(B), np.empty(B)
    grad = np.empty((rows, V)) if want_grad else None
    for b in range(B):
        xb = np.ascontiguousarray(x[off[b]:off[b + 1]])
        yb = _labels(tg[b], int(U[b]))
        ls = np.empty(2)
        gb = np.empty((int(off[b + 1] - off[b]), V)) if want_grad else None
        rc = lib.rnnt_oracle_mb_sample(_ptr(xb), _dtype_code(xb), V, int(T[b]), int(U[b]),
                                       _ptr(yb), blank, int(bool(fused_log_softmax)), K,
                                       _ptr(ids), _ptr(durs), float(sigma),
                                       float(fastemit_lambda), float(clamp), scale, _ptr(ls),
                                       _ptr(gb) if gb is not None else None)
        if rc != 0:
            raise ValueError("oracle multi-blank rejected its arguments")
        losses[b], losses_b[b] = ls
        if grad is not None:
            grad[off[b]:off[b + 1]] = gb
    red = losses.sum() * (1.0 / B if reduction == "mean" else 1.0)
    return BatchResult(losses, losses_b, float(red), grad)
