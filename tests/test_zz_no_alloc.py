"""rnnt_loss_fused_noalloc (scratch in a fixed device array, no caller
workspace) against rnnt_loss_fused (caller workspace) on the same inputs.

The file name sorts last so that pytest collects it after every other test;
it also passes alone in a fresh process.  Consecutive calls share the one
scratch array, so the second call below runs over what the first left there.
"""
import os
import re

import numpy as np
import pytest
import torch

from rnn_transducer_loss_gb300 import _native as N
from rnn_transducer_loss_gb300 import workloads as W
from rnn_transducer_loss_gb300.functional import _DT

from parity_util import TOL, assert_grad_close, assert_loss_close, to_np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _inputs(wl):
    dev = wl.logits.device
    return (torch.as_tensor(wl.targets, device=dev), torch.as_tensor(wl.T, device=dev),
            torch.as_tensor(wl.U, device=dev))


def _run(wl, noalloc):
    cfg = wl.cfg
    x = wl.logits
    t, Tl, Ul = _inputs(wl)
    loss = torch.full((cfg.B,), float("nan"), dtype=torch.float32, device=x.device)
    red = torch.full((), float("nan"), dtype=torch.float32, device=x.device)
    grad = torch.full_like(x, float("nan"))
    status = torch.full((1,), -1, dtype=torch.int32, device=x.device)
    stream = torch.cuda.current_stream().cuda_stream
    common = (x.data_ptr(), _DT[x.dtype], x.shape[0], cfg.V, t.data_ptr(), t.shape[1],
              Tl.data_ptr(), Ul.data_ptr(), cfg.B, cfg.blank, cfg.clamp, int(cfg.fused),
              N.REDUCTIONS[cfg.reduction], loss.data_ptr(), red.data_ptr(), grad.data_ptr())
    if noalloc:
        rc = N.rnnt_loss_fused_noalloc(*common, status.data_ptr(), stream)
    else:
        nb = N.rnnt_workspace_size(cfg.B, x.shape[0], cfg.V, _DT[x.dtype])
        ws = torch.empty(nb, dtype=torch.uint8, device=x.device)
        rc = N.rnnt_loss_fused(*common, ws.data_ptr(), nb, status.data_ptr(), stream)
    assert rc == N.RNNT_OK, N.status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == N.RNNT_OK, N.status_string(int(status.item()))
    return loss, red, grad


def _compare(got, want, dtype):
    assert_loss_close(to_np(got[0]), to_np(want[0]), dtype)
    assert_loss_close([float(got[1])], [float(want[1])], dtype)
    assert_grad_close(to_np(got[2].float()), to_np(want[2].float()).astype(np.float64), dtype)


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point_two_calls():
    first = W.make("char_asr", "cuda")
    second = W.custom(B=3, T=[40, 17, 1], U=[12, 0, 5], V=64, dtype="f16", reduction="sum",
                      seed=11, device="cuda")
    want = [_run(wl, noalloc=False) for wl in (first, second)]
    # Two calls in a row; the second, smaller problem starts over the scratch
    # contents the first one left.
    got = [_run(wl, noalloc=True) for wl in (first, second)]
    for wl, g, w in zip((first, second), got, want):
        _compare(g, w, wl.cfg.dtype)


@pytest.mark.gpu
def test_noalloc_persistent_kernel_over_used_scratch():
    # The first four BPE-ASR samples (about 120k rows) run as the one persistent
    # kernel, whose task queue and per-sample counters live in the scratch; the
    # call before it (a per-stage shape) and a repeat of it both leave their
    # contents behind.
    bpe = W.subset(W.make("bpe_asr", "cuda"), 4)
    small = W.custom(B=3, T=[40, 17, 1], U=[12, 0, 5], V=64, dtype="f16", reduction="sum",
                     seed=11, device="cuda")
    want = _run(bpe, noalloc=False)
    _run(small, noalloc=True)
    for _ in range(2):
        _compare(_run(bpe, noalloc=True), want, bpe.cfg.dtype)


def test_noalloc_rejects_sizes_beyond_scratch():
    limit = N.NOALLOC_SCRATCH_BYTES
    rows = 10_000_000
    assert N.rnnt_workspace_size(1, rows, 8, N.RNNT_F16) > limit
    # Rejected on the host before any device work: the pointers are never used.
    rc = N.rnnt_loss_fused_noalloc(4096, N.RNNT_F16, rows, 8, 8192, 1, 8448, 8704, 1, -1, -1.0,
                                   1, 0, 8960, None, None, None, None)
    assert rc == N.RNNT_WORKSPACE_TOO_SMALL
    assert N.rnnt_loss_fused_noalloc(4096, N.RNNT_F16, 0, 8, 8192, 1, 8448, 8704, 1, -1, -1.0,
                                     1, 0, 8960, None, None, None, None) == N.RNNT_INVALID_VALUE


def test_noalloc_limit_matches_header():
    src = open(os.path.join(ROOT, "include", "rnnt_gb300.h")).read()
    m = re.search(r"#define\s+RNNT_NOALLOC_SCRATCH_BYTES\s+\(\(size_t\)(\d+)\s*<<\s*(\d+)\)", src)
    assert m, "RNNT_NOALLOC_SCRATCH_BYTES not found"
    assert N.NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))
