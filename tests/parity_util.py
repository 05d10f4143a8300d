"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and compare it with the float64 oracle on the same seeded inputs."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from rnn_transducer_loss_gb300 import workloads as W
from rnn_transducer_loss_gb300.functional import rnnt_loss_forward

# Parity tolerances against the float64 oracle: fp32 inputs loss rel 1e-5 /
# grad abs 1e-5, fp16 inputs (fp32 accumulation) loss rel 1e-3 / grad abs
# 2e-3.  bf16 storage: the same loss bound as fp16, and a gradient bound of
# two bf16 half-ulps at magnitude 1 (the gradient is rounded once to 8
# significant bits; |grad| <= 1): 2 * 2^-9 ~ 4e-3.
TOL = {"f32": dict(loss_rel=1e-5, grad_abs=1e-5), "f16": dict(loss_rel=1e-3, grad_abs=2e-3),
       "bf16": dict(loss_rel=1e-3, grad_abs=4e-3)}


def to_np(x: torch.Tensor) -> np.ndarray:
    # bfloat16 has no numpy type; widening it to float32 is exact.
    x = x.detach()
    return (x.float() if x.dtype == torch.bfloat16 else x).cpu().numpy()


def gpu_run(wl: W.Workload, device="cuda", want_grad=True, inplace=False, **over):
    cfg = wl.cfg
    kw = dict(blank=cfg.blank, clamp=cfg.clamp, reduction=cfg.reduction,
              fused_log_softmax=cfg.fused)
    kw.update(over)
    x = wl.logits if wl.logits.is_cuda else wl.logits.to(device)
    if inplace:
        x = x.clone()
    loss, red, grad, _ = rnnt_loss_forward(
        x, torch.as_tensor(wl.targets, device=device), torch.as_tensor(wl.T, device=device),
        torch.as_tensor(wl.U, device=device), want_grad=want_grad, inplace_grad=inplace, **kw)
    torch.cuda.synchronize()
    return loss, red, grad


def oracle_full(wl: W.Workload, **over):
    cfg = wl.cfg
    kw = dict(blank=cfg.blank, clamp=cfg.clamp, reduction=cfg.reduction,
              fused_log_softmax=cfg.fused)
    kw.update(over)
    return oracle.rnnt_loss(to_np(wl.logits), wl.targets, wl.T, wl.U, **kw)


def assert_loss_close(got, want, dtype):
    tol = TOL[dtype]["loss_rel"]
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    # Relative error; below a loss of 1 nat the bound applies as an absolute one.
    err = np.abs(got - want) / np.maximum(np.abs(want), 1.0)
    assert np.all(err <= tol), f"loss rel err {err.max():.3e} > {tol}"


def assert_grad_close(got, want, dtype, what="grad"):
    tol = TOL[dtype]["grad_abs"]
    err = np.abs(np.asarray(got, dtype=np.float64) - want)
    i = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= tol, f"{what} abs err {err.max():.3e} > {tol} at {i}: got " \
                             f"{np.asarray(got)[i]!r} want {want[i]!r}"


def sampled_rows(wl: W.Workload, per_sample: int, seed: int = 0):
    """Per sample: row ids (relative) including the first, last and some random rows."""
    rng = np.random.default_rng(seed)
    out = {}
    for b in range(wl.cfg.B):
        n = int(wl.offsets[b + 1] - wl.offsets[b])
        k = min(n, per_sample)
        ids = set(rng.choice(n, size=k, replace=False).tolist()) | {0, n - 1}
        out[b] = np.array(sorted(ids), dtype=np.int64)
    return out
