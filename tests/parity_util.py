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
    """Relative loss error within the dtype's bound.  A loss that is exactly 0
    (a lattice with one possible alignment of probability 1, e.g. V = 1) has
    no relative error; there the bound applies to |got| itself."""
    tol = TOL[dtype]["loss_rel"]
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    zero = want == 0.0
    err = np.where(zero, np.abs(got), np.abs(got - want) / np.where(zero, 1.0, np.abs(want)))
    i = int(np.argmax(err))
    assert np.all(err <= tol), (f"loss rel err {err.max():.3e} > {tol} at {i}: "
                                f"got {got.reshape(-1)[i]!r} want {want.reshape(-1)[i]!r}")


def assert_grad_close(got, want, dtype, what="grad"):
    tol = TOL[dtype]["grad_abs"]
    err = np.abs(np.asarray(got, dtype=np.float64) - want)
    i = np.unravel_index(np.argmax(err), err.shape)
    assert err.max() <= tol, f"{what} abs err {err.max():.3e} > {tol} at {i}: got " \
                             f"{np.asarray(got)[i]!r} want {want[i]!r}"


def every_row_compare(wl: W.Workload, block_elems: int = 1 << 24, **over):
    """Run the CUDA path once on the whole workload (the launch the benchmark
    times), then compare every per-sample loss, the reduced loss and every
    gradient element with the oracle, sample by sample and in row blocks, so
    that the float64 reference of a multi-GB gradient is never held at once."""
    cfg = wl.cfg
    kw = dict(blank=cfg.blank, clamp=cfg.clamp, reduction=cfg.reduction,
              fused_log_softmax=cfg.fused)
    kw.update(over)
    loss, red, grad = gpu_run(wl, **over)
    gl = to_np(loss)
    dt = cfg.dtype
    scale = 1.0 / cfg.B if kw["reduction"] == "mean" else 1.0
    block = max(1, block_elems // cfg.V)
    ref = np.empty(cfg.B)
    for b in range(cfg.B):
        sl = wl.sample_rows(b)
        x = to_np(wl.logits[sl])
        T, U = int(wl.T[b]), int(wl.U[b])
        fw = oracle.sample_forward(x, T, U, wl.targets[b], kw["blank"], kw["fused_log_softmax"])
        ref[b] = fw.loss_alpha
        assert_loss_close([gl[b]], [fw.loss_alpha], dt)
        n = sl.stop - sl.start
        gs = grad[sl]
        for r0 in range(0, n, block):
            r1 = min(n, r0 + block)
            want = oracle.sample_grad(x, fw, wl.targets[b], kw["blank"], kw["fused_log_softmax"],
                                      kw["clamp"], scale, r0, r1)
            assert_grad_close(to_np(gs[r0:r1].float()), want, dt,
                              f"sample {b} (T={T}, U={U}) rows {r0}..{r1}")
        del x, gs
    if kw["reduction"] != "none":
        assert_loss_close([float(red)], [ref.sum() * scale], dt)
    return loss, red, grad, ref
