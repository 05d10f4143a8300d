"""GPU parity of the multi-blank transducer (rnnt_loss_fused_ex with big
blanks and the under-normalisation sigma; ESPnet compute_multiblank_grad_kernel
docs) against the float64 oracle on the same seeded inputs."""
import math

import numpy as np
import pytest
import torch

import oracle
from rnn_transducer_loss_gb300 import workloads as W
from rnn_transducer_loss_gb300.functional import rnnt_loss, rnnt_loss_forward

from parity_util import assert_grad_close, assert_loss_close, gpu_run, to_np

pytestmark = pytest.mark.gpu


def mb_workload(seed, B, Tmax, Umax, V, K, dtype="f32", fused=True, Tmin=1, **kw):
    """Random lengths; blank = V-1, big blanks V-2 .. V-1-K, labels below them."""
    rng = np.random.default_rng(seed)
    wl = W.custom(B, rng.integers(Tmin, Tmax + 1, size=B), rng.integers(0, Umax + 1, size=B), V,
                  dtype=dtype, fused=fused, blank=-1, seed=seed, device="cuda", **kw)
    wl.targets[:] = wl.targets % (V - 1 - K)
    big = [(V - 2 - i, [2, 4, 8][i % 3]) for i in range(K)]
    return wl, big


def compare(wl, big, sigma=0.0, fe=0.0, tol_dtype=None):
    cfg = wl.cfg
    loss, red, grad = gpu_run(wl, big_blanks=big, sigma=sigma, fastemit_lambda=fe)
    ref = oracle.rnnt_loss_multiblank(to_np(wl.logits), wl.targets, wl.T, wl.U, big,
                                      blank=cfg.blank, sigma=sigma, clamp=cfg.clamp,
                                      reduction=cfg.reduction, fused_log_softmax=cfg.fused,
                                      fastemit_lambda=fe)
    dt = tol_dtype or cfg.dtype
    assert_loss_close(to_np(loss), ref.losses, dt)
    if cfg.reduction != "none":
        assert_loss_close([float(red)], [ref.reduced], dt)
    assert_grad_close(to_np(grad.float()), ref.grad, dt)
    return loss, grad, ref


CASES = [
    dict(V=29, K=1, dtype="f32", fused=True, clamp=-1.0, reduction="sum", sigma=0.0),
    dict(V=64, K=2, dtype="f32", fused=True, clamp=0.2, reduction="mean", sigma=0.05),
    dict(V=64, K=3, dtype="f32", fused=False, clamp=-1.0, reduction="none", sigma=0.1),
    dict(V=512, K=2, dtype="f16", fused=True, clamp=-1.0, reduction="sum", sigma=0.05),
    dict(V=1024, K=3, dtype="bf16", fused=True, clamp=-1.0, reduction="mean", sigma=0.0),
    dict(V=37, K=1, dtype="f16", fused=False, clamp=0.5, reduction="sum", sigma=0.2),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_multiblank_elementwise(case):
    kw = dict(CASES[case])
    sigma = kw.pop("sigma")
    wl, big = mb_workload(500 + case, B=5, Tmax=60, Umax=25, sigma=1.3, **kw)
    compare(wl, big, sigma=sigma)


def test_multiblank_fastemit():
    wl, big = mb_workload(520, B=4, Tmax=50, Umax=20, V=64, K=2, reduction="sum", sigma=1.2)
    compare(wl, big, sigma=0.05, fe=0.7)


def test_multiblank_long_lattice_precision():
    # about 700 anti-diagonals of extended-range products, fp32 tolerances
    wl, big = mb_workload(521, B=2, Tmax=600, Umax=100, V=48, K=2, Tmin=550, reduction="sum",
                          sigma=1.0)
    compare(wl, big, sigma=0.02)


def test_sigma_alone_shifts_the_standard_loss():
    # No big blank: every alignment has T+U emissions, so the loss grows by
    # (T+U) sigma and the gradient is the standard one.
    wl, _ = mb_workload(522, B=4, Tmax=40, Umax=15, V=29, K=0, reduction="none", sigma=1.5)
    l0, _, g0 = gpu_run(wl)
    l1, _, g1 = gpu_run(wl, sigma=0.3)
    shift = 0.3 * (wl.T.astype(np.float64) + wl.U)
    assert_loss_close(to_np(l1).astype(np.float64) - shift, to_np(l0).astype(np.float64), "f32")
    assert_grad_close(to_np(g1), to_np(g0).astype(np.float64), "f32")


def test_multiblank_padded_and_autograd():
    wl, big = mb_workload(523, B=3, Tmax=30, Umax=10, V=64, K=2, reduction="none", sigma=1.0)
    ref = oracle.rnnt_loss_multiblank(to_np(wl.logits), wl.targets, wl.T, wl.U, big, blank=-1,
                                      sigma=0.1, reduction="none")
    xp = W.to_padded(wl, fill=float("nan"))
    d = "cuda"
    y, Tl, Ul = (torch.as_tensor(a, device=d) for a in (wl.targets, wl.T, wl.U))
    x = xp.clone().requires_grad_(True)
    out = rnnt_loss(x, y, Tl, Ul, blank=-1, reduction="none", big_blanks=big, sigma=0.1)
    assert_loss_close(to_np(out), ref.losses, "f32")
    w = torch.tensor([0.5, -2.0, 3.0], device=d)
    (out * w).sum().backward()
    g = to_np(x.grad)
    for b in range(3):
        T, U = int(wl.T[b]), int(wl.U[b])
        want = ref.grad[wl.sample_rows(b)].reshape(T, U + 1, -1) * float(w[b])
        assert_grad_close(g[b, :T, :U + 1], want, "f32", f"sample {b}")
        assert not np.any(g[b, T:]) and not np.any(g[b, :, U + 1:])


def test_multiblank_label_equal_to_a_big_blank_is_rejected():
    wl = W.custom(2, [6, 7], [3, 2], 16, blank=-1, reduction="sum", seed=524, device="cuda")
    big = [(14, 2), (13, 4)]
    wl.targets[:] = wl.targets % 13
    wl.targets[0, 0] = 13
    d = "cuda"
    with pytest.raises(ValueError):
        rnnt_loss_forward(wl.logits, torch.as_tensor(wl.targets, device=d),
                          torch.as_tensor(wl.T, device=d), torch.as_tensor(wl.U, device=d),
                          blank=-1, reduction="sum", big_blanks=big)
