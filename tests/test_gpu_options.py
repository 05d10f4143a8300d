"""GPU parity of the call's options (rnnt_loss_fused_ex): the FastEmit weight
and the padded (B, max_T, max_U+1, V) layout of the ESPnet GPURNNT docs, each
against the float64 oracle on the same seeded inputs, on the persistent
kernel and on the per-stage kernels."""
import numpy as np
import pytest
import torch

import oracle
from rnn_transducer_loss_gb300 import workloads as W
from rnn_transducer_loss_gb300 import _native as N
from rnn_transducer_loss_gb300.functional import rnnt_loss, rnnt_loss_forward

from parity_util import assert_grad_close, assert_loss_close, gpu_run, oracle_full, to_np

pytestmark = pytest.mark.gpu


def make(B, T, U, V, **kw):
    return W.custom(B, T, U, V, device="cuda", **kw)


def rand_wl(seed, B, Tmax, Umax, V, **kw):
    rng = np.random.default_rng(seed)
    return make(B, rng.integers(1, Tmax + 1, size=B), rng.integers(0, Umax + 1, size=B), V,
                seed=seed, **kw)


def run_padded(wl, xp, **over):
    cfg = wl.cfg
    kw = dict(blank=cfg.blank, clamp=cfg.clamp, reduction=cfg.reduction,
              fused_log_softmax=cfg.fused)
    kw.update(over)
    d = "cuda"
    loss, red, grad, _ = rnnt_loss_forward(xp, torch.as_tensor(wl.targets, device=d),
                                           torch.as_tensor(wl.T, device=d),
                                           torch.as_tensor(wl.U, device=d), **kw)
    torch.cuda.synchronize()
    return loss, red, grad


# Cases: the persistent kernel's TMA path (16-byte rows of 33..256 vectors),
# its plain non-fused path, and the per-stage kernels (V*s not 16-byte aligned).
CASES = [
    dict(V=1024, dtype="f16", fused=True, blank=-1, clamp=-1.0, reduction="sum"),
    dict(V=264, dtype="f32", fused=True, blank=0, clamp=0.3, reduction="mean"),
    dict(V=512, dtype="f16", fused=False, blank=-1, clamp=0.5, reduction="mean"),
    dict(V=29, dtype="f32", fused=True, blank=0, clamp=0.1, reduction="none"),
    dict(V=37, dtype="f16", fused=False, blank=5, clamp=-1.0, reduction="sum"),
]


# ------------------------------------------------------------------ FastEmit
@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("lam", [0.5, 2.0])
def test_fastemit_elementwise(case, lam):
    wl = rand_wl(60 + case, B=5, Tmax=80, Umax=40, sigma=1.4, **CASES[case])
    loss, red, grad = gpu_run(wl, fastemit_lambda=lam)
    ref = oracle_full(wl, fastemit_lambda=lam)
    assert_loss_close(to_np(loss), ref.losses, wl.cfg.dtype)
    assert_grad_close(to_np(grad.float()), ref.grad, wl.cfg.dtype)


def test_fastemit_zero_is_the_plain_call():
    wl = rand_wl(70, B=4, Tmax=60, Umax=30, V=512, dtype="f16", sigma=1.2)
    a = gpu_run(wl)
    b = gpu_run(wl, fastemit_lambda=0.0)
    d = "cuda"
    args = (torch.as_tensor(wl.targets, device=d), torch.as_tensor(wl.T, device=d),
            torch.as_tensor(wl.U, device=d))
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    # ... and through rnnt_loss_fused_ex with an explicit zero weight
    loss, red, grad, ws = rnnt_loss_forward(wl.logits, *args, blank=-1, reduction="mean",
                                            fastemit_lambda=1e-30)
    assert torch.equal(loss, a[0])


@pytest.mark.parametrize("sched", ["persistent", "kernels"])
def test_fastemit_schedules_agree(sched, monkeypatch):
    wl = rand_wl(71, B=6, Tmax=90, Umax=70, V=1024, dtype="f16", sigma=1.3, reduction="sum")
    if sched == "kernels":
        monkeypatch.setenv("RNNT_GB300_SCHEDULE", "kernels")
    got = gpu_run(wl, fastemit_lambda=0.8)
    monkeypatch.delenv("RNNT_GB300_SCHEDULE", raising=False)
    ref = gpu_run(wl, fastemit_lambda=0.8)
    for x, y in zip(got, ref):
        assert torch.equal(x, y)


def test_fastemit_bpe_asr_sampled():
    wl = W.subset(W.make("bpe_asr", "cuda"), 4)
    lam = 0.01   # a typical FastEmit weight
    loss, red, grad = gpu_run(wl, fastemit_lambda=lam)
    ref = oracle_full(wl, fastemit_lambda=lam)
    assert_loss_close(to_np(loss), ref.losses, "f16")
    assert_grad_close(to_np(grad.float()), ref.grad, "f16")


# ------------------------------------------------------------------ padded layout
@pytest.mark.parametrize("case", range(len(CASES)))
def test_padded_elementwise(case):
    wl = rand_wl(80 + case, B=5, Tmax=70, Umax=35, sigma=1.4, **CASES[case])
    xp = W.to_padded(wl, max_T=int(wl.T.max()) + 3, max_U=int(wl.U.max()) + 2, fill=30.0)
    loss, red, grad = run_padded(wl, xp)
    ref = oracle.rnnt_loss_padded(to_np(xp), wl.targets, wl.T, wl.U, blank=wl.cfg.blank,
                                  clamp=wl.cfg.clamp, reduction=wl.cfg.reduction,
                                  fused_log_softmax=wl.cfg.fused)
    assert grad.shape == xp.shape
    assert_loss_close(to_np(loss), ref.losses, wl.cfg.dtype)
    assert_grad_close(to_np(grad.float()), ref.grad, wl.cfg.dtype)


@pytest.mark.parametrize("case", range(len(CASES)))
def test_padded_equals_compact_bit_for_bit(case):
    # Same lattice bytes in either layout: identical losses and gradients, and
    # exact zeros at every padded position (NaN padding is never read).
    wl = rand_wl(90 + case, B=4, Tmax=50, Umax=30, sigma=1.2, **CASES[case])
    xp = W.to_padded(wl, max_T=int(wl.T.max()) + 1, max_U=int(wl.U.max()) + 1,
                     fill=float("nan"))
    lp, rp, gp = run_padded(wl, xp)
    lc, rc, gc = gpu_run(wl)
    assert torch.equal(lp, lc) and torch.equal(rp, rc)
    for b in range(wl.cfg.B):
        T, U = int(wl.T[b]), int(wl.U[b])
        assert torch.equal(gp[b, :T, :U + 1].reshape(-1, wl.cfg.V), gc[wl.sample_rows(b)])
        assert not gp[b, T:].any() and not gp[b, :, U + 1:].any()


@pytest.mark.parametrize("sched", ["persistent", "kernels"])
def test_padded_fastemit_schedules(sched, monkeypatch):
    wl = rand_wl(100, B=6, Tmax=60, Umax=40, V=1024, dtype="f16", sigma=1.3, reduction="mean",
                 clamp=0.2)
    xp = W.to_padded(wl, fill=-7.0)
    if sched == "kernels":
        monkeypatch.setenv("RNNT_GB300_SCHEDULE", "kernels")
    loss, red, grad = run_padded(wl, xp, fastemit_lambda=0.3)
    ref = oracle.rnnt_loss_padded(to_np(xp), wl.targets, wl.T, wl.U, blank=-1, clamp=0.2,
                                  reduction="mean", fastemit_lambda=0.3)
    assert_loss_close(to_np(loss), ref.losses, "f16")
    assert_grad_close(to_np(grad.float()), ref.grad, "f16")


def test_padded_inplace_and_autograd():
    wl = rand_wl(110, B=3, Tmax=30, Umax=12, V=64, dtype="f32", reduction="none")
    xp = W.to_padded(wl, fill=3.0)
    ref = oracle.rnnt_loss_padded(to_np(xp), wl.targets, wl.T, wl.U, blank=-1,
                                  reduction="none")
    d = "cuda"
    y, Tl, Ul = (torch.as_tensor(a, device=d) for a in (wl.targets, wl.T, wl.U))
    # in place: the gradient overwrites the padded logits (padding included)
    xi = xp.clone()
    _, _, gi, _ = rnnt_loss_forward(xi, y, Tl, Ul, blank=-1, reduction="none", inplace_grad=True)
    assert gi.data_ptr() == xi.data_ptr()
    assert_grad_close(to_np(xi), ref.grad, "f32")
    # autograd with per-sample upstream factors (rnnt_grad_scale on the padded layout)
    x = xp.clone().requires_grad_(True)
    out = rnnt_loss(x, y, Tl, Ul, blank=-1, reduction="none")
    w = torch.tensor([0.5, -2.0, 3.0], device=d)
    (out * w).sum().backward()
    want = ref.grad * to_np(w).reshape(3, 1, 1, 1)
    assert_grad_close(to_np(x.grad), want, "f32")


def test_padded_lengths_beyond_the_tensor_are_rejected():
    wl = make(2, [5, 4], [2, 3], 7, dtype="f32", blank=0, reduction="sum")
    xp = W.to_padded(wl)
    d = "cuda"
    T = torch.as_tensor([6, 4], dtype=torch.int32, device=d)   # T_0 > max_T
    with pytest.raises(ValueError):
        rnnt_loss_forward(xp, torch.as_tensor(wl.targets, device=d), T,
                          torch.as_tensor(wl.U, device=d), blank=0, reduction="sum")


# ------------------------------------------------------------------ bfloat16 storage
BF16_CASES = [
    dict(V=1024, fused=True, blank=-1, clamp=-1.0, reduction="sum"),     # persistent, TMA rows
    dict(V=512, fused=False, blank=-1, clamp=0.5, reduction="mean"),     # persistent, gather
    dict(V=2048, fused=True, blank=3, clamp=-1.0, reduction="none"),     # per-stage TMA (4 KB rows)
    dict(V=29, fused=True, blank=0, clamp=0.1, reduction="mean"),        # per-stage kernels
    dict(V=5000, fused=True, blank=0, clamp=-1.0, reduction="mean"),     # long rows (streamed)
]


@pytest.mark.parametrize("case", range(len(BF16_CASES)))
def test_bf16_elementwise(case):
    wl = rand_wl(120 + case, B=4, Tmax=60, Umax=30, dtype="bf16", sigma=1.5, **BF16_CASES[case])
    loss, red, grad = gpu_run(wl)
    ref = oracle_full(wl)
    assert grad.dtype == torch.bfloat16
    assert_loss_close(to_np(loss), ref.losses, "bf16")
    assert_grad_close(to_np(grad.float()), ref.grad, "bf16")


def test_bf16_schedules_agree_and_options(monkeypatch):
    wl = rand_wl(130, B=6, Tmax=80, Umax=50, V=1024, dtype="bf16", sigma=1.3, reduction="sum")
    monkeypatch.setenv("RNNT_GB300_SCHEDULE", "kernels")
    a = gpu_run(wl, fastemit_lambda=0.4)
    monkeypatch.delenv("RNNT_GB300_SCHEDULE")
    b = gpu_run(wl, fastemit_lambda=0.4)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    xp = W.to_padded(wl, fill=float("nan"))
    lp, rp, gp = run_padded(wl, xp, fastemit_lambda=0.4)
    assert torch.equal(lp, b[0])
    ref = oracle.rnnt_loss_padded(to_np(xp), wl.targets, wl.T, wl.U, blank=-1, reduction="sum",
                                  fastemit_lambda=0.4)
    assert_grad_close(to_np(gp.float()), ref.grad, "bf16")


# ------------------------------------------------------------------ degenerate shapes
def test_padded_degenerate_lattices():
    # T=1 and U=0 in every combination inside a padded tensor wider than all of them.
    wl = make(4, [1, 1, 9, 5], [0, 4, 0, 2], 16, dtype="f32", blank=2, reduction="sum")
    xp = W.to_padded(wl, max_T=10, max_U=6, fill=float("nan"))
    loss, red, grad = run_padded(wl, xp, fastemit_lambda=0.5)
    ref = oracle.rnnt_loss_padded(to_np(xp), wl.targets, wl.T, wl.U, blank=2, reduction="sum",
                                  fastemit_lambda=0.5)
    assert_loss_close(to_np(loss), ref.losses, "f32")
    assert_grad_close(to_np(grad), ref.grad, "f32")


def test_padded_single_slot_and_exact_fit():
    # max_T = T and max_U = U for every sample: the padded layout is the compact one.
    wl = make(2, [7, 7], [3, 3], 24, dtype="f16", blank=-1, reduction="mean")
    xp = W.to_padded(wl)
    assert xp.shape == (2, 7, 4, 24)
    lp, rp, gp = run_padded(wl, xp)
    lc, rc, gc = gpu_run(wl)
    assert torch.equal(lp, lc) and torch.equal(gp.reshape(-1, 24), gc)


def test_multiblank_degenerate_lattices():
    # T shorter than every big blank, T equal to a duration, U=0 and T=1.
    wl = make(5, [1, 2, 4, 3, 8], [0, 1, 0, 2, 0], 12, dtype="f32", blank=-1, reduction="sum")
    wl.targets[:] = wl.targets % 9
    big = [(10, 2), (9, 4)]
    loss, red, grad = gpu_run(wl, big_blanks=big, sigma=0.1)
    ref = oracle.rnnt_loss_multiblank(to_np(wl.logits), wl.targets, wl.T, wl.U, big, blank=-1,
                                      sigma=0.1, reduction="sum")
    assert_loss_close(to_np(loss), ref.losses, "f32")
    assert_grad_close(to_np(grad), ref.grad, "f32")


# ------------------------------------------------------------------ log-probability inputs, per-stage
# Without the in-kernel log-softmax, a call the persistent kernel does not take
# (here a lattice of 301 columns) zeroes the whole gradient buffer from extra
# CTAs of the recursion launch and then stores only the blank and label
# elements.  Every element must match the oracle whatever the buffer held
# before (in place: the log-probabilities themselves), with a byte count that
# is no multiple of 16 (74-byte rows), long rows, and padding rows.
LOGPROB_CASES = [
    dict(V=37, dtype="f16", blank=5, clamp=-1.0, reduction="sum"),
    dict(V=512, dtype="f16", blank=-1, clamp=0.5, reduction="mean"),
    dict(V=80, dtype="f32", blank=2, clamp=0.3, reduction="none"),
    dict(V=2500, dtype="bf16", blank=0, clamp=-1.0, reduction="mean"),
    dict(V=2200, dtype="f32", blank=-1, clamp=-1.0, reduction="sum"),   # 8.8 KB rows
]


@pytest.mark.parametrize("case", range(len(LOGPROB_CASES)))
def test_log_prob_inputs_zero_filled_buffer(case):
    kw = LOGPROB_CASES[case]
    wl = make(3, [7, 25, 4], [300, 9, 0], fused=False, sigma=1.0, seed=150 + case, **kw)
    dt = {"f32": 0, "f16": 1, "bf16": 2}[kw["dtype"]]
    plan = N.rnnt_plan(3, wl.logits.shape[0], kw["V"], dt, wl.targets.shape[1], False, True)
    assert plan == {"persistent": False, "launches": 4}
    ref = oracle_full(wl)
    loss, red, grad = gpu_run(wl, inplace=True)
    assert_loss_close(to_np(loss), ref.losses, kw["dtype"])
    assert_grad_close(to_np(grad.float()), ref.grad, kw["dtype"])
    # Exact zeros wherever the oracle's gradient is zero (every element but
    # the blank and label ones).
    assert not grad.float()[torch.as_tensor(ref.grad == 0.0, device="cuda")].any()
    lc, rc, gc = gpu_run(wl)
    assert torch.equal(lc, loss) and torch.equal(gc, grad)
    xp = W.to_padded(wl, max_T=27, max_U=302, fill=float("nan"))
    lp, rp, gp = run_padded(wl, xp)
    assert torch.equal(lp, lc) and torch.equal(rp, rc)
    for b in range(3):
        T, U = int(wl.T[b]), int(wl.U[b])
        assert torch.equal(gp[b, :T, :U + 1].reshape(-1, kw["V"]), gc[wl.sample_rows(b)])
        assert not gp[b, T:].any() and not gp[b, :, U + 1:].any()
