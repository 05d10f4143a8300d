"""GPU parity: the CUDA path (called through the C ABI) against the float64
oracle on identical seeded inputs.  Element-wise everywhere: every loss and
every gradient element of the small cases, and of the full-size workloads
sample by sample in row blocks; plus properties that hold at any size (zero
row sums, alpha/beta agreement via the status word)."""
import numpy as np
import pytest
import torch

import oracle
from rnn_transducer_loss_gb300 import workloads as W
from rnn_transducer_loss_gb300 import _native as N
from rnn_transducer_loss_gb300.functional import rnnt_loss, rnnt_loss_forward

from parity_util import (TOL, assert_grad_close, assert_loss_close, every_row_compare,
                         gpu_run, oracle_full, to_np)

pytestmark = pytest.mark.gpu


def full_compare(wl, **over):
    loss, red, grad = gpu_run(wl, **over)
    ref = oracle_full(wl, **over)
    dt = wl.cfg.dtype
    assert_loss_close(to_np(loss), ref.losses, dt)
    red_name = over.get("reduction", wl.cfg.reduction)
    if red_name != "none":
        assert_loss_close([float(red)], [ref.reduced], dt)
    assert_grad_close(to_np(grad.float()), ref.grad, dt)
    return loss, grad, ref


# ------------------------------------------------------------------ workloads
def test_tiny_elementwise():
    full_compare(W.make("tiny", "cuda"))


def test_char_asr_elementwise():
    wl = W.make("char_asr", "cuda")
    # 116-byte rows take the persistent kernel: one launch
    plan = N.rnnt_plan(wl.cfg.B, wl.logits.shape[0], wl.cfg.V, 0, wl.targets.shape[1], True, True)
    assert plan == {"persistent": True, "launches": 1}
    full_compare(wl)


@pytest.mark.parametrize("red", ["none", "sum", "mean"])
def test_char_asr_reductions(red):
    full_compare(W.make("char_asr", "cuda"), reduction=red, clamp=-1.0)


# Full-size workloads: one call on the whole batch, in the configuration the
# benchmark times, then every loss and every gradient element against the
# oracle (sample by sample, in row blocks).
def test_bpe_asr_every_row():
    wl = W.make("bpe_asr", "cuda")
    loss, red, grad, ref = every_row_compare(wl)
    # Row sums of the fused, unclamped gradient vanish at any size.
    s = grad.float().sum(dim=1)
    assert float(s.abs().max()) < 0.05


def test_skewed_every_row():
    every_row_compare(W.make("skewed", "cuda"))


@pytest.mark.slow
def test_large_vocab_every_row():
    wl = W.make("large_vocab", "cuda")
    loss, red, grad, ref = every_row_compare(wl)
    assert float(grad.sum(dim=1).abs().max()) < 1e-5


# The rnnt-loss-ascend README's accuracy table (精度测试: against a float64 CPU
# reference, reduction "mean"): per row the dtype, batch, T and U ranges and V.
# Lengths are drawn uniformly from the ranges; in the float32 B=4 row the first
# sample is set to the range maxima (T=2000, U=500: 2500 anti-diagonals, above
# the 2048-entry diagonal-base table, and 501 lattice columns), so the
# recursions' table-free path runs.
README_ACCURACY = [
    ("f32", 2, (100, 1000), (100, 300), 50),
    ("f32", 4, (200, 2000), (50, 500), 128),
    ("f16", 2, (100, 500), (50, 200), 64),
    ("f16", 4, (100, 1000), (50, 300), 128),
]


@pytest.mark.parametrize("row", range(len(README_ACCURACY)))
def test_readme_accuracy_table_shapes(row):
    dt, B, Tr, Ur, V = README_ACCURACY[row]
    rng = np.random.default_rng(500 + row)
    T = rng.integers(Tr[0], Tr[1] + 1, size=B)
    U = rng.integers(Ur[0], Ur[1] + 1, size=B)
    if row == 1:
        T[0], U[0] = Tr[1], Ur[1]
    wl = W.custom(B, T, U, V, dtype=dt, blank=-1, reduction="mean", seed=60 + row,
                  device="cuda")
    every_row_compare(wl)


@pytest.mark.parametrize("case", ["persistent", "staged"])
def test_more_than_2048_anti_diagonals(case):
    # T+U > 2048 on both schedules: a 101-column lattice in the persistent
    # kernel (fp16, V=1024) and a 21-column one on the per-stage kernels.
    if case == "persistent":
        wl = W.custom(2, [2100, 300], [100, 40], 1024, dtype="f16", sigma=1.5, blank=-1,
                      reduction="sum", seed=71, device="cuda")
    else:
        wl = W.custom(2, [2200, 50], [20, 7], 64, dtype="f32", blank=0, reduction="mean",
                      seed=72, device="cuda")
    every_row_compare(wl)


# ------------------------------------------------------------------ edge cases
def make(B, T, U, V, **kw):
    return W.custom(B, T, U, V, device="cuda", **kw)


@pytest.mark.parametrize("dtype", ["f32", "f16"])
@pytest.mark.parametrize("fused", [True, False])
def test_random_many_tiles(dtype, fused):
    rng = np.random.default_rng(11 if fused else 12)
    B = 9
    T = rng.integers(1, 70, size=B)
    U = rng.integers(0, 45, size=B)
    wl = make(B, T, U, 37, dtype=dtype, sigma=1.7, blank=5, clamp=-1.0, fused=fused,
              reduction="sum", seed=3)
    full_compare(wl)


@pytest.mark.parametrize("V", [1, 2, 7, 8, 29, 64, 1001])
def test_vocab_sizes(V):
    U = [0, 0] if V == 1 else [3, 1]
    wl = make(2, [5, 9], U, V, dtype="f32", blank=-1, reduction="none")
    full_compare(wl)


@pytest.mark.parametrize("U", [30, 31, 32, 33, 63, 64, 65, 127, 128, 129, 300, 520])
def test_lattice_widths(U):
    wl = make(2, [40, 3], [U, U // 2], 12, dtype="f32", blank=0, reduction="mean")
    full_compare(wl)


def test_degenerate_lattices():
    # T=1 and U=0 in every combination, incl. the single-node lattice.
    wl = make(5, [1, 1, 7, 1, 13], [0, 6, 0, 1, 0], 9, dtype="f32", blank=3, reduction="sum")
    full_compare(wl)


def test_single_node_closed_form():
    wl = make(1, [1], [0], 6, dtype="f32", blank=-1, reduction="none")
    loss, _, grad = gpu_run(wl)
    h = to_np(wl.logits).astype(np.float64)[0]
    lse = np.log(np.exp(h - h.max()).sum()) + h.max()
    assert float(loss[0]) == pytest.approx(-(h[-1] - lse), rel=1e-6)


@pytest.mark.parametrize("blank", [0, 4, 10, -11, -1])
def test_blank_positions(blank):
    wl = make(3, [12, 4, 20], [5, 2, 9], 11, dtype="f32", blank=blank, reduction="mean",
              clamp=0.05)
    full_compare(wl)


def test_long_targets_j32():
    wl = make(2, [30, 25], [700, 1000], 16, dtype="f32", blank=0, reduction="sum")
    full_compare(wl)


def test_large_batch_many_small_samples():
    rng = np.random.default_rng(4)
    B = 1500
    wl = make(B, rng.integers(1, 6, size=B), rng.integers(0, 4, size=B), 9, dtype="f16",
              blank=0, reduction="mean")
    full_compare(wl)


def test_inplace_gradient_matches():
    wl = make(3, [30, 17, 9], [8, 12, 0], 64, dtype="f16", blank=-1, reduction="sum")
    _, _, g_sep = gpu_run(wl)
    _, _, g_inp = gpu_run(wl, inplace=True)
    assert torch.equal(g_sep, g_inp)


def test_loss_only_matches():
    wl = make(3, [30, 17, 9], [8, 12, 0], 64, dtype="f32", blank=-1, reduction="sum")
    l1, r1, _ = gpu_run(wl)
    l2, r2, g2 = gpu_run(wl, want_grad=False)
    assert g2 is None
    assert torch.equal(l1, l2) and torch.equal(r1, r2)


def test_deterministic():
    wl = W.make("char_asr", "cuda")
    a = gpu_run(wl)
    b = gpu_run(wl)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_uniform_logits_closed_form_at_bpe_shape():
    # Constant logits: loss = (T+U) log V - log C(T-1+U, U) at a BPE-sized lattice.
    import math
    T, U, V = 400, 75, 1024
    wl = make(1, [T], [U], V, dtype="f16", blank=-1, reduction="none")
    wl.logits.zero_()
    loss, _, _ = gpu_run(wl)
    lb = math.lgamma(T + U) - math.lgamma(U + 1) - math.lgamma(T)
    assert float(loss[0]) == pytest.approx((T + U) * math.log(V) - lb, rel=1e-5)


# ------------------------------------------------------------------ errors
def _status_of(wl, **over):
    cfg = wl.cfg
    with pytest.raises((ValueError, N.RNNTError)) as e:
        rnnt_loss_forward(wl.logits, torch.as_tensor(over.get("targets", wl.targets), device="cuda"),
                          torch.as_tensor(over.get("T", wl.T), device="cuda"),
                          torch.as_tensor(over.get("U", wl.U), device="cuda"), cfg.blank,
                          cfg.clamp, cfg.reduction, cfg.fused)
    return e.value


def test_device_detects_bad_inputs():
    wl = make(2, [5, 4], [2, 3], 7, dtype="f32", blank=0, reduction="sum")
    bad = wl.targets.copy()
    bad[1, 0] = 0  # label equal to blank
    assert isinstance(_status_of(wl, targets=bad), ValueError)
    bad = wl.targets.copy()
    bad[0, 1] = 7  # label out of range
    assert isinstance(_status_of(wl, targets=bad), ValueError)
    assert isinstance(_status_of(wl, T=np.array([5, 5], dtype=np.int32)), ValueError)  # rows
    assert isinstance(_status_of(wl, T=np.array([0, 4], dtype=np.int32)), ValueError)
    # The workspace is reusable after an error: a valid call still succeeds.
    full_compare(wl)


@pytest.mark.parametrize("sched", ["persistent", "kernels"])
@pytest.mark.parametrize("k", [2, 6])
def test_non_finite_input_reports_mismatch(k, sched, monkeypatch):
    # A NaN that is the only element some lane of the row reduction sees (7
    # elements over 8-lane groups) must still reach the non-finite check.
    if sched == "kernels":
        monkeypatch.setenv("RNNT_GB300_SCHEDULE", "kernels")
    wl = make(2, [5, 4], [2, 3], 7, dtype="f32", blank=0, reduction="sum")
    wl.logits[3, k] = float("nan")
    e = _status_of(wl)
    assert isinstance(e, N.RNNTError) and e.code == N.RNNT_LOSS_MISMATCH


# ------------------------------------------------------------------ autograd
@pytest.mark.parametrize("red", ["none", "sum", "mean"])
def test_autograd_backward_scales(red):
    wl = make(3, [20, 11, 6], [4, 9, 2], 33, dtype="f32", blank=-1, reduction=red, clamp=-1.0)
    x = wl.logits.clone().requires_grad_(True)
    y = torch.as_tensor(wl.targets, device="cuda")
    Tl = torch.as_tensor(wl.T, device="cuda")
    Ul = torch.as_tensor(wl.U, device="cuda")
    out = rnnt_loss(x, y, Tl, Ul, blank=-1, reduction=red)
    w = torch.tensor([0.5, -2.0, 3.0], device="cuda") if red == "none" else torch.tensor(
        1.7, device="cuda")
    (out * w).sum().backward()
    ref = oracle_full(wl, reduction=red)
    want = ref.grad.copy()
    if red == "none":
        for b in range(3):
            sl = wl.sample_rows(b)
            want[sl] *= float(w[b])
    else:
        want *= float(w)
    assert_grad_close(to_np(x.grad), want, "f32")


def test_second_backward_raises():
    # The gradient is scaled in place by backward, so a second backward through
    # the same forward (retain_graph=True) must fail loudly, not return None.
    wl = make(2, [9, 5], [3, 2], 16, dtype="f32", blank=-1, reduction="sum")
    x = wl.logits.clone().requires_grad_(True)
    out = rnnt_loss(x, torch.as_tensor(wl.targets, device="cuda"),
                    torch.as_tensor(wl.T, device="cuda"), torch.as_tensor(wl.U, device="cuda"),
                    blank=-1, reduction="sum")
    out.backward(retain_graph=True)
    with pytest.raises(RuntimeError, match="only once"):
        out.backward()


# ------------------------------------------------------------------ schedules
# The library runs a call either as one persistent cooperative kernel (row,
# DP and gradient tasks scheduled on the device) or, for shapes that kernel
# does not cover, as one launch per stage.  RNNT_GB300_SCHEDULE=kernels forces
# the latter; both must agree bit for bit and with the oracle.
SCHED_CASES = [
    dict(B=5, V=512, dtype="f16", fused=True, blank=-1, reduction="sum", clamp=-1.0),
    dict(B=4, V=264, dtype="f32", fused=True, blank=0, reduction="mean", clamp=0.3),
    dict(B=6, V=1024, dtype="f16", fused=True, blank=7, reduction="none", clamp=-1.0),
    dict(B=5, V=512, dtype="f16", fused=False, blank=-1, reduction="mean", clamp=0.5),
    dict(B=3, V=80, dtype="f32", fused=False, blank=2, reduction="sum", clamp=-1.0),
    # 4 KB rows (8 vectors per lane): the persistent kernel's 3-stage rings
    dict(B=4, V=1024, dtype="f32", fused=True, blank=-1, reduction="sum", clamp=-1.0),
    dict(B=3, V=2048, dtype="f16", fused=True, blank=5, reduction="mean", clamp=0.2),
    # log-softmax on rows that are not 16-byte vectors (116-byte fp32 rows of
    # the character vocabulary, 74-byte fp16, 502-byte bf16 rows): plain loads
    dict(B=6, V=29, dtype="f32", fused=True, blank=0, reduction="mean", clamp=0.1),
    dict(B=4, V=37, dtype="f16", fused=True, blank=3, reduction="sum", clamp=-1.0),
    dict(B=3, V=251, dtype="bf16", fused=True, blank=-1, reduction="none", clamp=-1.0),
]


@pytest.mark.parametrize("case", range(len(SCHED_CASES)))
def test_persistent_and_staged_schedules_agree(case, monkeypatch):
    kw = dict(SCHED_CASES[case])
    rng = np.random.default_rng(40 + case)
    B = kw.pop("B")
    T = rng.integers(1, 90, size=B)
    U = rng.integers(0, 70, size=B)
    wl = make(B, T, U, kw.pop("V"), sigma=1.3, seed=case, **kw)
    monkeypatch.setenv("RNNT_GB300_SCHEDULE", "kernels")
    ref_gpu = gpu_run(wl)
    monkeypatch.delenv("RNNT_GB300_SCHEDULE")
    got = gpu_run(wl)
    for a, b in zip(ref_gpu, got):
        assert torch.equal(a, b)
    full_compare(wl)


def test_repeated_persistent_calls_all_succeed():
    # Task-list construction and the scheduler's counters are rebuilt on every
    # call: 25 calls in a row (one workspace, then fresh ones) must all succeed
    # and agree bit for bit.
    wl = W.subset(W.make("bpe_asr", "cuda"), 6)
    dev = "cuda"
    t = torch.as_tensor(wl.targets, device=dev)
    Tl, Ul = torch.as_tensor(wl.T, device=dev), torch.as_tensor(wl.U, device=dev)
    first = None
    for i in range(25):
        loss, red, grad, _ = rnnt_loss_forward(wl.logits, t, Tl, Ul, wl.cfg.blank, wl.cfg.clamp,
                                               wl.cfg.reduction, wl.cfg.fused)   # raises on a bad status
        if first is None:
            first = (loss.clone(), grad.clone())
        else:
            assert torch.equal(loss, first[0]) and torch.equal(grad, first[1])
