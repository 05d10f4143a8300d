"""Brute-force RNN-T loss by enumerating every alignment (tiny lattices only).

TEST INFRASTRUCTURE ONLY.  An independent second route to the loss and its
gradient, used to pin the C oracle: it never runs the alpha/beta recursions.

An alignment of a sample with T frames and U labels is a monotone walk on the
(t, u) lattice from (0, 0) to (T-1, U) made of T-1 blank steps (t+1) and U
label steps (u+1), followed by the terminal blank at (T-1, U); its
log-probability is the sum of the log-probs of its T+U emissions (ESPnet
GPURNNT docs: negative log likelihood over all alignments; warp-transducer
blog section 1.1: the loss sums over every legal alignment).  The loss is
-logsumexp over alignments; the gradient is float64 autograd of that
expression, through log_softmax when the rows are raw logits.

FastEmit (``fastemit_lambda``, the GPURNNT docs' regulariser weight): the
objective that is differentiated adds, for every alignment, lambda times its
posterior weight (a constant, computed here by enumeration) times the sum of
its label-emission log-probabilities, with a minus sign.  Its gradient is the
transducer gradient with every label-emission log-probability's term scaled
by 1 + lambda; the reported loss stays -log P(y|x).
"""
from __future__ import annotations

import itertools
import math

import torch


def alignments(T: int, U: int):
    """All move sequences: tuples of 'b'/'y' with T-1 blanks and U labels."""
    n = T - 1 + U
    for label_pos in itertools.combinations(range(n), U):
        s = ["b"] * n
        for p in label_pos:
            s[p] = "y"
        yield tuple(s)


def num_alignments(T: int, U: int) -> int:
    return math.comb(T - 1 + U, U)


def sample_loss(h: torch.Tensor, T: int, U: int, y, blank: int, fused: bool,
                fastemit_lambda: float = 0.0):
    """-log P(y|x) of one sample; h is its (T*(U+1), V) block (float64, may require grad).

    With ``fastemit_lambda`` != 0 returns (loss, objective): the objective is
    the loss plus the FastEmit term (module docstring); differentiate it for
    the gradient."""
    V = h.shape[1]
    blank = blank + V if blank < 0 else blank
    lp = torch.log_softmax(h, dim=1) if fused else h
    W = U + 1
    scores, label_scores = [], []
    for path in alignments(T, U):
        t = u = 0
        s = h.new_zeros(())
        sl = h.new_zeros(())
        for move in path:
            r = t * W + u
            if move == "b":
                s = s + lp[r, blank]
                t += 1
            else:
                e = lp[r, int(y[u])]
                s = s + e
                sl = sl + e
                u += 1
        s = s + lp[(T - 1) * W + U, blank]
        scores.append(s)
        label_scores.append(sl)
    sc = torch.stack(scores)
    loss = -torch.logsumexp(sc, dim=0)
    if not fastemit_lambda:
        return loss
    weight = torch.softmax(sc.detach(), dim=0)   # posterior of every alignment
    return loss, loss - fastemit_lambda * (weight * torch.stack(label_scores)).sum()


def rnnt_loss(logits, targets, logit_lengths, target_lengths, blank=-1, clamp=-1.0,
              reduction="mean", fused_log_softmax=True, fastemit_lambda=0.0):
    """Batch loss and gradient; returns (per-sample losses, reduced, grad) in float64."""
    x = torch.as_tensor(logits).to(torch.float64).detach().clone().requires_grad_(True)
    T = [int(v) for v in logit_lengths]
    U = [int(v) for v in target_lengths]
    B = len(T)
    rows = 0
    per = []
    grads = []
    for b in range(B):
        n = T[b] * (U[b] + 1)
        hb = x[rows:rows + n]
        yb = [int(v) for v in list(targets[b])[:U[b]]]
        lb = sample_loss(hb, T[b], U[b], yb, blank, fused_log_softmax, fastemit_lambda)
        lb, obj = lb if fastemit_lambda else (lb, lb)
        (g,) = torch.autograd.grad(obj, hb)
        per.append(lb.detach())
        grads.append(g)
        rows += n
    losses = torch.stack(per)
    scale = 1.0 / B if reduction == "mean" else 1.0
    grad = torch.cat(grads, dim=0)
    if clamp > 0:
        grad = grad.clamp(-clamp, clamp)
    grad = grad * scale
    reduced = losses.sum() * scale
    return losses.numpy(), float(reduced), grad.numpy()


def rnnt_loss_padded(logits, targets, logit_lengths, target_lengths, blank=-1, clamp=-1.0,
                     reduction="mean", fused_log_softmax=True, fastemit_lambda=0.0):
    """Brute force on the padded (B, max_T, max_U+1, V) layout: every alignment
    indexes node (t, u) of sample b as logits[b, t, u] directly; padded entries
    take no part, so their gradient is zero.  Returns (losses, reduced, grad)."""
    x = torch.as_tensor(logits).to(torch.float64).detach().clone().requires_grad_(True)
    B, maxT, maxW, V = x.shape
    per, objs = [], []
    for b in range(B):
        T, U = int(logit_lengths[b]), int(target_lengths[b])
        hb = x[b, :T, :U + 1, :].reshape(T * (U + 1), V)
        yb = [int(v) for v in list(targets[b])[:U]]
        lb = sample_loss(hb, T, U, yb, blank, fused_log_softmax, fastemit_lambda)
        lb, obj = lb if fastemit_lambda else (lb, lb)
        per.append(lb.detach())
        objs.append(obj)
    (grad,) = torch.autograd.grad(torch.stack(objs).sum(), x)
    losses = torch.stack(per)
    scale = 1.0 / B if reduction == "mean" else 1.0
    if clamp > 0:
        grad = grad.clamp(-clamp, clamp)
    grad = grad * scale
    return losses.numpy(), float(losses.sum() * scale), grad.numpy()


def multiblank_paths(T: int, U: int, durations):
    """Every multi-blank alignment: move sequences from (0, 0) to the end (frame
    T with U labels).  A move is 'b' (one frame), 'y' (one label) or an int i
    (big blank i, durations[i] frames); no move passes frame T, and a
    blank-type move may reach frame T only with every label emitted."""
    out = []

    def walk(t, u, seq):
        if t == T:
            if u == U:
                out.append(tuple(seq))
            return
        if u < U:
            walk(t, u + 1, seq + ["y"])
        for mv, d in [("b", 1)] + [(i, d) for i, d in enumerate(durations)]:
            if t + d < T or (t + d == T and u == U):
                walk(t + d, u, seq + [mv])

    walk(0, 0, [])
    return out


def multiblank_loss(h, T, U, y, blank, big_blanks, sigma, fused, fastemit_lambda=0.0):
    """(loss, objective) of one sample by enumeration of multi-blank alignments."""
    V = h.shape[1]
    blank = blank + V if blank < 0 else blank
    ids = [i + V if i < 0 else i for i, _ in big_blanks]
    durs = [d for _, d in big_blanks]
    lp = (torch.log_softmax(h, dim=1) if fused else h) - sigma
    W = U + 1
    scores, label_scores = [], []
    for path in multiblank_paths(T, U, durs):
        t = u = 0
        s = h.new_zeros(())
        sl = h.new_zeros(())
        for mv in path:
            r = t * W + u
            if mv == "y":
                e = lp[r, int(y[u])]
                s, sl = s + e, sl + e
                u += 1
            elif mv == "b":
                s = s + lp[r, blank]
                t += 1
            else:
                s = s + lp[r, ids[mv]]
                t += durs[mv]
        scores.append(s)
        label_scores.append(sl)
    sc = torch.stack(scores)
    loss = -torch.logsumexp(sc, dim=0)
    weight = torch.softmax(sc.detach(), dim=0)
    return loss, loss - fastemit_lambda * (weight * torch.stack(label_scores)).sum()


def rnnt_loss_multiblank(logits, targets, logit_lengths, target_lengths, big_blanks, blank=-1,
                         sigma=0.0, clamp=-1.0, reduction="mean", fused_log_softmax=True,
                         fastemit_lambda=0.0):
    """Brute-force multi-blank loss and gradient (compact layout); (losses, reduced, grad)."""
    x = torch.as_tensor(logits).to(torch.float64).detach().clone().requires_grad_(True)
    T = [int(v) for v in logit_lengths]
    U = [int(v) for v in target_lengths]
    B = len(T)
    rows, per, grads = 0, [], []
    for b in range(B):
        n = T[b] * (U[b] + 1)
        hb = x[rows:rows + n]
        yb = [int(v) for v in list(targets[b])[:U[b]]]
        lb, obj = multiblank_loss(hb, T[b], U[b], yb, blank, big_blanks, sigma,
                                  fused_log_softmax, fastemit_lambda)
        (g,) = torch.autograd.grad(obj, hb)
        per.append(lb.detach())
        grads.append(g)
        rows += n
    losses = torch.stack(per)
    scale = 1.0 / B if reduction == "mean" else 1.0
    grad = torch.cat(grads, dim=0)
    if clamp > 0:
        grad = grad.clamp(-clamp, clamp)
    return losses.numpy(), float(losses.sum() * scale), (grad * scale).numpy()
