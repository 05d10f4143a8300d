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


def sample_loss(h: torch.Tensor, T: int, U: int, y, blank: int, fused: bool) -> torch.Tensor:
    """-log P(y|x) of one sample; h is its (T*(U+1), V) block (float64, may require grad)."""
    V = h.shape[1]
    blank = blank + V if blank < 0 else blank
    lp = torch.log_softmax(h, dim=1) if fused else h
    W = U + 1
    scores = []
    for path in alignments(T, U):
        t = u = 0
        s = h.new_zeros(())
        for move in path:
            r = t * W + u
            if move == "b":
                s = s + lp[r, blank]
                t += 1
            else:
                s = s + lp[r, int(y[u])]
                u += 1
        s = s + lp[(T - 1) * W + U, blank]
        scores.append(s)
    return -torch.logsumexp(torch.stack(scores), dim=0)


def rnnt_loss(logits, targets, logit_lengths, target_lengths, blank=-1, clamp=-1.0,
              reduction="mean", fused_log_softmax=True):
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
        lb = sample_loss(hb, T[b], U[b], yb, blank, fused_log_softmax)
        (g,) = torch.autograd.grad(lb, hb)
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
