"""PyTorch entry points: ``rnnt_loss`` (torchaudio.functional.rnnt_loss semantics) and ``RNNTLoss``.

PyTorch supplies device memory and the current stream; every step of the loss
and its gradient runs in the CUDA kernels of librnnt_gb300.so.  As in the
rnnt-loss-ascend README (架构设计 "Python 层", 算子特性 "前反向融合"), the
forward call produces the loss and the gradient together; backward only
multiplies the saved gradient by the upstream gradient (a kernel that is a
no-op when that factor is 1).
"""
from __future__ import annotations

import torch

from . import _native as N

_DT = {torch.float32: N.RNNT_F32, torch.float16: N.RNNT_F16, torch.bfloat16: N.RNNT_BF16}


def _check_inputs(logits, targets, logit_lengths, target_lengths):
    if not logits.is_cuda:
        raise ValueError("logits must be a CUDA tensor")
    if logits.dtype not in _DT:
        raise ValueError(f"logits must be float32, float16 or bfloat16, got {logits.dtype}")
    if logits.dim() not in (2, 4):
        raise ValueError("logits must be 2-D (sum_b T_b*(U_b+1), V) or 4-D "
                         "(B, max_T, max_U+1, V)")
    for name, t in (("targets", targets), ("logit_lengths", logit_lengths),
                    ("target_lengths", target_lengths)):
        if t.dtype != torch.int32:
            raise ValueError(f"{name} must be int32, got {t.dtype}")
        if t.device != logits.device:
            raise ValueError(f"{name} must be on {logits.device}")
    if targets.dim() != 2 or logit_lengths.dim() != 1 or target_lengths.dim() != 1:
        raise ValueError("targets must be (B, S); lengths must be (B,)")
    B = logit_lengths.shape[0]
    if target_lengths.shape[0] != B or targets.shape[0] != B:
        raise ValueError("batch sizes of targets and lengths differ")
    if logits.dim() == 4 and logits.shape[0] != B:
        raise ValueError("padded logits must have the batch size of the lengths")
    if targets.shape[1] > N.MAX_TARGET_LENGTH:
        raise ValueError(f"targets wider than {N.MAX_TARGET_LENGTH} are not supported")


class Workspace:
    """Caller-owned scratch for one call (kept alive until backward)."""

    def __init__(self, B, rows, V, dt, device, **options):
        self.nbytes = (N.rnnt_workspace_size_ex(B, rows, V, dt, **options) if options
                       else N.rnnt_workspace_size(B, rows, V, dt))
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=device)


def rnnt_loss_forward(logits, targets, logit_lengths, target_lengths, blank=-1, clamp=-1.0,
                      reduction="mean", fused_log_softmax=True, want_grad=True,
                      inplace_grad=False, check=True, fastemit_lambda=0.0, big_blanks=(),
                      sigma=0.0):
    """One fused call.  Returns (loss[B] fp32, reduced fp32 scalar, grad or None, workspace).

    ``logits`` is the compact (sum_b T_b*(U_b+1), V) matrix or the padded
    (B, max_T, max_U+1, V) tensor; the gradient has the same shape (zero at
    padded positions)."""
    _check_inputs(logits, targets, logit_lengths, target_lengths)
    if reduction not in N.REDUCTIONS:
        raise ValueError(f"reduction must be one of {tuple(N.REDUCTIONS)}")
    if not fastemit_lambda >= 0.0:
        raise ValueError("fastemit_lambda must be >= 0")
    logits = logits.contiguous()
    targets = targets.contiguous()
    if targets.shape[1] == 0:
        targets = torch.zeros(targets.shape[0], 1, dtype=torch.int32, device=logits.device)
    padded = None
    if logits.dim() == 4:
        padded = (logits.shape[1], logits.shape[2] - 1)
        if padded[1] < 0 or padded[1] > N.MAX_TARGET_LENGTH:
            raise ValueError(f"padded logits need 1 <= max_U+1 <= {N.MAX_TARGET_LENGTH + 1}")
    V = logits.shape[-1]
    rows = logits.numel() // V
    B = logit_lengths.shape[0]
    dt = _DT[logits.dtype]
    dev = logits.device
    big_blanks = [(int(i), int(d)) for i, d in (big_blanks or ())]
    if len(big_blanks) > N.MAX_BIG_BLANKS:
        raise ValueError(f"at most {N.MAX_BIG_BLANKS} big blanks")
    options = {}
    if padded is not None or fastemit_lambda != 0.0 or big_blanks or sigma != 0.0:
        options = dict(fastemit_lambda=fastemit_lambda, padded=padded, big_blanks=big_blanks,
                       sigma=sigma)
    ws = Workspace(B, rows, V, dt, dev, **options)
    loss = torch.empty(B, dtype=torch.float32, device=dev)
    reduced = torch.empty((), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    grad = None
    if want_grad:
        grad = logits if inplace_grad else torch.empty_like(logits)
    stream = torch.cuda.current_stream(dev).cuda_stream
    args = (logits.data_ptr(), dt, rows, V, targets.data_ptr(), targets.shape[1],
            logit_lengths.contiguous().data_ptr(), target_lengths.contiguous().data_ptr(), B,
            int(blank), float(clamp), bool(fused_log_softmax), N.REDUCTIONS[reduction],
            loss.data_ptr(), reduced.data_ptr(), grad.data_ptr() if grad is not None else None,
            ws.buf.data_ptr(), ws.nbytes, status.data_ptr(), stream)
    with torch.cuda.device(dev):
        if not options:
            rc, where = N.rnnt_loss_fused(*args), "rnnt_loss_fused"
        else:
            rc, where = N.rnnt_loss_fused_ex(*args, **options), "rnnt_loss_fused_ex"
    if rc != N.RNNT_OK:
        raise N.RNNTError(rc, where)
    if check:
        code = int(status.item())
        if code == N.RNNT_INVALID_VALUE:
            raise ValueError("rnnt_loss: " + N.status_string(code) +
                             " (check T_b >= 1, 0 <= U_b <= targets.shape[1], labels in [0, V) "
                             "and != blank, rows == sum T_b*(U_b+1) for compact logits, "
                             "T_b <= max_T and U_b <= max_U for padded logits)")
        if code != N.RNNT_OK:
            raise N.RNNTError(code, "rnnt_loss")
    return loss, reduced, grad, ws


class _RNNTLossFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, logits, targets, logit_lengths, target_lengths, blank, clamp, reduction,
                fused_log_softmax, check, fastemit_lambda, big_blanks, sigma):
        loss, reduced, grad, ws = rnnt_loss_forward(
            logits, targets, logit_lengths, target_lengths, blank, clamp, reduction,
            fused_log_softmax, want_grad=ctx.needs_input_grad[0], check=check,
            fastemit_lambda=fastemit_lambda, big_blanks=big_blanks, sigma=sigma)
        ctx.reduction = reduction
        ctx.ws = ws
        V = logits.shape[-1]
        ctx.dims = (logits.numel() // V, V, logit_lengths.shape[0], _DT[logits.dtype])
        ctx.grad = grad
        ctx.used = False
        return loss if reduction == "none" else reduced

    @staticmethod
    def backward(ctx, grad_out):
        grad = ctx.grad
        if ctx.used:
            # The saved gradient was scaled in place by the first backward.
            raise RuntimeError("rnnt_loss: backward can run only once per forward call "
                               "(the gradient buffer is scaled in place); recompute the loss "
                               "to differentiate again")
        if grad is None:
            return (None,) * 12
        ctx.used = True
        rows, V, B, dt = ctx.dims
        factors = grad_out.detach().to(torch.float32).contiguous()
        per_sample = 1 if ctx.reduction == "none" else 0
        stream = torch.cuda.current_stream(grad.device).cuda_stream
        with torch.cuda.device(grad.device):
            rc = N.rnnt_grad_scale(grad.data_ptr(), dt, rows, V, B, ctx.ws.buf.data_ptr(),
                                   ctx.ws.nbytes, factors.data_ptr(), per_sample, stream)
        if rc != N.RNNT_OK:
            raise N.RNNTError(rc, "rnnt_grad_scale")
        ctx.grad = None
        ctx.ws = None
        return grad, None, None, None, None, None, None, None, None, None, None, None


def rnnt_loss(logits: torch.Tensor, targets: torch.Tensor, logit_lengths: torch.Tensor,
              target_lengths: torch.Tensor, blank: int = -1, clamp: float = -1.0,
              reduction: str = "mean", fused_log_softmax: bool = True,
              check: bool = True, fastemit_lambda: float = 0.0, big_blanks=(),
              sigma: float = 0.0) -> torch.Tensor:
    """RNN-T loss with the arguments of torchaudio.functional.rnnt_loss.

    ``logits`` is either the compact 2-D matrix of the rnnt-loss-ascend README
    ((sum_b T_b*(U_b+1), V), rows of sample b ordered t-major, u-minor) or the
    padded 4-D tensor (B, max_T, max_U+1, V) of torchaudio and the ESPnet
    GPURNNT docs; its gradient has the same layout (zero at padded
    positions).  ``fastemit_lambda`` (>= 0) scales the gradient of every
    label emission by 1 + lambda (FastEmit, GPURNNT docs); the loss is
    unchanged.  ``big_blanks`` = [(output index, duration), ...] and ``sigma``
    select the multi-blank transducer of the ESPnet compute_multiblank_grad_kernel
    docs (big blanks advance `duration` frames; sigma is subtracted from every
    log-probability).  Returns float32 per-sample losses (reduction="none") or a
    float32 scalar.  ``check`` reads the device status word after the call
    (one synchronisation) and raises on invalid lengths, labels or an
    alpha/beta loss mismatch.
    """
    return _RNNTLossFunction.apply(logits, targets, logit_lengths, target_lengths, blank, clamp,
                                   reduction, fused_log_softmax, check, float(fastemit_lambda),
                                   tuple(big_blanks or ()), float(sigma))


class RNNTLoss(torch.nn.Module):
    """Module form of :func:`rnnt_loss`."""

    def __init__(self, blank: int = -1, clamp: float = -1.0, reduction: str = "mean",
                 fused_log_softmax: bool = True, check: bool = True,
                 fastemit_lambda: float = 0.0, big_blanks=(), sigma: float = 0.0):
        super().__init__()
        self.blank, self.clamp, self.reduction = blank, clamp, reduction
        self.fused_log_softmax, self.check = fused_log_softmax, check
        self.fastemit_lambda, self.big_blanks, self.sigma = fastemit_lambda, big_blanks, sigma

    def forward(self, logits, targets, logit_lengths, target_lengths):
        return rnnt_loss(logits, targets, logit_lengths, target_lengths, self.blank, self.clamp,
                         self.reduction, self.fused_log_softmax, self.check,
                         self.fastemit_lambda, self.big_blanks, self.sigma)
