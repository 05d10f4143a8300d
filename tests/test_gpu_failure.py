"""Failure detection on the GPU without a fault: a bounded device wait that
runs out reports RNNT_TIMEOUT through the status word, and the context stays
usable for the next loss call."""
import pytest
import torch

from rnn_transducer_loss_gb300 import _native as N
from rnn_transducer_loss_gb300 import workloads as W

from parity_util import assert_grad_close, gpu_run, oracle_full, to_np

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    assert N.rnnt_selftest_wait_timeout(status.data_ptr(), 1 << 12, stream) == N.RNNT_OK
    torch.cuda.synchronize()
    assert int(status.item()) == N.RNNT_TIMEOUT
    assert N.rnnt_selftest_wait_timeout(None, 16, stream) == N.RNNT_INVALID_VALUE
    # the next loss call runs normally
    wl = W.make("tiny", "cuda")
    loss, red, grad = gpu_run(wl)
    assert_grad_close(to_np(grad), oracle_full(wl).grad, "f32")
