"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects bad host-side arguments before touching a device."""
import ctypes
import os
import re

import pytest

from rnn_transducer_loss_gb300 import _native as N
from rnn_transducer_loss_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return N.load()


def declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for fn in os.listdir(inc):
        if fn.endswith(".h"):
            src = open(os.path.join(inc, fn)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(rnnt_[a-z_0-9]+)\s*\(", src))
    return names


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert names, "no declarations found"
    assert names == set(N.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(6):
        assert N.status_string(code)
    assert N.abi_version() == 103


def test_workspace_size(lib):
    small = N.rnnt_workspace_size(2, 50, 16, N.RNNT_F32)
    big = N.rnnt_workspace_size(2, 5000, 16, N.RNNT_F32)
    assert small > 0 and big > small
    per_row = (N.rnnt_workspace_size(4, 2_000_000, 8, N.RNNT_F16)
               - N.rnnt_workspace_size(4, 1_000_000, 8, N.RNNT_F16)) / 1_000_000
    assert 34 <= per_row <= 40
    with pytest.raises(N.RNNTError):
        N.rnnt_workspace_size(0, 50, 16, N.RNNT_F32)
    with pytest.raises(N.RNNTError):
        N.rnnt_workspace_size(2, 50, 16, 7)


def _call(**kw):
    args = dict(logits=4096, dt=N.RNNT_F32, rows=50, V=16, targets=8192, targets_stride=3,
                logit_lengths=8448, target_lengths=8704, B=2, blank=-1, clamp=-1.0,
                fused_log_softmax=1, reduction=0, loss=8960, loss_reduced=None, grad=None,
                workspace=1 << 20, workspace_bytes=1 << 30, status_dev=None, stream=None)
    args.update(kw)
    return N.rnnt_loss_fused(**args)


@pytest.mark.parametrize("bad", [
    dict(logits=None), dict(loss=None), dict(workspace=None), dict(targets=None),
    dict(V=0), dict(B=0), dict(rows=1, B=2), dict(dt=3), dict(blank=16), dict(blank=-17),
    dict(reduction=5), dict(targets_stride=0), dict(targets_stride=1024),
    dict(logits=4100), dict(grad=4104), dict(workspace=(1 << 20) + 16),
    dict(clamp=float("nan")),
    dict(grad=4096 + 64),          # partly overlaps the logits
])
def test_host_validation_rejects(lib, bad):
    assert _call(**bad) == N.RNNT_INVALID_VALUE


def _call_ex(fastemit_lambda=0.0, padded=None, big_blanks=(), sigma=0.0, **kw):
    args = dict(logits=4096, dt=N.RNNT_F32, rows=50, V=16, targets=8192, targets_stride=3,
                logit_lengths=8448, target_lengths=8704, B=2, blank=-1, clamp=-1.0,
                fused_log_softmax=1, reduction=0, loss=8960, loss_reduced=None, grad=None,
                workspace=1 << 20, workspace_bytes=1 << 30, status_dev=None, stream=None)
    args.update(kw)
    return N.rnnt_loss_fused_ex(**args, fastemit_lambda=fastemit_lambda, padded=padded,
                                big_blanks=big_blanks, sigma=sigma)


@pytest.mark.parametrize("bad", [
    dict(fastemit_lambda=-0.1), dict(fastemit_lambda=float("nan")),
    dict(fastemit_lambda=float("inf")),
    dict(padded=(8, 3), rows=50),            # rows must be B*max_T*(max_U+1) = 64
    dict(padded=(0, 3), rows=0),
    dict(padded=(8, -1), rows=0),
    dict(padded=(8, 1024), rows=2 * 8 * 1025),
    dict(padded=(1 << 22, 1023), rows=2 * (1 << 22) * 1024),   # a slot of 2^32 rows
    dict(sigma=-0.1), dict(sigma=float("nan")),
    dict(big_blanks=[(3, 1)]),                 # duration below 2
    dict(big_blanks=[(3, 17)]),                # duration above the maximum
    dict(big_blanks=[(15, 2)]),                # the standard blank (-1 -> 15)
    dict(big_blanks=[(-1, 2)]),                # the standard blank, counted from the end
    dict(big_blanks=[(3, 2), (3, 4)]),         # repeated output
    dict(big_blanks=[(16, 2)]),                # outside the vocabulary
    dict(big_blanks=[(i, 2) for i in range(9)]),   # more than 8
])
def test_ex_options_validation_rejects(lib, bad):
    assert _call_ex(**bad) == N.RNNT_INVALID_VALUE


def test_workspace_size_ex(lib):
    base = N.rnnt_workspace_size(2, 5000, 16, N.RNNT_F32)
    assert N.rnnt_workspace_size_ex(2, 5000, 16, N.RNNT_F32) == base
    assert N.rnnt_workspace_size_ex(2, 5000, 16, N.RNNT_F32, fastemit_lambda=0.5,
                                    padded=(50, 49)) == base
    two = N.rnnt_workspace_size_ex(2, 5000, 16, N.RNNT_F32, big_blanks=[(3, 2), (4, 4)])
    assert two >= base + 2 * 8 * 5000
    assert N.rnnt_workspace_size_ex(2, 5000, 16, N.RNNT_F32, sigma=0.1) >= base
    # the multi-blank call wants the larger workspace (rejected before any launch)
    base50 = N.rnnt_workspace_size(2, 50, 16, N.RNNT_F32)
    assert _call_ex(big_blanks=[(3, 2)], workspace_bytes=base50) == N.RNNT_WORKSPACE_TOO_SMALL


def test_plan_host_validation(lib):
    bad = ctypes.c_void_p(None)
    assert lib.rnnt_plan(2, 50, 16, 0, 3, 1, 1, None, None) == N.RNNT_INVALID_VALUE
    p = N.Plan()
    for args in [(0, 50, 16, 0, 3), (2, 0, 16, 0, 3), (2, 50, 0, 0, 3), (2, 50, 16, 9, 3),
                 (2, 50, 16, 0, 0), (2, 50, 16, 0, 1024)]:
        assert lib.rnnt_plan(*args, 1, 1, None, ctypes.byref(p)) == N.RNNT_INVALID_VALUE
    del bad


def test_workspace_too_small(lib):
    assert _call(workspace_bytes=1024) == N.RNNT_WORKSPACE_TOO_SMALL


def test_grad_scale_host_validation(lib):
    assert N.rnnt_grad_scale(None, 0, 10, 4, 1, 1 << 20, 1 << 30, 4096, 0, None) \
        == N.RNNT_INVALID_VALUE
    assert N.rnnt_grad_scale(4096, 0, 10, 4, 1, 1 << 20, 16, 4096, 0, None) \
        == N.RNNT_WORKSPACE_TOO_SMALL


def test_library_has_no_torch_dependency(lib):
    # The boundary is plain C: the shared object must not link libtorch/libc10.
    with open(N.LIB_PATH, "rb") as f:
        blob = f.read()
    assert b"libtorch" not in blob and b"libc10" not in blob


def _declared_param_counts():
    src = open(os.path.join(ROOT, "include", "rnnt_gb300.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for m in re.finditer(r"\b(rnnt_[a-z_0-9]+)\s*\(([^)]*)\)\s*;", src):
        args = m.group(2).strip()
        out[m.group(1)] = 0 if args in ("", "void") else args.count(",") + 1
    return out


def test_binding_argument_counts_match_the_header(lib):
    counts = _declared_param_counts()
    assert set(counts) == set(N.EXPORTS)
    for name, n in counts.items():
        assert len(getattr(lib, name).argtypes) == n, name


def test_options_struct_layout_matches_the_header():
    # float, 4 int32, 8 int32 ids, 8 int32 durations, float: 22 four-byte fields
    assert ctypes.sizeof(N.Options) == 4 * (1 + 4 + 2 * N.MAX_BIG_BLANKS + 1)
    assert N.Options.sigma.offset == 4 * (1 + 4 + 2 * N.MAX_BIG_BLANKS)
    hdr = open(os.path.join(ROOT, "include", "rnnt_gb300.h")).read()
    assert f"#define RNNT_MAX_BIG_BLANKS {N.MAX_BIG_BLANKS}" in hdr
    assert f"#define RNNT_MAX_BIG_BLANK_DURATION {N.MAX_BIG_BLANK_DURATION}" in hdr
