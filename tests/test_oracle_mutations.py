"""The oracle's pins catch plausible mistakes (CPU only).

Each case plants one mistake in a copy of oracle/rnnt_oracle.c (a dropped
term, a wrong sign, a wrong index, a swapped order), compiles the copy, and
runs the independent pins against it: brute-force enumeration, the constant-
logit closed form and the alpha/beta agreement.  Every planted mistake must
fail at least one of them; the unmodified source must pass them all."""
import math
import os
import shutil
import subprocess

import numpy as np
import pytest
from scipy.special import log_softmax

import oracle
from oracle import brute

SRC = os.path.join(os.path.dirname(oracle.__file__), "rnnt_oracle.c")

# (name, [(original text, planted text, which occurrence or None for all)])
MUTANTS = [
    ("lse without the max shift", [("s += exp(lp[k] - m);", "s += exp(lp[k]);", 0)]),
    ("label of the previous position", [("lpy[r] = (u < U) ? lp[y[u]] : -INFINITY;",
                                         "lpy[r] = (u < U) ? lp[y[u > 0 ? u - 1 : 0]] : -INFINITY;",
                                         0)]),
    ("alpha label arc from the wrong node", [("alpha[r - 1] + lpy[r - 1] : -INFINITY",
                                              "alpha[r - 1] + lpy[r] : -INFINITY", 0)]),
    ("terminal blank dropped", [("losses[0] = -(alpha[last] + lpb[last]);",
                                 "losses[0] = -(alpha[last]);", 0)]),
    ("blank successor one column over", [("beta_after_blank = beta[r + W];",
                                          "beta_after_blank = beta[r + 1];", 0)]),
    ("chain rule sign", [("g[k] -= exp(lp[k]) * s;", "g[k] += exp(lp[k]) * s;", 0)]),
    ("scale before clamp", [("double v = g[k];", "double v = g[k] * scale;", 0),
                            ("g[k] = v * scale;", "g[k] = v;", 0)]),
    ("FastEmit on the blank", [("g[blank] -= post_blank;",
                                "g[blank] -= (1.0 + fastemit_lambda) * post_blank;", 0)]),
    ("multi-blank: sigma not on labels", [("lpy[r] = (u < U) ? lp[y[u]] - sigma : -INFINITY;",
                                           "lpy[r] = (u < U) ? lp[y[u]] : -INFINITY;", 0)]),
    ("multi-blank: big blank ending with labels left", [("else if (t1 == T && u == U)",
                                                          "else if (t1 == T)", 0)]),
]


def _plant(src: str, edits):
    for old, new, occ in edits:
        idx = -1
        for _ in range(occ + 1):
            idx = src.index(old, idx + 1)
        src = src[:idx] + new + src[idx + len(old):]
    return src


def _case(seed, B=3, Tmax=4, Umax=3, V=5, fused=True):
    rng = np.random.default_rng(seed)
    T = rng.integers(1, Tmax + 1, size=B).astype(np.int32)
    U = rng.integers(0, Umax + 1, size=B).astype(np.int32)
    T[0], U[0] = Tmax, Umax
    y = rng.integers(0, V - 3, size=(B, max(1, Umax))).astype(np.int32)   # below V-3
    rows = int((T.astype(np.int64) * (U + 1)).sum())
    x = rng.normal(0.0, 1.3, size=(rows, V))
    return (x if fused else log_softmax(x, axis=1)), y, T, U


def _pins_pass() -> bool:
    """True when every pin holds for the currently loaded oracle library."""
    try:
        for seed, fused, clamp, red, lam in [(1, True, -1.0, "sum", 0.0), (2, False, 0.2, "mean", 0.0),
                                             (3, True, 0.15, "mean", 0.0), (4, True, -1.0, "sum", 0.7)]:
            x, y, T, U = _case(seed, fused=fused)
            got = oracle.rnnt_loss(x, y, T, U, blank=-1, clamp=clamp, reduction=red,
                                   fused_log_softmax=fused, fastemit_lambda=lam)
            wl, wr, wg = brute.rnnt_loss(x, y, T, U, blank=-1, clamp=clamp, reduction=red,
                                         fused_log_softmax=fused, fastemit_lambda=lam)
            if not (np.allclose(got.losses, wl, rtol=1e-10, atol=1e-12)
                    and np.allclose(got.losses_beta, got.losses, rtol=1e-10, atol=1e-12)
                    and np.allclose(got.grad, wg, rtol=1e-8, atol=1e-11)):
                return False
        # constant logits: loss (T+U) log V - log C(T-1+U, U)
        T, U, V = 5, 3, 7
        r = oracle.rnnt_loss(np.zeros((T * (U + 1), V)), [[0, 1, 2]], [T], [U], blank=-1,
                             reduction="sum")
        if abs(r.losses[0] - ((T + U) * math.log(V) - math.log(math.comb(T - 1 + U, U)))) > 1e-10:
            return False
        # multi-blank against its enumeration
        for seed, sigma in [(5, 0.0), (6, 0.3)]:
            x, y, T, U = _case(seed, Tmax=6, Umax=2, V=6)
            big = [(4, 2), (3, 3)]
            y = y % 3
            got = oracle.rnnt_loss_multiblank(x, y, T, U, big, blank=-1, sigma=sigma,
                                              reduction="sum")
            wl, wr, wg = brute.rnnt_loss_multiblank(x, y, T, U, big, blank=-1, sigma=sigma,
                                                    reduction="sum")
            if not (np.allclose(got.losses, wl, rtol=1e-10, atol=1e-12)
                    and np.allclose(got.losses_beta, got.losses, rtol=1e-10, atol=1e-12)
                    and np.allclose(got.grad, wg, rtol=1e-8, atol=1e-11)):
                return False
    except (ValueError, FloatingPointError):
        return False
    return True


def _use_library(monkeypatch, path):
    monkeypatch.setattr(oracle, "_lib", None)
    monkeypatch.setattr(oracle, "build", lambda force=False: path)


@pytest.fixture(scope="module")
def gcc():
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    return "gcc"


def _compile(gcc, src_text, out_dir, name):
    c = os.path.join(out_dir, name + ".c")
    so = os.path.join(out_dir, name + ".so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run([gcc, "-O1", "-std=gnu11", "-fPIC", "-shared", c, "-o", so, "-lm"],
                   check=True, capture_output=True)
    return so


def test_unmodified_oracle_passes_the_pins(gcc, tmp_path, monkeypatch):
    _use_library(monkeypatch, _compile(gcc, open(SRC).read(), str(tmp_path), "clean"))
    assert _pins_pass()


@pytest.mark.parametrize("name,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(gcc, tmp_path, monkeypatch, name, edits):
    src = open(SRC).read()
    mutated = _plant(src, edits)
    assert mutated != src, "the planted edit did not apply"
    _use_library(monkeypatch, _compile(gcc, mutated, str(tmp_path), "mutant"))
    assert not _pins_pass(), f"no pin caught: {name}"
