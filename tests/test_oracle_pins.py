"""Pins of the float64 oracle to things other than itself (CPU only).

No page prints a worked numeric example, so the oracle is pinned by:
  * brute-force enumeration of every alignment (oracle/brute.py, autograd
    for the gradient) on tiny lattices, fused and non-fused, clamp and every
    reduction, float32 and float16 rows;
  * closed forms: T=1,U=0 (loss = -log_softmax(h)[blank]); U=0 (blanks
    only); T=1 (all labels then the terminal blank); constant logits
    (combinatorial loss, occupancies and gradient) incl. the stored fixture
    tests/golden/uniform_logits.json;
  * invariants: loss from alpha == loss from beta, per-anti-diagonal
    occupancy sums to 1, zero gradient row sums with fused log-softmax,
    each frame crossed by exactly one blank and each label emitted once;
  * central finite differences of the oracle's own loss.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import log_softmax, logsumexp

import oracle
from oracle import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_case(rng, B, Tmax, Umax, V, dtype=np.float32, sigma=1.0, blank=None, fused=True):
    T = rng.integers(1, Tmax + 1, size=B).astype(np.int32)
    U = rng.integers(0, Umax + 1, size=B).astype(np.int32)
    if blank is None:
        blank = int(rng.integers(-V, V))
    bl = blank + V if blank < 0 else blank
    S = max(1, int(U.max()))
    y = rng.integers(0, V - 1, size=(B, S))
    y = np.where(y >= bl, y + 1, y).astype(np.int32)
    rows = int((T.astype(np.int64) * (U + 1)).sum())
    x = rng.normal(0.0, sigma, size=(rows, V))
    if not fused:
        x = log_softmax(x, axis=1)
    return x.astype(dtype), y, T, U, blank


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("fused", [True, False])
def test_brute_force_loss_and_grad(seed, fused):
    rng = np.random.default_rng(100 + seed)
    V = int(rng.integers(2, 7))
    x, y, T, U, blank = rand_case(rng, B=3, Tmax=4, Umax=4, V=V, fused=fused,
                                  dtype=np.float16 if seed % 3 == 0 else np.float32)
    clamp = [-1.0, 0.0, 0.05, 0.3][seed % 4]
    red = ["none", "sum", "mean"][seed % 3]
    got = oracle.rnnt_loss(x, y, T, U, blank=blank, clamp=clamp, reduction=red,
                           fused_log_softmax=fused)
    want_l, want_red, want_g = brute.rnnt_loss(x.astype(np.float64), y, T, U, blank=blank,
                                               clamp=clamp, reduction=red,
                                               fused_log_softmax=fused)
    np.testing.assert_allclose(got.losses, want_l, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(got.losses_beta, want_l, rtol=1e-12, atol=1e-12)
    assert got.reduced == pytest.approx(want_red, rel=1e-12, abs=1e-12)
    np.testing.assert_allclose(got.grad, want_g, rtol=1e-10, atol=1e-12)


def test_brute_force_enumerates_binomial_paths():
    for T in range(1, 6):
        for U in range(0, 5):
            assert sum(1 for _ in brute.alignments(T, U)) == math.comb(T - 1 + U, U)


@pytest.mark.parametrize("V,blank", [(5, -1), (7, 0), (3, 1)])
def test_closed_form_single_node(V, blank):
    rng = np.random.default_rng(V)
    h = rng.normal(0, 2.0, size=(1, V))
    fw = oracle.sample_forward(h, 1, 0, [], blank, True)
    bl = blank + V if blank < 0 else blank
    assert fw.loss_alpha == pytest.approx(-(h[0, bl] - logsumexp(h[0])), abs=1e-13)
    assert fw.loss_beta == pytest.approx(fw.loss_alpha, abs=1e-13)


def test_closed_form_blanks_only():
    rng = np.random.default_rng(1)
    T, V = 23, 9
    h = rng.normal(0, 1.5, size=(T, V))
    fw = oracle.sample_forward(h, T, 0, [], 4, True)
    assert fw.loss_alpha == pytest.approx(-log_softmax(h, axis=1)[:, 4].sum(), rel=1e-13)


def test_closed_form_single_frame():
    rng = np.random.default_rng(2)
    U, V = 6, 10
    y = [3, 1, 1, 8, 2, 5]
    h = rng.normal(0, 1.5, size=(U + 1, V))
    lp = log_softmax(h, axis=1)
    want = -(sum(lp[u, y[u]] for u in range(U)) + lp[U, 0])
    fw = oracle.sample_forward(h, 1, U, y, 0, True)
    assert fw.loss_alpha == pytest.approx(want, rel=1e-13)


def log_binom(n, k):
    return math.lgamma(n + 1) - math.lgamma(k + 1) - math.lgamma(n - k + 1)


def uniform_grad(T, U, V, y, blank, fused=True):
    """Closed-form gradient for constant logits (every p = 1/V).

    Occupancy of node (t,u) = C(t+u,u) C(T-1-t+U-u, U-u) / C(T-1+U, U); the
    blank arc out of it is taken by C(t+u,u) C(T-2-t+U-u, U-u) of those
    alignments (all of them at the terminal node), the label arc by
    C(t+u,u) C(T-1-t+U-u-1, U-u-1).
    """
    W = U + 1
    tot = log_binom(T - 1 + U, U)
    g = np.zeros((T * W, V))
    for t in range(T):
        for u in range(W):
            before = log_binom(t + u, u)
            occ = math.exp(before + log_binom(T - 1 - t + U - u, U - u) - tot)
            if t < T - 1:
                eb = math.exp(before + log_binom(T - 2 - t + U - u, U - u) - tot)
            else:
                eb = occ if u == U else 0.0
            ey = math.exp(before + log_binom(T - 1 - t + U - u - 1, U - u - 1) - tot) \
                if u < U else 0.0
            r = t * W + u
            if fused:
                g[r, :] = occ / V
            g[r, blank] -= eb
            if u < U:
                g[r, y[u]] -= ey
    return g


@pytest.mark.parametrize("T,U,V,blank", [(1, 0, 4, 0), (5, 3, 6, 5), (40, 12, 16, 0),
                                         (120, 30, 8, 7)])
def test_closed_form_uniform_logits(T, U, V, blank):
    rng = np.random.default_rng(T * 31 + U)
    y = rng.integers(0, V - 1, size=max(U, 1))
    y = np.where(y >= blank, y + 1, y).astype(np.int32)
    h = np.full((T * (U + 1), V), 0.37)
    fw = oracle.sample_forward(h, T, U, y, blank, True)
    want = (T + U) * math.log(V) - log_binom(T - 1 + U, U)
    assert fw.loss_alpha == pytest.approx(want, rel=1e-12, abs=1e-12)
    g = oracle.sample_grad(h, fw, y, blank, True, -1.0, 1.0)
    np.testing.assert_allclose(g, uniform_grad(T, U, V, y, blank), rtol=1e-9, atol=1e-13)
    # Same lattice given as log-probabilities (in-kernel log-softmax off).
    lp = np.full_like(h, -math.log(V))
    fwn = oracle.sample_forward(lp, T, U, y, blank, False)
    assert fwn.loss_alpha == pytest.approx(want, rel=1e-12, abs=1e-12)
    gn = oracle.sample_grad(lp, fwn, y, blank, False, -1.0, 1.0)
    np.testing.assert_allclose(gn, uniform_grad(T, U, V, y, blank, fused=False), rtol=1e-9,
                               atol=1e-13)


def test_golden_uniform_fixture():
    with open(os.path.join(GOLDEN, "uniform_logits.json")) as f:
        fx = json.load(f)
    for case in fx["cases"]:
        V = case["V"]
        for T, U, want in zip(case["T"], case["U"], case["losses"]):
            y = np.arange(U, dtype=np.int32) % (V - 1)  # blank = V-1 never used as a label
            h = np.zeros((T * (U + 1), V), dtype=np.float32)
            fw = oracle.sample_forward(h, T, U, y, -1, True)
            assert fw.loss_alpha == pytest.approx(want, rel=1e-11), case["name"]
            assert fw.loss_beta == pytest.approx(want, rel=1e-11), case["name"]


@pytest.mark.parametrize("fused", [True, False])
def test_invariants_random(fused):
    rng = np.random.default_rng(5 if fused else 6)
    T, U, V, blank = 60, 17, 12, 0
    y = rng.integers(1, V, size=U).astype(np.int32)
    h = rng.normal(0, 2.0, size=(T * (U + 1), V))
    if not fused:
        h = log_softmax(h, axis=1)
    fw = oracle.sample_forward(h, T, U, y, blank, fused)
    assert fw.loss_alpha == pytest.approx(fw.loss_beta, rel=1e-12)
    W = U + 1
    a = fw.alpha.reshape(T, W)
    b = fw.beta.reshape(T, W)
    for d in range(T + U):
        cells = [(t, d - t) for t in range(max(0, d - U), min(T - 1, d) + 1)]
        occ = sum(math.exp(a[t, u] + b[t, u] - fw.ll) for t, u in cells)
        assert occ == pytest.approx(1.0, abs=1e-10)
    g = oracle.sample_grad(h, fw, y, blank, fused, -1.0, 1.0)
    if fused:
        np.testing.assert_allclose(g.sum(axis=1), 0.0, atol=1e-12)
    else:
        gb = g[:, blank].reshape(T, W)
        np.testing.assert_allclose(gb.sum(axis=1), -1.0, atol=1e-10)
        gy = np.array([[g[t * W + u, y[u]] for u in range(U)] for t in range(T)])
        np.testing.assert_allclose(gy.sum(axis=0), -1.0, atol=1e-10)
        mask = np.ones_like(g, dtype=bool)
        mask[:, blank] = False
        for t in range(T):
            for u in range(U):
                mask[t * W + u, y[u]] = False
        assert np.all(g[mask] == 0.0)


@pytest.mark.parametrize("fused", [True, False])
def test_central_finite_differences(fused):
    rng = np.random.default_rng(9 if fused else 10)
    T, U, V, blank = 5, 3, 5, 2
    y = np.array([0, 4, 1], dtype=np.int32)
    h = rng.normal(0, 1.0, size=(T * (U + 1), V))
    if not fused:
        h = log_softmax(h, axis=1)
    fw = oracle.sample_forward(h, T, U, y, blank, fused)
    g = oracle.sample_grad(h, fw, y, blank, fused, -1.0, 1.0)
    eps = 1e-6
    fd = np.zeros_like(h)
    for i in range(h.shape[0]):
        for k in range(V):
            hp = h.copy()
            hp[i, k] += eps
            hm = h.copy()
            hm[i, k] -= eps
            lp_ = oracle.sample_forward(hp, T, U, y, blank, fused).loss_alpha
            lm_ = oracle.sample_forward(hm, T, U, y, blank, fused).loss_alpha
            fd[i, k] = (lp_ - lm_) / (2 * eps)
    np.testing.assert_allclose(g, fd, atol=2e-8)


def test_offsets_exact():
    T = np.array([8, 6, 1, 1000], dtype=np.int32)
    U = np.array([3, 2, 0, 299], dtype=np.int32)
    np.testing.assert_array_equal(oracle.offsets(T, U), [0, 32, 50, 51, 300051])


def test_grad_rows_slice_matches_full():
    rng = np.random.default_rng(3)
    T, U, V = 9, 4, 7
    y = np.array([1, 2, 3, 4], dtype=np.int32)
    h = rng.normal(size=(T * (U + 1), V)).astype(np.float32)
    fw = oracle.sample_forward(h, T, U, y, 0, True)
    full = oracle.sample_grad(h, fw, y, 0, True, 0.2, 0.5)
    part = oracle.sample_grad(h, fw, y, 0, True, 0.2, 0.5, 11, 29)
    np.testing.assert_array_equal(full[11:29], part)


def test_rejects_bad_arguments():
    h = np.zeros((4, 3))
    with pytest.raises(ValueError):
        oracle.sample_forward(h, 0, 3, [0, 1, 0], 2, True)
    with pytest.raises(ValueError):
        oracle.rnnt_loss(h.astype(np.float32), [[0]], [2], [2], blank=2)


@pytest.mark.parametrize("bad", [-1, 5, 4, -3])
def test_rejects_invalid_labels(bad):
    # A label outside [0, V) or equal to blank is an invalid input (warp-transducer
    # blog 4.4 / 5.2); the oracle refuses it in every entry point, as the CUDA path
    # reports RNNT_INVALID_VALUE for it.  V = 5, blank = -1 -> 4; -3 stays invalid
    # (labels are never counted from the end).
    V, T, U = 5, 3, 2
    rng = np.random.default_rng(0)
    x = rng.normal(size=(T * (U + 1), V)).astype(np.float32)
    good = [1, 2]
    fw = oracle.sample_forward(x, T, U, good, -1, True)
    y = [1, bad]
    with pytest.raises(ValueError):
        oracle.sample_forward(x, T, U, y, -1, True)
    with pytest.raises(ValueError):
        oracle.sample_grad(x, fw, y, -1, True, -1.0, 1.0)
    with pytest.raises(ValueError):
        oracle.rnnt_loss(x, [y], [T], [U], blank=-1)
    with pytest.raises(ValueError):
        oracle.rnnt_loss_multiblank(x, [y], [T], [U], [(3, 2)], blank=-1)
    # Entries past the target length are padding and are never read.
    r = oracle.rnnt_loss(x, [[1, 2, bad]], [T], [U], blank=-1)
    assert np.isfinite(r.losses[0])


def test_multiblank_rejects_a_label_equal_to_a_big_blank():
    V, T, U = 6, 4, 2
    x = np.random.default_rng(1).normal(size=(T * (U + 1), V))
    with pytest.raises(ValueError):
        oracle.rnnt_loss_multiblank(x, [[1, 3]], [T], [U], [(3, 2)], blank=-1)
    r = oracle.rnnt_loss_multiblank(x, [[1, 2]], [T], [U], [(3, 2)], blank=-1)
    assert np.isfinite(r.losses[0])


# ---------------------------------------------------------------- FastEmit
# The GPURNNT docs and compute_multiblank_grad_kernel take a FastEmit weight
# lambda; the reading used here: the gradient term of every label-emission
# log-probability is scaled by 1 + lambda, blank terms and the loss are not.

@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("fused", [True, False])
def test_fastemit_brute_force(seed, fused):
    rng = np.random.default_rng(700 + seed)
    V = int(rng.integers(2, 7))
    x, y, T, U, blank = rand_case(rng, B=3, Tmax=4, Umax=4, V=V, fused=fused)
    lam = [0.01, 0.3, 1.0, 2.5][seed % 4]
    clamp = [-1.0, 0.2][seed % 2]
    red = ["none", "sum", "mean"][seed % 3]
    got = oracle.rnnt_loss(x, y, T, U, blank=blank, clamp=clamp, reduction=red,
                           fused_log_softmax=fused, fastemit_lambda=lam)
    want_l, want_red, want_g = brute.rnnt_loss(x.astype(np.float64), y, T, U, blank=blank,
                                               clamp=clamp, reduction=red,
                                               fused_log_softmax=fused, fastemit_lambda=lam)
    np.testing.assert_allclose(got.losses, want_l, rtol=1e-12, atol=1e-12)
    assert got.reduced == pytest.approx(want_red, rel=1e-12, abs=1e-12)
    np.testing.assert_allclose(got.grad, want_g, rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("fused", [True, False])
def test_fastemit_linear_in_lambda_and_loss_unchanged(fused):
    rng = np.random.default_rng(77)
    x, y, T, U, blank = rand_case(rng, B=4, Tmax=9, Umax=6, V=6, fused=fused)
    r = {lam: oracle.rnnt_loss(x, y, T, U, blank=blank, reduction="sum", fused_log_softmax=fused,
                               fastemit_lambda=lam) for lam in (0.0, 1.0, 0.37)}
    np.testing.assert_array_equal(r[0.37].losses, r[0.0].losses)
    d1 = r[1.0].grad - r[0.0].grad
    np.testing.assert_allclose(r[0.37].grad - r[0.0].grad, 0.37 * d1, rtol=1e-9, atol=1e-13)
    assert np.abs(d1).max() > 1e-3   # the term is not empty


def test_fastemit_label_gradients_sum_per_label():
    # Non-fused: the gradient at label entries is -(1+lambda) times the label
    # posteriors, and every label is emitted exactly once on every alignment,
    # so summing over frames gives -(1+lambda) for each label position u.
    rng = np.random.default_rng(78)
    lam = 0.6
    x, y, T, U, blank = rand_case(rng, B=1, Tmax=12, Umax=7, V=9, fused=False, blank=-1)
    T0, U0 = int(T[0]), int(U[0])
    if U0 == 0:
        pytest.skip("no labels drawn")
    res = oracle.rnnt_loss(x, y, T, U, blank=blank, reduction="sum", fused_log_softmax=False,
                           fastemit_lambda=lam)
    g = res.grad.reshape(T0, U0 + 1, -1)
    for u in range(U0):
        assert g[:, u, y[0, u]].sum() == pytest.approx(-(1 + lam), abs=1e-12)
    # blank entries: each frame is left by exactly one blank
    for t in range(T0):
        assert g[t, :, 8].sum() == pytest.approx(-1.0, abs=1e-12)


def test_fastemit_fused_rows_sum_to_zero():
    rng = np.random.default_rng(79)
    x, y, T, U, blank = rand_case(rng, B=3, Tmax=10, Umax=6, V=7)
    g = oracle.rnnt_loss(x, y, T, U, blank=blank, reduction="sum", fastemit_lambda=1.3).grad
    np.testing.assert_allclose(g.sum(axis=1), 0.0, atol=1e-12)


# ---------------------------------------------------------------- padded layout
# The ESPnet GPURNNT docs take activations of shape [B, T, U, V+1]: node (t, u)
# of sample b at [b, t, u]; positions outside a sample's lattice are padding.

def rand_padded(rng, B, maxT, maxU, V, fused=True, junk=50.0):
    T = rng.integers(1, maxT + 1, size=B).astype(np.int32)
    U = rng.integers(0, maxU + 1, size=B).astype(np.int32)
    T[0], U[-1] = maxT, maxU          # some sample fills each padded dimension
    x = rng.normal(0.0, 1.0, size=(B, maxT, maxU + 1, V))
    if not fused:
        x = log_softmax(x, axis=-1)
    for b in range(B):                # junk outside the lattices
        x[b, T[b]:] = junk
        x[b, :, U[b] + 1:] = -junk
    blank = -1
    y = rng.integers(0, V - 1, size=(B, max(1, maxU))).astype(np.int32)
    return x, y, T, U, blank


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("fused", [True, False])
def test_padded_brute_force(seed, fused):
    rng = np.random.default_rng(900 + seed)
    x, y, T, U, blank = rand_padded(rng, B=3, maxT=4, maxU=3, V=5, fused=fused)
    lam = [0.0, 0.5][seed % 2]
    clamp = [-1.0, 0.1, 0.3][seed % 3]
    red = ["none", "sum", "mean"][seed % 3]
    got = oracle.rnnt_loss_padded(x, y, T, U, blank=blank, clamp=clamp, reduction=red,
                                  fused_log_softmax=fused, fastemit_lambda=lam)
    wl, wr, wg = brute.rnnt_loss_padded(x, y, T, U, blank=blank, clamp=clamp, reduction=red,
                                        fused_log_softmax=fused, fastemit_lambda=lam)
    np.testing.assert_allclose(got.losses, wl, rtol=1e-12, atol=1e-12)
    assert got.reduced == pytest.approx(wr, rel=1e-12, abs=1e-12)
    np.testing.assert_allclose(got.grad, wg, rtol=1e-10, atol=1e-12)


def test_padded_ignores_padding_and_zeroes_its_gradient():
    rng = np.random.default_rng(950)
    x, y, T, U, blank = rand_padded(rng, B=4, maxT=9, maxU=6, V=7)
    a = oracle.rnnt_loss_padded(x, y, T, U, blank=blank, reduction="sum")
    x2 = x.copy()
    for b in range(4):
        x2[b, T[b]:] = rng.normal(size=x2[b, T[b]:].shape) * 1e3
        x2[b, :, U[b] + 1:] = np.nan
    b2 = oracle.rnnt_loss_padded(x2, y, T, U, blank=blank, reduction="sum")
    np.testing.assert_array_equal(a.losses, b2.losses)
    np.testing.assert_array_equal(a.grad, b2.grad)
    for b in range(4):
        assert not a.grad[b, T[b]:].any() and not a.grad[b, :, U[b] + 1:].any()
        # inside the lattice the gradient is the compact oracle's
        c = oracle.rnnt_loss(np.ascontiguousarray(x[b, :T[b], :U[b] + 1].reshape(-1, 7)),
                             y[b:b + 1], T[b:b + 1], U[b:b + 1], blank=blank, reduction="sum")
        np.testing.assert_array_equal(a.grad[b, :T[b], :U[b] + 1].reshape(-1, 7), c.grad)


# ---------------------------------------------------------------- multi-blank
# ESPnet compute_multiblank_grad_kernel docs: big blanks with durations and a
# logit under-normalisation sigma.  Readings are stated in rnnt_oracle.c.

def rand_mb(rng, B, Tmax, Umax, V, K, fused=True):
    x, y, T, U, _ = rand_case(rng, B=B, Tmax=Tmax, Umax=Umax, V=V, fused=fused, blank=V - 1)
    # big blanks take the outputs just below the standard blank (V-1); labels avoid them
    big = [(V - 2 - i, [2, 3, 4][i % 3]) for i in range(K)]
    y = (y % (V - 1 - K)).astype(np.int32)
    return x, y, T, U, V - 1, big


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("fused", [True, False])
def test_multiblank_brute_force(seed, fused):
    rng = np.random.default_rng(300 + seed)
    K = 1 + seed % 2
    x, y, T, U, blank, big = rand_mb(rng, B=3, Tmax=6, Umax=3, V=6, K=K, fused=fused)
    sigma = [0.0, 0.05, 0.3][seed % 3]
    lam = [0.0, 0.4][seed % 2]
    clamp = [-1.0, 0.2][(seed // 2) % 2]
    red = ["none", "sum", "mean"][seed % 3]
    got = oracle.rnnt_loss_multiblank(x, y, T, U, big, blank=blank, sigma=sigma, clamp=clamp,
                                      reduction=red, fused_log_softmax=fused,
                                      fastemit_lambda=lam)
    wl, wr, wg = brute.rnnt_loss_multiblank(x.astype(np.float64), y, T, U, big, blank=blank,
                                            sigma=sigma, clamp=clamp, reduction=red,
                                            fused_log_softmax=fused, fastemit_lambda=lam)
    np.testing.assert_allclose(got.losses, wl, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(got.losses_beta, wl, rtol=1e-12, atol=1e-12)
    assert got.reduced == pytest.approx(wr, rel=1e-12, abs=1e-12)
    np.testing.assert_allclose(got.grad, wg, rtol=1e-10, atol=1e-12)


def test_multiblank_path_counts():
    # one big blank of duration 2, U=0: compositions of T into parts 1 and 2
    # (Fibonacci numbers); with U labels interleaved the count grows accordingly.
    fib = [1, 1]
    for _ in range(10):
        fib.append(fib[-1] + fib[-2])
    for T in range(1, 9):
        assert len(brute.multiblank_paths(T, 0, [2])) == fib[T]
    assert len(brute.multiblank_paths(4, 0, [])) == 1
    assert len(brute.multiblank_paths(3, 2, [])) == math.comb(3 - 1 + 2, 2)


def test_multiblank_without_big_blanks_is_the_transducer_loss():
    rng = np.random.default_rng(310)
    x, y, T, U, blank = rand_case(rng, B=4, Tmax=9, Umax=5, V=7, blank=-1)
    a = oracle.rnnt_loss_multiblank(x, y, T, U, [], blank=blank, reduction="sum")
    b = oracle.rnnt_loss(x, y, T, U, blank=blank, reduction="sum")
    np.testing.assert_allclose(a.losses, b.losses, rtol=1e-13)
    np.testing.assert_allclose(a.grad, b.grad, atol=1e-14)


def test_multiblank_sigma_shifts_standard_loss_exactly():
    # With no big blanks every alignment has T+U emissions: the loss grows by
    # (T+U)*sigma and the gradient is unchanged.
    rng = np.random.default_rng(311)
    x, y, T, U, blank = rand_case(rng, B=3, Tmax=8, Umax=5, V=6, blank=2)
    a = oracle.rnnt_loss_multiblank(x, y, T, U, [], blank=blank, sigma=0.0, reduction="sum")
    b = oracle.rnnt_loss_multiblank(x, y, T, U, [], blank=blank, sigma=0.7, reduction="sum")
    np.testing.assert_allclose(b.losses - a.losses, 0.7 * (T + U), rtol=1e-12)
    np.testing.assert_allclose(a.grad, b.grad, atol=1e-13)


def test_multiblank_rows_sum_to_zero_and_finite_differences():
    rng = np.random.default_rng(312)
    x, y, T, U, blank, big = rand_mb(rng, B=2, Tmax=9, Umax=4, V=7, K=2)
    x = x.astype(np.float64)
    r = oracle.rnnt_loss_multiblank(x, y, T, U, big, blank=blank, sigma=0.1, reduction="sum")
    np.testing.assert_allclose(r.grad.sum(axis=1), 0.0, atol=1e-12)
    eps = 1e-6
    for (i, k) in [(0, 0), (3, blank), (5, big[0][0]), (7, big[1][0]), (x.shape[0] - 1, 1)]:
        xp, xm = x.copy(), x.copy()
        xp[i, k] += eps
        xm[i, k] -= eps
        lp_ = oracle.rnnt_loss_multiblank(xp, y, T, U, big, blank=blank, sigma=0.1,
                                          reduction="sum", want_grad=False).reduced
        lm_ = oracle.rnnt_loss_multiblank(xm, y, T, U, big, blank=blank, sigma=0.1,
                                          reduction="sum", want_grad=False).reduced
        assert (lp_ - lm_) / (2 * eps) == pytest.approx(r.grad[i, k], abs=1e-7)


# ---------------------------------------------------------------- degenerate vocabularies
def test_blank_only_vocabulary_has_zero_loss_and_gradient():
    # V = 1: the blank is the only output, so p(blank) = 1 at every node, no
    # label can exist (U = 0), the only alignment has probability 1.
    x = np.random.default_rng(5).normal(size=(9, 1))
    r = oracle.rnnt_loss(x, [[0]], [9], [0], blank=0, reduction="sum")
    assert r.losses[0] == pytest.approx(0.0, abs=1e-15)
    np.testing.assert_allclose(r.grad, 0.0, atol=1e-15)


def test_certain_alignment_has_zero_loss_and_a_sharp_gradient():
    # Log-probabilities that put probability 1 on one monotone path (labels at
    # frame 0, then blanks): loss 0, and the non-fused gradient is -1 exactly on
    # that path's arcs, 0 elsewhere.
    T, U, V = 4, 2, 4
    y = [1, 2]
    lp = np.full((T * (U + 1), V), -np.inf)
    W = U + 1
    for t in range(T):
        for u in range(W):
            r = t * W + u
            if t == 0 and u < U:
                lp[r, y[u]] = 0.0           # emit the labels first
            elif u == U:
                lp[r, 0] = 0.0              # then only blanks
    got = oracle.rnnt_loss(lp, [y], [T], [U], blank=0, reduction="sum",
                           fused_log_softmax=False)
    assert got.losses[0] == pytest.approx(0.0, abs=1e-15)
    want = np.zeros_like(lp)
    want[0 * W + 0, 1] = want[0 * W + 1, 2] = -1.0
    for t in range(T):
        want[t * W + U, 0] = -1.0
    np.testing.assert_allclose(got.grad, want, atol=1e-15)


def test_padded_multiblank_matches_its_enumeration():
    # Padded layout and big blanks together, against the enumerator that
    # indexes the padded tensor (big blanks folded into the compact pass).
    rng = np.random.default_rng(960)
    x, y, T, U, blank = rand_padded(rng, B=2, maxT=6, maxU=2, V=6)
    big = [(4, 2), (3, 3)]
    y = (y % 3).astype(np.int32)
    got = oracle.rnnt_loss_padded(x, y, T, U, blank=-1, reduction="sum", big_blanks=big,
                                  sigma=0.1)
    comp = np.concatenate([x[b, :T[b], :U[b] + 1].reshape(-1, 6) for b in range(2)])
    wl, wr, wg = brute.rnnt_loss_multiblank(comp, y, T, U, big, blank=-1, sigma=0.1,
                                            reduction="sum")
    np.testing.assert_allclose(got.losses, wl, rtol=1e-12, atol=1e-12)
    r = 0
    for b in range(2):
        n = int(T[b] * (U[b] + 1))
        np.testing.assert_allclose(got.grad[b, :T[b], :U[b] + 1].reshape(-1, 6), wg[r:r + n],
                                   rtol=1e-10, atol=1e-12)
        assert not got.grad[b, T[b]:].any() and not got.grad[b, :, U[b] + 1:].any()
        r += n
