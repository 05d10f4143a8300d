"""The node-index arithmetic the CUDA kernels use, pinned to its definition.

Every per-node array (transition records, alpha, beta) is laid out in
anti-diagonal-packed order: the nodes of diagonal d = t + u, d = 0, 1, ...,
each diagonal ordered by frame t.  The kernels never build that order; they
compute positions in closed form, step them from frame to frame or column to
column, invert them (node -> (t, u)), and take a 32-bit shortcut for lattices
with T + W <= 65536.  Each formula is restated here as the kernels state it and
checked against a brute-force enumeration of the packing, so that a wrong
term, sign or bound in any of them fails a test."""
import numpy as np
import pytest

M32 = (1 << 32) - 1


def packing(T, U):
    """{(t, u): position} by enumerating the diagonals (the definition)."""
    pos, k = {}, 0
    for d in range(T + U):
        for t in range(max(0, d - U), min(d, T - 1) + 1):
            pos[(t, d - t)] = k
            k += 1
    return pos


def tri(n):
    return n * (n + 1) // 2 if n > 0 else 0


def diag_start(d, T, W):   # nodes before diagonal d, by inclusion-exclusion
    return tri(d) - tri(d - T) - tri(d - W) + tri(d - T - W)


def node_index(t, u, T, U):
    d = t + u
    return diag_start(d, T, U + 1) + t - max(0, d - U)


def node_index32(t, u, T, U):   # unsigned 32-bit arithmetic, wrapping
    d, W = t + u, U + 1
    tri32 = lambda n: ((n * (n + 1)) & M32) >> 1 if n > 0 else 0
    ds = (tri32(d) - tri32(d - T) - tri32(d - W) + tri32(d - T - W)) & M32
    return (ds + t - max(0, d - U)) & M32


def diag_len(d, T, W):
    return min(min(d + 1, min(T, W)), T + W - 1 - d)


def node_diag(k, T, W):
    """Diagonal of node k: a first guess from the lattice's three parts
    (float32 square roots, as on the device), corrected against diag_start."""
    m, M, D = min(T, W), max(T, W), T + W - 1
    head = (m - 1) * m // 2
    f32 = np.float32
    if k < head:
        d = int((np.sqrt(f32(8.0) * f32(k) + f32(1.0)) - f32(1.0)) * f32(0.5))
    elif k < head + (M - m + 1) * m:
        d = m - 1 + (k - head) // m
    else:
        kr = T * W - 1 - k
        d = D - 1 - int((np.sqrt(f32(8.0) * f32(kr) + f32(1.0)) - f32(1.0)) * f32(0.5))
    d = max(0, min(d, D - 1))
    while d > 0 and diag_start(d, T, W) > k:
        d -= 1
    while d + 1 < D and diag_start(d + 1, T, W) <= k:
        d += 1
    return d


SHAPES = [(1, 0), (1, 4), (5, 0), (2, 2), (3, 1), (4, 6), (9, 3), (7, 7), (12, 30), (31, 5)]


@pytest.mark.parametrize("T,U", SHAPES)
def test_closed_form_matches_the_enumerated_packing(T, U):
    pos = packing(T, U)
    assert sorted(pos.values()) == list(range(T * (U + 1)))
    for (t, u), k in pos.items():
        assert node_index(t, u, T, U) == k
        assert node_index32(t, u, T, U) == k


@pytest.mark.parametrize("T,U", SHAPES)
def test_frame_and_column_steps(T, U):
    # idx(t+1, u) - idx(t, u) = len(d) + 1 - [d >= U];  idx(t, u+1) - idx(t, u) = len(d) - [d >= U]
    pos, W = packing(T, U), U + 1
    for (t, u), k in pos.items():
        d = t + u
        if t + 1 < T:
            assert pos[(t + 1, u)] - k == diag_len(d, T, W) + 1 - (d >= U)
        if u < U:
            assert pos[(t, u + 1)] - k == diag_len(d, T, W) - (d >= U)


@pytest.mark.parametrize("T,U", SHAPES)
def test_node_to_frame_and_column(T, U):
    pos, W = packing(T, U), U + 1
    for (t, u), k in pos.items():
        d = node_diag(k, T, W)
        assert d == t + u
        assert k - diag_start(d, T, W) + max(0, d - U) == t


def test_node_diag_on_long_lattices():
    rng = np.random.default_rng(11)
    for T, U in [(1500, 300), (300, 1023), (65536, 0), (40000, 1023), (1, 1023)]:
        W = U + 1
        ks = list(rng.integers(0, T * W, 3000)) + [0, T * W - 1]
        for k in map(int, ks):
            d = node_diag(k, T, W)
            assert diag_start(d, T, W) <= k < diag_start(d + 1, T, W)


def test_32_bit_path_on_the_largest_lattices_it_takes():
    # T + W <= 65536: every triangular number is below 2^32, the index below 2^31.
    rng = np.random.default_rng(12)
    for T, U in [(65535, 0), (64512, 1023), (32768, 32767), (2, 65533)]:
        assert T + U + 1 <= 65536
        for _ in range(2000):
            t, u = int(rng.integers(0, T)), int(rng.integers(0, U + 1))
            k = node_index(t, u, T, U)
            assert node_index32(t, u, T, U) == k < 2 ** 31


def test_offsets_inside_the_band_of_full_length_diagonals():
    # For T >= W and U <= t + u, t + u + k <= T - 1: (t + k, u) is k W nodes
    # further and (t, u + 1) is W - 1 nodes further.
    for T, U in [(12, 3), (40, 9), (9, 8)]:
        pos, W = packing(T, U), U + 1
        for (t, u), i in pos.items():
            d = t + u
            for k in range(1, 17):
                if d >= U and d + k <= T - 1:
                    assert pos[(t + k, u)] == i + k * W
            if d >= U and d + 1 <= T - 1 and u < U:
                assert pos[(t, u + 1)] == i + W - 1


def test_warp_wide_sample_search():
    # The 32-way search over sample offsets: off[lo] <= r < off[lo + 1].
    def search(off, B, r):
        lo, n = 0, B
        while n > 1:
            step = (n + 31) // 32
            hits = [lo + l * step < lo + n and off[lo + l * step] <= r for l in range(32)]
            k = max(i for i, h in enumerate(hits) if h)
            lo += k * step
            n = min(step, n - k * step)
        return lo
    rng = np.random.default_rng(13)
    for B in [1, 2, 31, 32, 33, 64, 1000, 1025, 5000]:
        off = np.concatenate([[0], np.cumsum(rng.integers(1, 40, B))])
        for r in list(rng.integers(0, off[-1], 500)) + [0, off[-1] - 1]:
            assert search(off, B, int(r)) == int(np.searchsorted(off, r, side="right") - 1)
