"""Seeded synthetic inputs for the RNN-T loss: lengths, targets and logits.

This module only draws random numbers and lays them out; it holds none of the
loss arithmetic.  The same generator feeds both the CUDA path and the float64
oracle, so both read identical bytes.

The five workloads follow the shapes and value distributions of the
rnnt-loss-ascend README accuracy/performance tables ("精度测试", "性能数据":
batches of 2-32, T up to 2000, U up to 500, V from 50 to 50000, random
logits) narrowed to one configuration each:

=============  ==  ==================  ================  =====  =====  =====  =====  =====  =========
name           B   T_b                 U_b               V      dtype  blank  clamp  fused  reduction
=============  ==  ==================  ================  =====  =====  =====  =====  =====  =========
tiny           2   [8, 6]              [3, 2]            16     f32    -1     -1     yes    none
char_asr       32  U[150, 200]         U[20, 40]         29     f32    0      0.1    yes    mean
bpe_asr        16  U[300, 500]         U[50, 100]        1024   f16    -1     off    yes    sum
large_vocab    8   U[500, 1000]        U[100, 200]       5000   f32    0      off    yes    mean
skewed         64  lognormal(5, 0.6)   round(T*U(.1,.2)) 512    f16    -1     0.5    no     mean
=============  ==  ==================  ================  =====  =====  =====  =====  =====  =========

Logits are N(0, sigma) drawn in float32 on the host and cast to the stored
dtype; "skewed" stores float16 log-probabilities (float32 log_softmax of
N(0, 1) draws, via torch.log_softmax) because it runs with the in-kernel
log-softmax disabled; its sample 32 is forced to T=1500, U=300.  Targets are
uniform over the non-blank ids.  Lengths and targets come from
``numpy.random.default_rng(seed)``; the logits of sample b come from a
``torch.Generator`` seeded with ``seed * 1000 + b``, so one sample can be
regenerated on its own for a sampled comparison at full size.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

_DT = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Config:
    name: str
    B: int
    V: int
    dtype: str
    sigma: float
    blank: int
    clamp: float
    fused: bool
    reduction: str
    seed: int
    T: tuple = ()            # fixed lengths (tiny) ...
    U: tuple = ()
    T_range: tuple = ()      # ... or uniform integer ranges (inclusive)
    U_range: tuple = ()
    skewed: bool = False


CONFIGS = {
    "tiny": Config("tiny", 2, 16, "f32", 1.0, -1, -1.0, True, "none", 1001,
                   T=(8, 6), U=(3, 2)),
    "char_asr": Config("char_asr", 32, 29, "f32", 2.0, 0, 0.1, True, "mean", 1002,
                       T_range=(150, 200), U_range=(20, 40)),
    "bpe_asr": Config("bpe_asr", 16, 1024, "f16", 1.5, -1, -1.0, True, "sum", 1003,
                      T_range=(300, 500), U_range=(50, 100)),
    "large_vocab": Config("large_vocab", 8, 5000, "f32", 1.0, 0, -1.0, True, "mean", 1004,
                          T_range=(500, 1000), U_range=(100, 200)),
    "skewed": Config("skewed", 64, 512, "f16", 1.0, -1, 0.5, False, "mean", 1005,
                     skewed=True),
}


def lengths(cfg: Config):
    """(T, U) as int32 arrays of length B."""
    rng = np.random.default_rng(cfg.seed)
    if cfg.T:
        return np.asarray(cfg.T, dtype=np.int32), np.asarray(cfg.U, dtype=np.int32)
    if cfg.skewed:
        T = np.clip(np.rint(rng.lognormal(5.0, 0.6, size=cfg.B)), 20, 1500).astype(np.int64)
        T[cfg.B // 2] = 1500
        U = np.maximum(1, np.rint(T * rng.uniform(0.1, 0.2, size=cfg.B))).astype(np.int64)
        U[cfg.B // 2] = 300
        return T.astype(np.int32), U.astype(np.int32)
    T = rng.integers(cfg.T_range[0], cfg.T_range[1] + 1, size=cfg.B)
    U = rng.integers(cfg.U_range[0], cfg.U_range[1] + 1, size=cfg.B)
    return T.astype(np.int32), U.astype(np.int32)


def targets(cfg: Config, U: np.ndarray) -> np.ndarray:
    """(B, max(U, 1)) int32 labels, uniform over the non-blank ids; padding is 0."""
    rng = np.random.default_rng(cfg.seed + 7919)
    blank = cfg.blank + cfg.V if cfg.blank < 0 else cfg.blank
    S = max(1, int(U.max()))
    if cfg.V == 1:                      # blank is the only class: no labels exist
        return np.zeros((cfg.B, S), dtype=np.int32)
    y = rng.integers(0, cfg.V - 1, size=(cfg.B, S))
    y = np.where(y >= blank, y + 1, y)
    for b in range(cfg.B):
        y[b, int(U[b]):] = 0
    return y.astype(np.int32)


def sample_logits(cfg: Config, b: int, T_b: int, U_b: int) -> torch.Tensor:
    """Host tensor (T_b*(U_b+1), V) of sample b in the stored dtype."""
    g = torch.Generator().manual_seed(cfg.seed * 1000 + b)
    x = torch.randn(T_b * (U_b + 1), cfg.V, generator=g, dtype=torch.float32)
    if cfg.fused:
        x.mul_(cfg.sigma)
    else:
        x = torch.log_softmax(x * cfg.sigma, dim=1)
    return x.to(_DT[cfg.dtype])


@dataclass
class Workload:
    cfg: Config
    T: np.ndarray
    U: np.ndarray
    targets: np.ndarray
    offsets: np.ndarray          # int64, B+1 (plain cumulative sum, layout bookkeeping)
    logits: torch.Tensor         # (rows, V), on the requested device
    extra: dict = field(default_factory=dict)

    @property
    def rows(self) -> int:
        return int(self.offsets[-1])

    @property
    def elements(self) -> int:
        return self.rows * self.cfg.V

    def sample_rows(self, b: int) -> slice:
        return slice(int(self.offsets[b]), int(self.offsets[b + 1]))


def make(name_or_cfg, device="cpu", with_logits: bool = True) -> Workload:
    """Build a workload; logits are generated per sample on the host and copied over."""
    cfg = CONFIGS[name_or_cfg] if isinstance(name_or_cfg, str) else name_or_cfg
    T, U = lengths(cfg)
    y = targets(cfg, U)
    off = np.zeros(cfg.B + 1, dtype=np.int64)
    off[1:] = np.cumsum(T.astype(np.int64) * (U.astype(np.int64) + 1))
    logits = None
    if with_logits:
        logits = torch.empty(int(off[-1]), cfg.V, dtype=_DT[cfg.dtype], device=device)
        for b in range(cfg.B):
            logits[off[b]:off[b + 1]].copy_(sample_logits(cfg, b, int(T[b]), int(U[b])))
    return Workload(cfg, T, U, y, off, logits)


def subset(wl: Workload, n: int) -> Workload:
    """The first n samples of a workload (same bytes), e.g. for a smaller profiling run."""
    from dataclasses import replace
    n = max(1, min(n, wl.cfg.B))
    cfg = replace(wl.cfg, B=n)
    r1 = int(wl.offsets[n])
    return Workload(cfg, wl.T[:n].copy(), wl.U[:n].copy(),
                    np.ascontiguousarray(wl.targets[:n, :max(1, int(wl.U[:n].max()))]),
                    wl.offsets[:n + 1].copy(), wl.logits[:r1])


def custom(B, T, U, V, dtype="f32", sigma=1.0, blank=-1, clamp=-1.0, fused=True,
           reduction="mean", seed=7, device="cpu") -> Workload:
    """A workload with explicit lengths (tests of edge cases)."""
    cfg = Config("custom", B, V, dtype, sigma, blank, clamp, fused, reduction, seed,
                 T=tuple(int(t) for t in T), U=tuple(int(u) for u in U))
    return make(cfg, device=device)


def to_padded(wl: Workload, max_T: int | None = None, max_U: int | None = None,
              fill: float = 0.0) -> torch.Tensor:
    """The workload's logits laid out as a padded (B, max_T, max_U+1, V) tensor.

    Node (t, u) of sample b goes to [b, t, u]; every other entry holds `fill`
    (padding).  Layout only: the same bytes as the compact rows."""
    cfg = wl.cfg
    mT = int(wl.T.max()) if max_T is None else int(max_T)
    mU = int(wl.U.max()) if max_U is None else int(max_U)
    x = torch.full((cfg.B, mT, mU + 1, cfg.V), fill, dtype=wl.logits.dtype,
                   device=wl.logits.device)
    for b in range(cfg.B):
        T, U = int(wl.T[b]), int(wl.U[b])
        x[b, :T, :U + 1].copy_(wl.logits[wl.sample_rows(b)].view(T, U + 1, cfg.V))
    return x
