"""Seeded synthetic inputs for the SparseGemv workloads.

This module draws random numbers and describes workload shapes; it holds
none of the method's arithmetic (no pruning, quantisation, packing or
products), so both the CUDA path's tests/benchmark and the CPU oracle's
tests take their inputs from here without sharing any computation.

All randomness comes from numpy's PCG64 generator seeded explicitly, so a
seed names the same matrix on every machine.

The shapes follow the linear layers of a 7B-class decoder (the paper targets
decode-time GEMV of an LLM's linear layers: Dong et al., "Efficient LLM ad
generation via model compression and parallel verification", sections 1 and
3.2); the paper's own model and ad datasets are not public, so these seeded
LLM-shaped weights stand in for them.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(int(seed)))


def weight_normal(seed: int, rows: int, cols: int, std: float) -> np.ndarray:
    """W ~ N(0, std^2), fp32, rows x cols (out features x in features)."""
    return (rng(seed).standard_normal((rows, cols), dtype=np.float32)
            * np.float32(std))


def weight_outliers(seed: int, rows: int, cols: int, std: float = 0.02,
                    p: float = 0.005, outlier_std: float = 0.2) -> np.ndarray:
    """N(0, std^2) with each element independently replaced, with
    probability p, by a draw from N(0, outlier_std^2)."""
    g = rng(seed)
    w = g.standard_normal((rows, cols), dtype=np.float32) * np.float32(std)
    mask = g.random((rows, cols)) < p
    out = g.standard_normal(int(mask.sum()), dtype=np.float32)
    w[mask] = out * np.float32(outlier_std)
    return w


def weight_heavy_channels(seed: int, rows: int, cols: int, std: float = 0.015,
                          frac: float = 0.01, df: float = 4.0) -> np.ndarray:
    """N(0, std^2), except a seeded `frac` of input channels (columns) drawn
    as std * t(df) / sqrt(df / (df - 2)) so their variance matches."""
    g = rng(seed)
    w = g.standard_normal((rows, cols), dtype=np.float32) * np.float32(std)
    nheavy = max(1, int(round(frac * cols)))
    chans = np.sort(g.choice(cols, size=nheavy, replace=False))
    t = g.standard_t(df, size=(rows, nheavy)).astype(np.float32)
    w[:, chans] = t * np.float32(std / math.sqrt(df / (df - 2.0)))
    return w


def activations(seed: int, m: int, cols: int) -> np.ndarray:
    """x ~ N(0, 1) rounded to binary16 (numpy's round-to-nearest-even),
    m x cols."""
    return rng(seed).standard_normal((m, cols), dtype=np.float32).astype(
        np.float16)


# ---------------------------------------------------------------------------
# Workloads.
# ---------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Gemv:
    """One SparseGemv: a weight matrix with its (N, g) and how to draw it."""
    name: str
    rows: int
    cols: int
    n_keep: int
    group: int
    dist: str          # "normal" | "outliers" | "heavy"
    std: float
    w_seed: int
    x_seed: int

    def weight(self) -> np.ndarray:
        if self.dist == "normal":
            return weight_normal(self.w_seed, self.rows, self.cols, self.std)
        if self.dist == "outliers":
            return weight_outliers(self.w_seed, self.rows, self.cols, self.std)
        if self.dist == "heavy":
            return weight_heavy_channels(self.w_seed, self.rows, self.cols,
                                         self.std)
        raise ValueError(self.dist)

    def x(self, m: int = 1) -> np.ndarray:
        return activations(self.x_seed, m, self.cols)

    def packed_bytes(self) -> int:
        """Algorithmic packed-weight bytes: INT4 values + 2-bit positions +
        binary16 scale and zero per group."""
        kept = self.rows * self.cols * self.n_keep // 4
        return kept // 2 + kept // 4 + 4 * self.rows * (self.cols // self.group)

    def bytes(self, m: int = 1) -> int:
        """Algorithmic bytes of one call: packed W + x + y (binary16)."""
        return self.packed_bytes() + 2 * m * self.cols + 2 * m * self.rows

    def flops(self, m: int = 1) -> int:
        return 2 * m * self.rows * self.cols * self.n_keep // 4


LAYER_7B = (("q", 4096, 4096), ("k", 4096, 4096), ("v", 4096, 4096),
            ("o", 4096, 4096), ("gate", 11008, 4096), ("up", 11008, 4096),
            ("down", 4096, 11008))


def seeded_assignment(seed: int, n: int):
    """Seeded stand-in for the paper's sensitivity analysis (which needs
    calibration data): draw u ~ U(0,1) per matrix, rank by u descending;
    the top ceil(n/2) keep 2:4, the rest 1:4; by rank tertile (sizes
    ceil(n/3), then the rest split evenly) g = 64, 128, 256.
    Returns [(n_keep, group, u)] in matrix order."""
    u = rng(seed).random(n)
    order = np.argsort(-u, kind="stable")
    n24 = (n + 1) // 2
    t1 = -(-n // 3)
    t2 = t1 + (n - t1 + 1) // 2
    out = [None] * n
    for rank, i in enumerate(order):
        n_keep = 2 if rank < n24 else 1
        group = 64 if rank < t1 else (128 if rank < t2 else 256)
        out[i] = (n_keep, group, float(u[i]))
    return out


def config1(seed: int = 0):
    """Single 4096x4096 GEMV, W ~ N(0, 0.02), 2:4, g = 128."""
    return [Gemv("w4096_2of4_g128", 4096, 4096, 2, 128, "normal", 0.02,
                 1000 * seed + 1, 1000 * seed + 501)]


def config2(seed: int = 0):
    """4096x4096 with 0.5% N(0, 0.2) outliers: 1:4 g256 (non-sensitive
    layer) and 2:4 g64 (sensitive layer)."""
    return [Gemv("w4096_1of4_g256_outl", 4096, 4096, 1, 256, "outliers", 0.02,
                 1000 * seed + 11, 1000 * seed + 511),
            Gemv("w4096_2of4_g64_outl", 4096, 4096, 2, 64, "outliers", 0.02,
                 1000 * seed + 12, 1000 * seed + 512)]


def config3(seed: int = 0):
    """7B-style decoder layer set with seeded (N, g) per matrix."""
    asg = seeded_assignment(1000 * seed + 99, len(LAYER_7B))
    return [Gemv(name, r, c, n, g, "normal", 0.02, 1000 * seed + 20 + i,
                 1000 * seed + 520 + i)
            for i, ((name, r, c), (n, g, _)) in enumerate(zip(LAYER_7B, asg))]


def config4(seed: int = 0):
    """The layer set, all 2:4 g = 128 (x has M rows, chosen by the caller)."""
    return [Gemv(name, r, c, 2, 128, "normal", 0.02, 1000 * seed + 40 + i,
                 1000 * seed + 540 + i)
            for i, (name, r, c) in enumerate(LAYER_7B)]


CONFIG4_M = (4, 8, 16, 32, 64)

LARGE = (("w8192", 8192, 8192), ("w28672x8192", 28672, 8192),
         ("w8192x28672", 8192, 28672))


def config5(seed: int = 0):
    """Large layers, g = 128, N(0, 0.015) with 1% Student-t(4) channels;
    N per matrix by the seeded rule."""
    asg = seeded_assignment(1000 * seed + 199, len(LARGE))
    return [Gemv(name, r, c, n, 128, "heavy", 0.015, 1000 * seed + 60 + i,
                 1000 * seed + 560 + i)
            for i, ((name, r, c), (n, _g, _)) in enumerate(zip(LARGE, asg))]


CONFIGS = {"1": config1, "2": config2, "3": config3, "4": config4,
           "5": config5}


def row_groups(seed: int, rows: int, choices=(64, 128, 256)) -> np.ndarray:
    """A group size per row drawn uniformly from `choices` (the stand-in for
    per-channel sensitivity: finer groups for some rows of a layer)."""
    rng = np.random.default_rng([seed, 0x52475250])
    return rng.choice(np.asarray(choices), rows).astype(np.int32)
