"""Seeded synthetic inputs for the SNACK sparse layer.

This module only draws inputs: sparsity patterns, weight values and dense
activations / gradients.  It contains none of the layer's arithmetic, so both
the CUDA path and the CPU oracle can be fed from it without sharing any
computation.  Everything is numpy (PCG64) seeded; the same seed gives the same
arrays on every machine.

The shapes follow the workloads of "Beyond Masked Sparsity: SNACK Enables
Truly Sparse Neural Networks on GPU": the 256x256 toy layer, the GPT-2-small
MLP projections (768<->3072), the 10000x10000 single-layer training cycle
(§4.2), a skewed graph-style 8192x8192 layer standing in for the GAMLP
feature head on ogbn-products (§5, Appendix G; no graph data is used), and a
GPT-2-small-shaped decoder's projections (Tables 4-5; no WikiText data).

Patterns are returned in a shuffled "user" order: the library must
canonicalise them itself.
"""

from __future__ import annotations

from dataclasses import dataclass, field
from fractions import Fraction

import numpy as np


def nnz_for(out: int, inp: int, sparsity_pct) -> int:
    """Stored entries of an out x in layer at the given sparsity (percent).

    (1 - eta) * out * in rounded half up, computed exactly: 90% of 256x256
    gives 6553.6 -> 6554."""
    dens = 1 - Fraction(str(sparsity_pct)) / 100
    x = dens * out * inp
    return int((2 * x + 1) // 2)


def _rng(seed: int, *salt: int) -> np.random.Generator:
    return np.random.default_rng([int(seed)] + [int(s) for s in salt])


def uniform_pattern(out: int, inp: int, nnz: int, seed: int):
    """nnz distinct cells drawn uniformly without replacement, shuffled.

    Returns (row, col) int32 arrays in a random order."""
    g = _rng(seed, 1)
    n = out * inp
    if nnz * 2 > n:
        cells = g.choice(n, size=nnz, replace=False, shuffle=True).astype(np.int64)
    else:
        # Distinct values of an i.i.d. uniform stream form, given their
        # number, a uniform random subset; a uniform random nnz-subset of it
        # (in random order) is then a uniform sample without replacement.
        m = int(nnz * 1.25) + 64
        while True:
            cells = np.sort(g.integers(0, n, size=m, dtype=np.int64))
            cells = cells[np.concatenate(([True], cells[1:] != cells[:-1]))]
            if cells.size >= nnz:
                break
            m *= 2
        cells = g.permutation(cells)[:nnz]
    return (cells // inp).astype(np.int32), (cells % inp).astype(np.int32)


def zipf_rank_degrees(out: int, inp: int, nnz: int, s: float, seed: int) -> np.ndarray:
    """Per-row counts with a rank-Zipf(s) profile, capped at `inp`, summing to nnz.

    Row of rank r (1-based) gets weight r^-s; a common scale c is found so
    that sum_r min(inp, c * w_r) = nnz (water filling), counts are rounded by
    largest remainder with at least one entry per row, and the rows are then
    placed in a seeded random order."""
    if nnz < out or nnz > out * inp:
        raise ValueError("zipf_rank_degrees needs out <= nnz <= out*in")
    w = np.arange(1, out + 1, dtype=np.float64) ** (-float(s))
    lo, hi = 0.0, float(inp) / w[-1] * 2 + 1
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if np.minimum(inp, np.maximum(1.0, mid * w)).sum() < nnz:
            lo = mid
        else:
            hi = mid
    target = np.minimum(float(inp), np.maximum(1.0, hi * w))
    counts = np.floor(target).astype(np.int64)
    short = nnz - int(counts.sum())
    if short > 0:
        frac = target - counts
        frac[counts >= inp] = -1.0
        order = np.argsort(-frac, kind="stable")
        counts[order[:short]] += 1
    elif short < 0:
        order = np.argsort(target - counts, kind="stable")
        i = 0
        while short < 0:
            if counts[order[i]] > 1:
                counts[order[i]] -= 1
                short += 1
            i += 1
    assert counts.sum() == nnz and counts.min() >= 1 and counts.max() <= inp
    perm = _rng(seed, 2).permutation(out)
    deg = np.empty(out, np.int64)
    deg[perm] = counts
    return deg


def zipf_pattern(out: int, inp: int, nnz: int, s: float, seed: int):
    """Skewed pattern: rank-Zipf row degrees, columns uniform without
    replacement within each row.  Returns shuffled (row, col) int32."""
    deg = zipf_rank_degrees(out, inp, nnz, s, seed)
    g = _rng(seed, 3)
    rows = np.repeat(np.arange(out, dtype=np.int64), deg)
    cols = np.empty(nnz, np.int64)
    pos = 0
    for r in range(out):
        d = int(deg[r])
        if d == inp:
            cols[pos:pos + d] = np.arange(inp)
        else:
            cols[pos:pos + d] = g.choice(inp, size=d, replace=False)
        pos += d
    order = _rng(seed, 4).permutation(nnz)
    return rows[order].astype(np.int32), cols[order].astype(np.int32)


def normal(shape, std: float, seed: int, salt: int) -> np.ndarray:
    """fp32 N(0, std^2) array (std is the standard deviation)."""
    return (_rng(seed, 10 + salt).standard_normal(shape) * std).astype(np.float32)


@dataclass
class Layer:
    """One sparse layer of a workload: shape, pattern and values."""
    name: str
    out: int
    inp: int
    sparsity: float
    pattern: str = "uniform"  # or "zipf"
    val_std: float = 1.0
    seed: int = 0

    @property
    def nnz(self) -> int:
        return nnz_for(self.out, self.inp, self.sparsity)

    def coo(self):
        """(row, col, val) in shuffled user order."""
        if self.pattern == "zipf":
            row, col = zipf_pattern(self.out, self.inp, self.nnz, 1.1, self.seed)
        else:
            row, col = uniform_pattern(self.out, self.inp, self.nnz, self.seed)
        val = normal(row.size, self.val_std, self.seed, 0)
        return row, col, val

    def activations(self, B: int, salt: int = 0):
        """(X [B][in], dY [B][out]) ~ N(0, 1) fp32."""
        X = normal((B, self.inp), 1.0, self.seed, 100 + 2 * salt)
        dY = normal((B, self.out), 1.0, self.seed, 101 + 2 * salt)
        return X, dY


@dataclass
class Workload:
    name: str
    layers: list
    batches: list
    kernels: tuple = ("fwd", "bwd_input", "bwd_weight")
    notes: str = ""
    extra: dict = field(default_factory=dict)


def workload(name: str, seed: int = 0) -> Workload:
    """The named synthetic workloads.

    toy256     256x256 at 90%, values N(0, 1/sqrt(nnz/out)), batch 4
    gpt2_mlp   768->3072 and 3072->768 at 95%, values N(0, 0.02), batch 1/8/32
    large{90,95,99}  10000x10000, values N(0, 1/sqrt(in)), batch 1/4/16/64
    large      the three 10000x10000 layers together, batch 1/4/8/16/64
    skewed     8192x8192 at 99%, rank-Zipf(1.1) rows, values N(0, 1), batch 1/16
    gpt2_decoder  12 blocks x (c_attn 768->2304, attn c_proj 768->768,
               c_fc 768->3072, mlp c_proj 3072->768) at 99%, 256 tokens
    """
    if name == "toy256":
        nnz = nnz_for(256, 256, 90)
        std = 1.0 / np.sqrt(nnz / 256)
        return Workload(name, [Layer("toy", 256, 256, 90, val_std=std, seed=seed)], [4])
    if name == "gpt2_mlp":
        return Workload(name, [Layer("c_fc", 3072, 768, 95, val_std=0.02, seed=seed),
                               Layer("c_proj", 768, 3072, 95, val_std=0.02, seed=seed + 1)],
                        [1, 8, 32])
    if name == "large":
        # the whole 10000x10000 sweep: 90 / 95 / 99 %, batches 1-64 (8 added
        # for the batch >= 8 operating point)
        return Workload(name, [Layer(f"large{sp}", 10000, 10000, sp, val_std=0.01, seed=seed)
                               for sp in (90, 95, 99)], [1, 4, 8, 16, 64])
    if name.startswith("large"):
        sp = int(name[5:] or 95)
        return Workload(name, [Layer(f"large{sp}", 10000, 10000, sp, val_std=0.01,
                                     seed=seed)], [1, 4, 16, 64])
    if name == "skewed":
        return Workload(name, [Layer("skewed", 8192, 8192, 99, pattern="zipf",
                                     val_std=1.0, seed=seed)], [1, 16])
    if name == "gpt2_decoder":
        layers = []
        for blk in range(12):
            for j, (nm, o, i) in enumerate([("c_attn", 2304, 768), ("attn_c_proj", 768, 768),
                                            ("c_fc", 3072, 768), ("mlp_c_proj", 768, 3072)]):
                layers.append(Layer(f"h{blk}.{nm}", o, i, 99, val_std=0.02,
                                    seed=seed + 1000 * blk + j))
        return Workload(name, layers, [256],
                        extra=dict(vocab=50257, d=768, heads=12, ctx=256, lr=1e-2,
                                   prune_frac=0.30, prune_every=100))
    raise KeyError(name)
