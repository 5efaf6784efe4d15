"""Seeded synthetic inputs with the shapes and structure of the pages' workloads.

This module only draws random numbers.  It holds none of the layer's
arithmetic (no product, gradient, sort, prune or regrow), so both the CUDA
path and the CPU oracle can take their inputs from it.

Workloads (page titles):
  * "Beyond Masked Sparsity: SNACK Enables Truly Sparse Neural Networks on GPU"
    - Fig. 2 (5000x5000, sparsity sweep, batch 1 and 2), Table 2 (500^2 ...
    10000^2 at 95%, batch 1), Fig. 3 / Table 3 (10000x10000, batch 1..64,
    SGD iterations), Tables 4-5 (GPT-2 small, whose MLP is 768 -> 3072 -> 768).
  * "Padded-CSR: A sparse storage format for dynamic sparse training on CPU"
    - sec. 8.2 (SET with drop_fraction 0.3).

All draws use numpy's ``Generator(PCG64(seed))``.  The support is drawn
uniformly without replacement over the out*in positions unless a power-law
(Zipf) row-degree profile is asked for.  The triple is returned in a random
order (not sorted), so that the library's own canonical sort is exercised.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

__all__ = [
    "nnz_for", "rng", "uniform_support", "zipf_row_degrees", "zipf_support",
    "normal", "Layer", "make_layer", "WORKLOADS",
]


def nnz_for(out_f: int, in_f: int, sparsity_pct: float) -> int:
    """nnz = round(out*in*(100 - s)/100), half up, in integer arithmetic for
    integer percentages."""
    total = out_f * in_f
    if float(sparsity_pct).is_integer():
        return (total * (100 - int(sparsity_pct)) * 2 + 100) // 200
    return int(np.floor(total * (100.0 - sparsity_pct) / 100.0 + 0.5))


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def uniform_support(out_f: int, in_f: int, nnz: int, seed: int):
    """nnz distinct positions, uniform without replacement, in draw order."""
    g = rng(seed)
    lin = g.choice(out_f * in_f, size=nnz, replace=False, shuffle=True).astype(np.int64)
    return (lin // in_f).astype(np.int32), (lin % in_f).astype(np.int32)


def zipf_row_degrees(out_f: int, in_f: int, nnz: int, s: float, seed: int) -> np.ndarray:
    """Row degrees that follow rank^(-s), capped at in_f, summing to nnz.

    A seeded permutation assigns ranks to rows.  Target degrees are water-filled
    (rows that would exceed in_f are capped and the excess is shared among the
    others in proportion to their weights), then rounded by largest remainder
    with ties going to the lower rank.
    """
    if nnz > out_f * in_f:
        raise ValueError("nnz exceeds out*in")
    w = np.arange(1, out_f + 1, dtype=np.float64) ** (-float(s))
    capped = np.zeros(out_f, dtype=bool)
    target = np.zeros(out_f, dtype=np.float64)
    while True:
        free_budget = nnz - in_f * capped.sum()
        wf = np.where(capped, 0.0, w)
        target = np.where(capped, float(in_f), free_budget * wf / wf.sum())
        over = (~capped) & (target > in_f)
        if not over.any():
            break
        capped |= over
    base = np.floor(target).astype(np.int64)
    base = np.minimum(base, in_f)
    rem = nnz - int(base.sum())
    frac = target - base
    # largest remainder first; among equal remainders the lower rank wins
    order = np.lexsort((np.arange(out_f), -frac))
    eligible = [i for i in order if base[i] < in_f]
    for i in eligible[:rem]:
        base[i] += 1
    assert int(base.sum()) == nnz
    rank_of_row = rng(seed).permutation(out_f)
    return base[rank_of_row].astype(np.int64)


def zipf_support(out_f: int, in_f: int, nnz: int, s: float, seed: int):
    """Support with Zipf(s) row degrees; columns uniform without replacement
    within each row; entries returned in a random order."""
    deg = zipf_row_degrees(out_f, in_f, nnz, s, seed)
    g = rng(seed + 1)
    rows = np.repeat(np.arange(out_f, dtype=np.int32), deg)
    cols = np.empty(nnz, dtype=np.int32)
    pos = 0
    for o in range(out_f):
        d = int(deg[o])
        if d:
            cols[pos:pos + d] = g.choice(in_f, size=d, replace=False)
            pos += d
    order = g.permutation(nnz)
    return rows[order], cols[order]


def normal(shape, std: float, seed: int) -> np.ndarray:
    return (rng(seed).standard_normal(shape) * std).astype(np.float32)


@dataclass
class Layer:
    out_f: int
    in_f: int
    values: np.ndarray
    rows: np.ndarray
    cols: np.ndarray

    @property
    def nnz(self) -> int:
        return int(self.values.shape[0])


def make_layer(out_f: int, in_f: int, sparsity_pct: float, value_std: float,
               seed_support: int, seed_values: int, zipf_s: float | None = None) -> Layer:
    nnz = nnz_for(out_f, in_f, sparsity_pct)
    if zipf_s is None:
        r, c = uniform_support(out_f, in_f, nnz, seed_support)
    else:
        r, c = zipf_support(out_f, in_f, nnz, zipf_s, seed_support)
    v = normal(nnz, value_std, seed_values)
    return Layer(out_f, in_f, v, r, c)


# Workload recipes: shape, sparsities, value scale, batches and seeds
# (support, values, X, dY or target, regrow).
WORKLOADS = {
    "layer500_s95": dict(out=500, inp=500, sparsity=[95], std=0.05, batches=[1],
                         seeds=(1, 2, 3, 4, None)),
    "layer5000_sweep": dict(out=5000, inp=5000, sparsity=[80, 90, 95, 99], std=0.01,
                            batches=[1, 2], seeds=(11, 12, 13, 14, None)),
    "layer10000_train": dict(out=10000, inp=10000, sparsity=[90, 95, 99], std=0.01,
                             batches=[1, 2, 4, 8, 16, 32, 64], seeds=(21, 22, 23, 24, None)),
    "layer10000_set": dict(out=10000, inp=10000, sparsity=[90], std=0.01, batches=[4],
                           seeds=(31, 32, 33, 34, 0x5E7), zeta=0.3, every=10),
    "gpt2_mlp_zipf": dict(blocks=12, d_model=768, d_ff=3072, sparsity=[90, 99], zipf_s=1.2,
                          batches=[1, 8, 64], seeds=(41, 42, 43, 44, None)),
}
