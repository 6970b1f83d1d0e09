"""An encode pass over several units, in the pages' order: factor every unit,
score its whole candidate grid, allocate under one byte budget, serialize the
chosen candidates.  Test infrastructure (see oracle/__init__.py).

[Joint Tucker-rank and residual-bit KV allocator, Implementation notes:
 separate candidate tables per group and cache type, one lambda for all.]
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional, Sequence

import numpy as np

from . import jolt


@dataclasses.dataclass
class EncodeResult:
    factors: List[jolt.Factors]
    dist: np.ndarray        # [U][n_rT][n_rd][n_b]
    cost: np.ndarray        # same shape, int64
    choice: np.ndarray      # [U] flat candidate index
    lam: float
    status: int
    blobs: List[bytes]


def unit_grid(H, T, D, rT_grid, rd_grid):
    return ([jolt.resolve(r, T) for r in rT_grid], [jolt.resolve(r, D) for r in rd_grid])


def encode_units(Xs: Sequence[np.ndarray], signs: Sequence[np.ndarray],
                 rT_grid, rd_grid, bits, block: int, budget: int,
                 token_mode: str = "exact", sketches: Optional[Sequence[np.ndarray]] = None,
                 power_iters: int = 2, cost_model: str = "formula", align: int = 256,
                 serialize: bool = True) -> EncodeResult:
    facs, dists, costs = [], [], []
    for u, X in enumerate(Xs):
        X = np.asarray(X, dtype=np.float64)
        H, T, D = X.shape
        sk = None if sketches is None else sketches[u]
        fac = jolt.factorize(X, rT_grid, rd_grid, token_mode, sk, power_iters)
        facs.append(fac)
        dists.append(jolt.dist_table(X, fac, signs[u], bits))
        costs.append(jolt.cost_table(H, T, D, fac.rT_list, fac.rd_list, bits, block,
                                     cost_model, align))
    dist = np.stack(dists)
    cost = np.stack(costs)
    U = dist.shape[0]
    choice, lam, status = jolt.allocate(dist.reshape(U, -1), cost.reshape(U, -1), budget, align)
    blobs = []
    if serialize:
        cands = jolt.candidate_list(facs[0].rT_list, facs[0].rd_list, bits)
        for u, X in enumerate(Xs):
            iT, idd, ib = cands[int(choice[u])]
            f = facs[u]
            blobs.append(jolt.encode_unit(X, f, signs[u], f.rT_list[iT], f.rd_list[idd],
                                          bits[ib], block, align))
    return EncodeResult(facs, dist, cost, choice, lam, status, blobs)
